"""Pins for the fp64 oracle: checks against facts the mathematics fixes.

Each ``pin_*`` function takes an ``oracle.Oracle`` instance and raises
AssertionError when the oracle disagrees with a closed form, an invariant, a
special case that reduces to a textbook formula, finite differences, or a
hand-derived fixture.  None of them re-types the oracle's own formula.
``test_oracle_pins.py`` runs them on the oracle; ``test_oracle_mutants.py``
runs them on deliberately broken copies of it, each of which must fail at
least one pin.
"""
import json
import math
import os

import mpmath
import numpy as np

mpmath.mp.dps = 50   # closed forms are evaluated well beyond double precision

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def _rng(seed):
    return np.random.default_rng(seed)


def _close(a, b, atol, rtol=0.0, what=""):
    a = np.asarray(a, np.float64)
    b = np.asarray(b, np.float64)
    err = np.abs(a - b)
    lim = atol + rtol * np.abs(b)
    assert np.all(err <= lim), "%s: max err %.3e (limit %.3e)" % (what, float(err.max()), float(lim.max()))


def pin_zero_weight_forward(o):
    """W = 0: every logit is 0, so p is uniform: lse = ln V, logp = -ln V, H = ln V."""
    r = _rng(1)
    for V, H in ((2048, 8), (151936, 4), (3, 5)):
        T = 6
        h = r.normal(size=(T, H))
        W = np.zeros((V, H))
        y = np.array([0, V - 1, 1, -1, -V, 2 % V], np.int32)
        logp, ent, lse = o.forward(h, W, y, None, 0.7)
        lnV = math.log(V)
        _close(lse, lnV, 1e-12, what="lse")
        _close(logp, -lnV, 1e-12, what="logp")
        _close(ent, lnV, 1e-11, what="entropy")


def pin_one_hot_dominant(o):
    """One logit a, the others 0: lse = ln(e^a + V - 1), logp = a - lse,
    H = lse - a e^(a - lse); as a grows, logp -> 0 and H -> 0."""
    V = 1000
    prev = None
    for a in (0.25, 3.0, 20.0, 60.0, 300.0):
        for tau in (1.0, 0.7):
            y = 123
            W = np.zeros((V, 1))
            W[y, 0] = a * tau              # z_y = (1 * a tau) / tau = a
            h = np.ones((1, 1))
            logp, ent, lse = o.forward(h, W, np.array([y], np.int32), None, tau)
            A = mpmath.mpf(a)
            L = mpmath.log(mpmath.exp(A) + (V - 1))
            Hx = L - A * mpmath.exp(A - L)
            # a plain left-to-right sum of V terms carries up to ~V ulps of
            # error in the exp-sum; the entropy amplifies it by |z| ~ a
            bound = 4 * V * 2.0 ** -52 * (1.0 + a)
            _close(lse, float(L), bound, 0.0, "lse a=%g" % a)
            _close(logp, float(A - L), bound, 0.0, "logp a=%g" % a)
            _close(ent, float(Hx), bound, 0.0, "entropy a=%g" % a)
        if prev is not None:
            assert logp[0] >= prev[0] and ent[0] <= prev[1]
        prev = (logp[0], ent[0])
    assert abs(prev[0]) < 1e-100 and abs(prev[1]) < 1e-100


def pin_softmax_sums_to_one(o):
    """One hidden row scored against every target: sum_y exp(logp(y)) = 1."""
    r = _rng(2)
    for V, H, tau in ((64, 16, 1.0), (257, 7, 0.7)):
        hrow = r.normal(size=(1, H))
        W = r.normal(size=(V, H))
        h = np.repeat(hrow, V, axis=0)
        y = np.arange(V, dtype=np.int32)
        logp, ent, lse = o.forward(h, W, y, None, tau)
        total = math.fsum(np.exp(logp))
        assert abs(total - 1.0) < 1e-12, total
        assert np.all(lse == lse[0]) and np.all(ent == ent[0])


def pin_two_class_is_sigmoid(o):
    """V = 2 reduces to the logistic function and the binary entropy."""
    r = _rng(3)
    T, H = 40, 3
    h = r.normal(size=(T, H)) * 3
    W = r.normal(size=(2, H))
    y = r.integers(0, 2, size=T).astype(np.int32)
    tau = 0.7
    logp, ent, _ = o.forward(h, W, y, None, tau)
    for t in range(T):
        z = [sum(h[t, k] * W[v, k] for k in range(H)) / tau for v in range(2)]
        d = z[y[t]] - z[1 - y[t]]
        want_logp = -math.log1p(math.exp(-d)) if d > 0 else d - math.log1p(math.exp(d))
        q = 1.0 / (1.0 + math.exp(-(z[1] - z[0])))
        want_h = -(q * math.log(q) + (1 - q) * math.log(1 - q))
        assert abs(logp[t] - want_logp) < 1e-12, (t, logp[t], want_logp)
        assert abs(ent[t] - want_h) < 1e-12, (t, ent[t], want_h)


def pin_golden_fixture(o):
    """Hand-derived fixture (tests/golden/softmax_123.json): logits ln1, ln2, ln3."""
    with open(os.path.join(GOLDEN, "softmax_123.json")) as f:
        fx = json.load(f)
    env = {"log": mpmath.log, "mpf": mpmath.mpf}
    W = np.array([[float(mpmath.log(k))] for k in (1, 2, 3)])
    h = np.ones((1, 1))
    for case in fx["forward"]:
        y = np.array([case["target"]], np.int32)
        logp, ent, lse = o.forward(h, W, y, None, 1.0)
        _close(lse, float(eval(case["lse"], env)), 1e-15, 1e-15, "golden lse")
        _close(logp, float(eval(case["logp"], env)), 1e-15, 1e-15, "golden logp")
        _close(ent, float(eval(case["entropy"], env)), 1e-15, 1e-15, "golden entropy")
    for case in fx["backward"]:
        y = np.array([case["target"]], np.int32)
        gl = np.array([case["grad_logp"]], np.float64)
        ge = np.array([case["grad_entropy"]], np.float64)
        dh, dw = o.backward(h, W, y, None, 1.0, gl, ge)
        _close(dh[0, 0], float(eval(case["d_hidden"], env)), 1e-15, 1e-14, "golden d_hidden")
        want = [float(eval(e, env)) for e in case["d_weight"]]
        _close(dw[:, 0], want, 1e-15, 1e-14, "golden d_weight")


def pin_entropy_bounds(o):
    """0 <= H <= ln V always; sharper logits give lower entropy."""
    r = _rng(4)
    T, H, V = 30, 6, 50
    h = r.normal(size=(1, H)) * np.linspace(0.01, 20, T)[:, None]
    W = r.normal(size=(V, H))
    _, ent, _ = o.forward(h, W, np.zeros(T, np.int32), None, 1.0)
    assert np.all(ent >= -1e-12) and np.all(ent <= math.log(V) + 1e-12)
    assert ent[0] > ent[-1]
    assert abs(ent[0] - math.log(V)) < 1e-3


def pin_temperature_power_of_two(o):
    """tau = 2^k scales exactly: head(h, W, tau) == head(h / tau, W, 1) bit for bit."""
    r = _rng(5)
    T, H, V = 9, 12, 40
    h = r.normal(size=(T, H))
    W = r.normal(size=(V, H))
    y = r.integers(-V, V, size=T).astype(np.int32)
    for tau in (0.5, 2.0, 0.25):
        a = o.forward(h, W, y, None, tau)
        b = o.forward(h / tau, W, y, None, 1.0)
        for u, v in zip(a, b):
            assert np.array_equal(u, v)


def pin_shift_invariance(o):
    """W_v -> W_v + c for every v: logp, H, d_hidden unchanged; lse += h.c / tau."""
    r = _rng(6)
    T, H, V, tau = 7, 10, 33, 0.7
    h = r.normal(size=(T, H))
    W = r.normal(size=(V, H))
    c = r.normal(size=H)
    y = r.integers(0, V, size=T).astype(np.int32)
    gl, ge = r.normal(size=T), r.normal(size=T)
    a = o.forward(h, W, y, None, tau)
    b = o.forward(h, W + c, y, None, tau)
    _close(b[0], a[0], 1e-11, what="logp shift")
    _close(b[1], a[1], 1e-11, what="entropy shift")
    _close(b[2], a[2] + h @ c / tau, 1e-11, what="lse shift")
    da, _ = o.backward(h, W, y, None, tau, gl, ge, want_dweight=False)
    db, _ = o.backward(h, W + c, y, None, tau, gl, ge, want_dweight=False)
    # d_hidden picks up sum_v dz_v c / tau = 0 since sum_v dz_v = 0
    _close(db, da, 1e-10, what="d_hidden shift")


def _loss(o, h, W, y, mask, tau, gl, ge):
    logp, ent, _ = o.forward(h, W, y, mask, tau)
    return math.fsum(gl * logp) + math.fsum(ge * ent)


def pin_finite_differences(o):
    """Central differences of L = sum g_l logp + g_e H with respect to h and W."""
    r = _rng(7)
    T, H, V, tau = 5, 8, 16, 0.7
    h = r.normal(size=(T, H))
    W = r.normal(size=(V, H)) * 0.8
    y = np.array([3, -2, 15, 0, 7], np.int32)
    mask = np.array([1, 1, 1, 0, 1], np.uint8)
    gl = r.normal(size=T)
    ge = r.normal(size=T)
    dh, dw = o.backward(h, W, y, mask, tau, gl, ge)
    eps = 1e-6
    for t in range(T):
        for k in range(H):
            hp, hm = h.copy(), h.copy()
            hp[t, k] += eps
            hm[t, k] -= eps
            fd = (_loss(o, hp, W, y, mask, tau, gl, ge) - _loss(o, hm, W, y, mask, tau, gl, ge)) / (2 * eps)
            assert abs(fd - dh[t, k]) <= 1e-7 + 1e-6 * abs(fd), ("d_hidden", t, k, fd, dh[t, k])
    for v in range(V):
        for k in range(H):
            wp, wm = W.copy(), W.copy()
            wp[v, k] += eps
            wm[v, k] -= eps
            fd = (_loss(o, h, wp, y, mask, tau, gl, ge) - _loss(o, h, wm, y, mask, tau, gl, ge)) / (2 * eps)
            assert abs(fd - dw[v, k]) <= 1e-7 + 1e-6 * abs(fd), ("d_weight", v, k, fd, dw[v, k])


def pin_zero_weight_backward(o):
    """W = 0: p = 1/V and log p + H = 0, so dz = g_l (onehot - 1/V); d_hidden = 0
    and d_weight[v] = sum_t g_l,t (delta_{v,y_t} - 1/V) h_t / tau."""
    r = _rng(8)
    T, H, V, tau = 6, 5, 9, 0.7
    h = r.normal(size=(T, H))
    W = np.zeros((V, H))
    y = np.array([1, -1, 4, 0, 8, 3], np.int32)
    gl, ge = r.normal(size=T), r.normal(size=T)
    dh, dw = o.backward(h, W, y, None, tau, gl, ge)
    assert np.all(dh == 0.0)
    want = np.zeros((V, H))
    for t in range(T):
        yy = y[t] % V
        for v in range(V):
            want[v] += gl[t] * ((1.0 if v == yy else 0.0) - 1.0 / V) * h[t] / tau
    _close(dw, want, 1e-13, 1e-12, "d_weight with W = 0")


def pin_dweight_column_sums(o):
    """sum_v dz_v = 0 for every token, so the column sums of d_weight vanish."""
    r = _rng(9)
    T, H, V = 11, 7, 29
    h = r.normal(size=(T, H))
    W = r.normal(size=(V, H))
    y = r.integers(0, V, size=T).astype(np.int32)
    _, dw = o.backward(h, W, y, None, 0.7, r.normal(size=T), r.normal(size=T))
    scale = np.abs(dw).max()
    assert scale > 0
    assert np.abs(dw.sum(axis=0)).max() < 1e-12 * scale * V


def pin_masks_and_targets(o):
    """Unscored rows give +0.0 everywhere; a NaN hidden row that is unscored
    changes nothing; a negative id equals its wrapped twin bit for bit; an id
    outside [-V, V) gives logp = NaN and drops the one-hot term."""
    r = _rng(10)
    T, H, V, tau = 8, 6, 20, 0.7
    h = r.normal(size=(T, H))
    W = r.normal(size=(V, H))
    y = r.integers(0, V, size=T).astype(np.int32)
    mask = np.array([1, 0, 1, 1, 0, 1, 1, 1], np.uint8)
    gl, ge = r.normal(size=T), r.normal(size=T)
    logp, ent, lse = o.forward(h, W, y, mask, tau)
    for a in (logp, ent, lse):
        assert np.all(a[mask == 0] == 0.0) and not np.any(np.signbit(a[mask == 0]))
    dh, dw = o.backward(h, W, y, mask, tau, gl, ge)
    assert np.all(dh[mask == 0] == 0.0)
    h_nan = h.copy()
    h_nan[mask == 0] = np.nan
    dh2, dw2 = o.backward(h_nan, W, y, mask, tau, gl, ge)
    assert np.array_equal(dw, dw2) and np.array_equal(dh, dh2)
    # wrap of negative ids
    y_neg = y.copy()
    y_neg[::2] -= V
    a = o.forward(h, W, y_neg, mask, tau)
    b = o.forward(h, W, y, mask, tau)
    for u, v in zip(a, b):
        assert np.array_equal(u, v)
    assert np.array_equal(o.backward(h, W, y_neg, mask, tau, gl, ge)[1], dw)
    # ids outside the vocabulary
    y_bad = y.copy()
    y_bad[0], y_bad[2] = V, -V - 1
    lp, en, ls = o.forward(h, W, y_bad, None, tau)
    ref = o.forward(h, W, y, None, tau)
    assert np.isnan(lp[0]) and np.isnan(lp[2])
    assert np.array_equal(en, ref[1]) and np.array_equal(ls, ref[2])
    assert np.array_equal(lp[[1, 3, 4, 5, 6, 7]], ref[0][[1, 3, 4, 5, 6, 7]])
    one = np.zeros(T)
    one[0] = 1.0
    dh_bad, _ = o.backward(h, W, y_bad, None, tau, one, np.zeros(T))
    dh_ok, _ = o.backward(h, W, y, None, tau, one, np.zeros(T))
    _close(dh_bad[0], dh_ok[0] - W[y[0]] / tau, 1e-12, what="dropped one-hot")


def pin_bf16_storage(o):
    """bf16 bit patterns decode to the same numbers torch gives them."""
    import torch
    r = _rng(11)
    T, H, V = 4, 16, 24
    ht = torch.from_numpy(r.normal(size=(T, H))).to(torch.bfloat16)
    wt = torch.from_numpy(r.normal(size=(V, H)) * 0.1).to(torch.bfloat16)
    hb = ht.view(torch.int16).numpy().view(np.uint16)
    wb = wt.view(torch.int16).numpy().view(np.uint16)
    hd = ht.to(torch.float64).numpy()
    wd = wt.to(torch.float64).numpy()
    y = np.arange(T, dtype=np.int32)
    a = o.forward(hb, wb, y, None, 1.0)
    b = o.forward(hd, wd, y, None, 1.0)
    for u, v in zip(a, b):
        assert np.array_equal(u, v)
    ga = o.backward(hb, wb, y, None, 1.0, np.ones(T), np.ones(T))
    gb = o.backward(hd, wd, y, None, 1.0, np.ones(T), np.ones(T))
    for u, v in zip(ga, gb):
        assert np.array_equal(u, v)


def _logits_via_head(o, logits, y, mask, tau, gl, ge):
    """Score logits with the hidden-state oracle: hidden = one-hot rows,
    W[v, t] = logits[t, v], so z[t, v] = logits[t, v] / tau; d logits[t, v]
    is then d_weight[v, t]."""
    T, V = logits.shape
    h = np.eye(T)
    W = np.ascontiguousarray(logits.T)
    f = o.forward(h, W, y, mask, tau)
    _, dw = o.backward(h, W, y, mask, tau, gl, ge)
    return f, np.ascontiguousarray(dw.T)


def pin_logits_match_head(o):
    """Finite logits: the logits-level scoring equals the head's definition."""
    r = _rng(12)
    T, V, tau = 7, 40, 0.7
    logits = r.normal(size=(T, V)) * 2
    y = r.integers(-V, V, size=T).astype(np.int32)
    mask = np.array([1, 1, 0, 1, 1, 1, 1], np.uint8)
    gl, ge = r.normal(size=T), r.normal(size=T)
    (hl, he, hs), hd = _logits_via_head(o, logits, y, mask, tau, gl, ge)
    lp, en, ls = o.logits_forward(logits, y, mask, tau)
    d = o.logits_backward(logits, y, mask, tau, gl, ge)
    _close(lp, hl, 1e-12, 1e-12, "logits logp")
    _close(en, he, 1e-12, 1e-12, "logits entropy")
    _close(ls, hs, 1e-12, 1e-12, "logits lse")
    _close(d, hd, 1e-12, 1e-10, "logits gradient")


def pin_logits_neg_inf_is_removal(o):
    """-inf entries behave as if those vocabulary entries were absent, and get
    a zero cotangent (isfinite mask); a -inf target logit gives logp = -inf."""
    r = _rng(13)
    V, tau = 30, 0.9
    row = r.normal(size=V)
    gone = np.array([1, 5, 6, 17, 29])
    row[gone] = -np.inf
    keep = np.setdiff1d(np.arange(V), gone)
    y = np.array([8, 5], np.int32)            # a kept id, then a -inf id
    gl, ge = np.array([0.7, 1.3]), np.array([-0.4, 0.8])
    z = np.stack([row, row])
    lp, en, ls = o.logits_forward(z, y, None, tau)
    d = o.logits_backward(z, y, None, tau, gl, ge)
    short = row[keep][None, :]
    ys = np.array([int(np.searchsorted(keep, 8))], np.int32)
    (hl, he, hs), hd = _logits_via_head(o, short, ys, None, tau, gl[:1], ge[:1])
    _close(lp[0], hl[0], 1e-12, 1e-12, "removal logp")
    _close(en, he[0], 1e-12, 1e-12, "removal entropy")
    _close(ls, hs[0], 1e-12, 1e-12, "removal lse")
    assert lp[1] == -np.inf
    assert np.all(d[:, gone] == 0.0)
    _close(d[0, keep], hd[0], 1e-12, 1e-10, "removal gradient")
    # the -inf target: no one-hot term, the rest as for a target of zero weight
    (h2, _, _), hd2 = _logits_via_head(o, short, np.array([-1000], np.int32), None, tau,
                                       np.array([gl[1]]), np.array([ge[1]]))
    assert np.isnan(h2[0])
    _close(d[1, keep], hd2[0], 1e-12, 1e-10, "-inf target gradient")


def pin_logits_nonfinite_rows(o):
    """NaN or +inf anywhere -> NaN statistics, NaN cotangent on finite entries,
    zero on the rest; a row with no finite logit -> lse = -inf, logp and
    entropy NaN, zero cotangent."""
    V = 6
    z = np.array([[0.1, np.nan, 0.3, -np.inf, 1.0, 2.0],
                  [0.1, np.inf, 0.3, -np.inf, 1.0, 2.0],
                  [-np.inf] * V,
                  [0.5, -1.0, 0.0, 2.0, -np.inf, 1.0]])
    y = np.array([0, 0, 2, 3], np.int32)
    lp, en, ls = o.logits_forward(z, y, None, 1.0)
    d = o.logits_backward(z, y, None, 1.0, np.ones(4), np.ones(4))
    for t in (0, 1):
        assert np.isnan(lp[t]) and np.isnan(en[t]) and np.isnan(ls[t])
        fin = np.isfinite(z[t])
        assert np.all(np.isnan(d[t][fin])) and np.all(d[t][~fin] == 0.0)
    assert ls[2] == -np.inf and np.isnan(lp[2]) and np.isnan(en[2]) and np.all(d[2] == 0.0)
    assert np.all(np.isfinite([lp[3], en[3], ls[3]])) and d[3, 4] == 0.0


ALL_PINS = [
    pin_zero_weight_forward,
    pin_one_hot_dominant,
    pin_softmax_sums_to_one,
    pin_two_class_is_sigmoid,
    pin_golden_fixture,
    pin_entropy_bounds,
    pin_temperature_power_of_two,
    pin_shift_invariance,
    pin_finite_differences,
    pin_zero_weight_backward,
    pin_dweight_column_sums,
    pin_masks_and_targets,
    pin_bf16_storage,
    pin_logits_match_head,
    pin_logits_neg_inf_is_removal,
    pin_logits_nonfinite_rows,
]
