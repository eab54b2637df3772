"""Logits-level scoring (lmhead_score_logits_fwd / _bwd) against the fp64
oracle, including -inf, +inf and NaN logits, a row with no finite logit,
unscored rows, negative and invalid ids, both load paths (V % 4 == 0 or
not) and the in-place backward."""
import numpy as np
import pytest
import torch

import chunked_lm_head_tcgen05_gb300 as lm
import oracle

from gpu_helpers import ensure_built

pytestmark = pytest.mark.gpu


def _case(T, V, seed):
    r = np.random.default_rng(seed)
    z = (r.normal(size=(T, V)) * 2.0).astype(np.float32)
    z[r.random((T, V)) < 0.05] = -np.inf
    z[3, :] = -np.inf                      # no finite logit
    z[5, 7] = np.nan
    z[6, 11] = np.inf
    y = r.integers(0, V, size=T).astype(np.int32)
    y[8] = -2                              # wraps
    y[9] = V + 4                           # invalid id
    y[10] = int(np.flatnonzero(np.isneginf(z[10]))[0])   # target logit is -inf
    m = (r.random(T) > 0.15).astype(np.uint8)
    m[[3, 5, 6, 8, 9, 10]] = 1
    gl = r.normal(size=T).astype(np.float32)
    ge = r.normal(size=T).astype(np.float32)
    return z, y, m, gl, ge


def _same_pattern(a, b):
    return np.array_equal(np.isnan(a), np.isnan(b)) and np.array_equal(np.isposinf(a), np.isposinf(b)) \
        and np.array_equal(np.isneginf(a), np.isneginf(b))


# 3000 / 3001: one CTA per row; 70000 / 70001: rows spread over a cluster of 4 CTAs in
# the forward and 4 independent CTAs in the backward (16-byte and scalar load paths)
@pytest.mark.parametrize("V", [3001, 3000, 70001, 70000])
@pytest.mark.parametrize("in_place", [False, True])
def test_score_logits_against_oracle(V, in_place):
    ensure_built()
    T, tau = 200, 0.7
    z, y, m, gl, ge = _case(T, V, 17 + V)
    o = oracle.default()
    olp, oen, ols = o.logits_forward(z.astype(np.float64), y, m, tau)
    od = o.logits_backward(z.astype(np.float64), y, m, tau, gl.astype(np.float64),
                           ge.astype(np.float64))
    dz = torch.from_numpy(z).cuda()
    dy, dm = torch.from_numpy(y).cuda(), torch.from_numpy(m).cuda()
    logp, ent, lse = (torch.empty(T, device="cuda") for _ in range(3))
    assert lm.lmhead_score_logits_fwd(dz, dy, dm, tau, logp, ent, lse) == 0
    out = dz if in_place else torch.empty_like(dz)
    assert lm.lmhead_score_logits_bwd(dz, dy, dm, tau, torch.from_numpy(gl).cuda(),
                                      torch.from_numpy(ge).cuda(), lse, ent, out) == 0
    torch.cuda.synchronize()
    for name, a, b in (("logp", logp, olp), ("entropy", ent, oen), ("lse", lse, ols)):
        a = a.cpu().double().numpy()
        assert _same_pattern(a, b), name
        fin = np.isfinite(b)
        assert np.abs(a[fin] - b[fin]).max() < 1e-4, name
    g = out.cpu().double().numpy()
    assert _same_pattern(g, od)
    fin = np.isfinite(od)
    assert np.all(g[~np.isfinite(z)] == 0.0)           # isfinite mask
    assert np.abs(g[fin] - od[fin]).max() <= 1e-5 + 1e-4 * np.abs(od[fin]).max()
    assert np.all(g[m == 0] == 0.0)
