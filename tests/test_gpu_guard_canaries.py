"""Out-of-bounds writes, checked without a sanitizer.

Every buffer handed to the library is a view into a larger allocation. The
guard regions before and after the view hold a seeded random byte pattern:
the outputs, the caller's workspace, and the read-only inputs alike. After
each call the guards must hold the same bytes, and the inputs must be
entirely unchanged. A kernel that writes one byte past a buffer's end, or
before its start, or writes into an input, fails here. The shapes are ragged
in tokens, hidden size and vocabulary, with masked rows, so partial tiles,
partial K steps and the masked-row paths all run. Every entry point that
writes device memory is covered: the forward, the backward in its
persistent and per-block forms (with and without accumulation), the single
call in both strategies, the logits-level scoring pair, the forward
without a workspace, and the vocabulary-sharded forward, combine and
backward.
"""
import os

import numpy as np
import pytest
import torch

import chunked_lm_head_tcgen05_gb300 as lm
from chunked_lm_head_tcgen05_gb300 import workloads as W

from gpu_helpers import ensure_built

pytestmark = pytest.mark.gpu

GUARD = 4096   # bytes before and after each buffer (a multiple of 256: alignment is kept)


class Guarded:
    """A tensor of `shape` / `dtype` inside a guarded byte allocation."""

    def __init__(self, shape, dtype, seed, init=None):
        n = int(np.prod(shape)) * torch.empty((), dtype=dtype).element_size()
        self.n = n
        g = torch.Generator().manual_seed(seed)
        raw = torch.randint(0, 256, (GUARD + n + GUARD,), dtype=torch.uint8, generator=g)
        self.raw = raw.cuda()
        self.t = self.raw[GUARD:GUARD + n].view(dtype).view(shape)
        if init is not None:
            self.t.copy_(init)
        self.snap = self.raw.clone()

    def guards_intact(self):
        torch.cuda.synchronize()
        head = torch.equal(self.raw[:GUARD], self.snap[:GUARD])
        tail = torch.equal(self.raw[GUARD + self.n:], self.snap[GUARD + self.n:])
        return head and tail

    def unchanged(self):
        torch.cuda.synchronize()
        return torch.equal(self.raw, self.snap)

    def rearm(self):
        """Take the current bytes as the reference (after a call that writes the view)."""
        torch.cuda.synchronize()
        self.snap = self.raw.clone()


CASES = [
    # T, H, V, chunk, tau, mask, extra
    (333, 192, 3001, 64, 0.7, "bernoulli", dict(mask_drop=0.3)),
    (257, 320, 1025, 7, 1.3, "none", {}),
    (1, 64, 100, 1, 1.0, "none", {}),
]


def _inputs(case, seed):
    T, H, V, chunk, tau, mask, extra = case
    w = W.WORKLOADS["tiny"].with_(T=T, H=H, V=V, chunk_size=chunk, temperature=tau, mask=mask,
                                  hidden_dist="rms", weight_std=0.05, seed=seed, **extra)
    x = W.make_inputs(w)
    s = 1000 * seed
    gin = {
        "hidden": Guarded((T, H), torch.bfloat16, s + 1, x["hidden"]),
        "weight": Guarded((V, H), torch.bfloat16, s + 2, x["weight"]),
        "targets": Guarded((T,), torch.int32, s + 3, x["targets"]),
        "grad_logp": Guarded((T,), torch.float32, s + 4, x["grad_logp"]),
        "grad_entropy": Guarded((T,), torch.float32, s + 5, x["grad_entropy"]),
    }
    if x["loss_mask"] is not None:
        gin["loss_mask"] = Guarded((T,), torch.uint8, s + 6, x["loss_mask"])
    return w, gin


def _mask(gin):
    return gin["loss_mask"].t if "loss_mask" in gin else None


def _check(inputs, outputs, what):
    for name, b in inputs.items():
        assert b.unchanged(), "%s wrote into input %s" % (what, name)
    for name, b in outputs.items():
        assert b.guards_intact(), "%s wrote outside %s" % (what, name)


@pytest.mark.parametrize("ci", range(len(CASES)))
def test_two_call_path_stays_in_bounds(ci):
    ensure_built()
    w, gin = _inputs(CASES[ci], 40 + ci)
    T, H, V, c, tau = w.T, w.H, w.V, w.chunk_size, w.temperature
    ws_bytes = max(lm.lmhead_workspace_size(0, T, H, V, c), lm.lmhead_workspace_size(1, T, H, V, c))
    ws = Guarded((ws_bytes,), torch.uint8, 7)
    out = {n: Guarded((T,), torch.float32, 8 + i) for i, n in enumerate(("logp", "entropy", "lse"))}
    rc = lm.lmhead_logps_fwd(gin["hidden"].t, gin["weight"].t, gin["targets"].t, _mask(gin), tau, c,
                             out["logp"].t, out["entropy"].t, out["lse"].t, ws.t)
    assert rc == 0 and lm.lmhead_read_device_status(ws.t) == 0
    _check(gin, dict(out, workspace=ws), "lmhead_logps_fwd")
    saved = {"lse": out["lse"], "entropy": out["entropy"]}
    for b in saved.values():
        b.rearm()   # the backward reads these: from here on they are inputs

    old = os.environ.get("LMHEAD_BWD_PERSISTENT")
    try:
        for form in ("1", "0", "2"):
            os.environ["LMHEAD_BWD_PERSISTENT"] = form
            for accumulate in (0, 1):
                dh = Guarded((T, H), torch.float32, 11)
                dw = Guarded((V, H), torch.float32, 12, torch.randn((V, H)))
                rc = lm.lmhead_logps_bwd(gin["hidden"].t, gin["weight"].t, gin["targets"].t,
                                         _mask(gin), tau, c, gin["grad_logp"].t,
                                         gin["grad_entropy"].t, saved["lse"].t,
                                         saved["entropy"].t, dh.t, dw.t, accumulate, ws.t)
                assert rc == 0 and lm.lmhead_read_device_status(ws.t) == 0
                assert torch.isfinite(dh.t).all() and torch.isfinite(dw.t).all()
                _check(dict(gin, **saved), {"d_hidden": dh, "d_weight": dw, "workspace": ws},
                       "lmhead_logps_bwd (form %s, accumulate %d)" % (form, accumulate))
    finally:
        if old is None:
            os.environ.pop("LMHEAD_BWD_PERSISTENT", None)
        else:
            os.environ["LMHEAD_BWD_PERSISTENT"] = old


@pytest.mark.parametrize("ci", range(len(CASES)))
@pytest.mark.parametrize("strategy", ["keep_logits", "recompute"])
def test_single_call_stays_in_bounds(ci, strategy):
    ensure_built()
    w, gin = _inputs(CASES[ci], 50 + ci)
    T, H, V, c, tau = w.T, w.H, w.V, w.chunk_size, w.temperature
    ws = Guarded((lm.lmhead_workspace_size(2, T, H, V, c),), torch.uint8, 13)
    out = {n: Guarded((T,), torch.float32, 14 + i) for i, n in enumerate(("logp", "entropy", "lse"))}
    dh = Guarded((T, H), torch.float32, 17)
    dw = Guarded((V, H), torch.float32, 18)
    st = (lm.LMHEAD_STRATEGY_KEEP_LOGITS if strategy == "keep_logits"
          else lm.LMHEAD_STRATEGY_RECOMPUTE)
    rc = lm.lmhead_logps_fwd_bwd(gin["hidden"].t, gin["weight"].t, gin["targets"].t, _mask(gin),
                                 tau, c, gin["grad_logp"].t, gin["grad_entropy"].t, out["logp"].t,
                                 out["entropy"].t, out["lse"].t, dh.t, dw.t, 0, st, ws.t)
    assert rc == 0 and lm.lmhead_read_device_status(ws.t) == 0
    _check(gin, dict(out, d_hidden=dh, d_weight=dw, workspace=ws), "lmhead_logps_fwd_bwd")


def test_noalloc_forward_stays_in_bounds():
    ensure_built()
    w, gin = _inputs(CASES[0], 60)
    T = w.T
    out = {n: Guarded((T,), torch.float32, 20 + i) for i, n in enumerate(("logp", "entropy", "lse"))}
    rc = lm.lmhead_logps_fwd_noalloc(gin["hidden"].t, gin["weight"].t, gin["targets"].t,
                                     _mask(gin), w.temperature, w.chunk_size, out["logp"].t,
                                     out["entropy"].t, out["lse"].t)
    assert rc == 0
    _check(gin, out, "lmhead_logps_fwd_noalloc")


@pytest.mark.parametrize("V", [3001, 3000, 40001, 40000])
def test_score_logits_stays_in_bounds(V):
    ensure_built()
    T, tau = 133, 0.9
    r = np.random.default_rng(V)
    z = (r.normal(size=(T, V)) * 2.0).astype(np.float32)
    z[r.random((T, V)) < 0.05] = -np.inf
    gin = {
        "logits": Guarded((T, V), torch.float32, 30, torch.from_numpy(z)),
        "targets": Guarded((T,), torch.int32, 31,
                           torch.from_numpy(r.integers(0, V, size=T).astype(np.int32))),
        "loss_mask": Guarded((T,), torch.uint8, 32,
                             torch.from_numpy((r.random(T) > 0.2).astype(np.uint8))),
        "grad_logp": Guarded((T,), torch.float32, 33, torch.from_numpy(r.normal(size=T).astype(np.float32))),
        "grad_entropy": Guarded((T,), torch.float32, 34, torch.from_numpy(r.normal(size=T).astype(np.float32))),
    }
    out = {n: Guarded((T,), torch.float32, 35 + i) for i, n in enumerate(("logp", "entropy", "lse"))}
    rc = lm.lmhead_score_logits_fwd(gin["logits"].t, gin["targets"].t, gin["loss_mask"].t, tau,
                                    out["logp"].t, out["entropy"].t, out["lse"].t)
    assert rc == 0
    _check(gin, out, "lmhead_score_logits_fwd")
    for b in out.values():
        b.rearm()
    d = Guarded((T, V), torch.float32, 38)
    rc = lm.lmhead_score_logits_bwd(gin["logits"].t, gin["targets"].t, gin["loss_mask"].t, tau,
                                    gin["grad_logp"].t, gin["grad_entropy"].t, out["lse"].t,
                                    out["entropy"].t, d.t)
    assert rc == 0
    _check(dict(gin, lse=out["lse"], entropy=out["entropy"]), {"d_logits": d},
           "lmhead_score_logits_bwd")


@pytest.mark.parametrize("ci", range(len(CASES)))
def test_vocabulary_shards_stay_in_bounds(ci):
    """Each shard's table rows, statistics, d_hidden share and d_weight rows are
    buffers of their own, so a write past a shard's rows is caught."""
    ensure_built()
    w, gin = _inputs(CASES[ci], 70 + ci)
    T, H, V, c, tau = w.T, w.H, w.V, w.chunk_size, w.temperature
    cuts = sorted({0, V} | ({V // 3, (2 * V) // 3} if V >= 3 else set()))
    shards = list(zip(cuts[:-1], cuts[1:]))
    parts = []
    for j, (a, b) in enumerate(shards):
        wsh = Guarded((b - a, H), torch.bfloat16, 80 + j, gin["weight"].t[a:b])
        ws = Guarded((lm.lmhead_workspace_size(0, T, H, b - a, c),), torch.uint8, 90 + j)
        part = Guarded((T, 4), torch.float32, 100 + j)
        rc = lm.lmhead_logps_fwd_shard(gin["hidden"].t, wsh.t, gin["targets"].t, _mask(gin), a,
                                       V, tau, c, part.t, ws.t)
        assert rc == 0 and lm.lmhead_read_device_status(ws.t) == 0
        _check(dict(gin, weight_shard=wsh), {"partials": part, "workspace": ws},
               "lmhead_logps_fwd_shard (shard %d)" % j)
        parts.append(part)
    allp = Guarded((len(shards), T, 4), torch.float32, 110,
                   torch.stack([p_.t for p_ in parts]).cpu())
    out = {n: Guarded((T,), torch.float32, 111 + i) for i, n in enumerate(("logp", "entropy", "lse"))}
    rc = lm.lmhead_combine_shards(allp.t, gin["targets"].t, _mask(gin), V, out["logp"].t,
                                  out["entropy"].t, out["lse"].t)
    assert rc == 0
    _check(dict(gin, partials=allp), out, "lmhead_combine_shards")
    for b in out.values():
        b.rearm()
    for j, (a, b) in enumerate(shards):
        wsh = Guarded((b - a, H), torch.bfloat16, 120 + j, gin["weight"].t[a:b])
        ws = Guarded((lm.lmhead_workspace_size(1, T, H, b - a, c),), torch.uint8, 130 + j)
        dh = Guarded((T, H), torch.float32, 140 + j)
        dw = Guarded((b - a, H), torch.float32, 150 + j, torch.randn((b - a, H)))
        rc = lm.lmhead_logps_bwd_shard(gin["hidden"].t, wsh.t, gin["targets"].t, _mask(gin), a,
                                       V, tau, c, gin["grad_logp"].t, gin["grad_entropy"].t,
                                       out["lse"].t, out["entropy"].t, dh.t, dw.t, j % 2, ws.t)
        assert rc == 0 and lm.lmhead_read_device_status(ws.t) == 0
        assert torch.isfinite(dh.t).all() and torch.isfinite(dw.t).all()
        _check(dict(gin, weight_shard=wsh, lse=out["lse"], entropy=out["entropy"]),
               {"d_hidden": dh, "d_weight_shard": dw, "workspace": ws},
               "lmhead_logps_bwd_shard (shard %d)" % j)
