"""The forward entry point that allocates nothing (lmhead_logps_fwd_noalloc).

Some callers cannot call cudaMalloc: a plugin inside a host program that owns
every device allocation and gives it no allocator, or code on a path where an
allocation would synchronise the device.  For them the library keeps the
forward's scratch in a static per-GPU device array.  This test calls that
entry point through the C ABI twice in a row, on different inputs (so that
anything left in the shared array by the first call would show), and checks
each result against the regular workspace-taking forward within the parity
tolerances.  It also checks that sizes beyond the array are rejected.

The file is named so that pytest collects it last.
"""
import ctypes

import numpy as np
import pytest
import torch

import chunked_lm_head_tcgen05_gb300 as lm
from chunked_lm_head_tcgen05_gb300 import workloads as W

from gpu_helpers import LIMITS, ensure_built, to_device

pytestmark = pytest.mark.gpu


def _regular_forward(g, w):
    T, H, V = w.T, w.H, w.V
    ws = torch.empty(lm.lmhead_workspace_size(0, T, H, V, w.chunk_size), dtype=torch.uint8,
                     device="cuda")
    out = [torch.empty(T, device="cuda") for _ in range(3)]
    rc = lm.lmhead_logps_fwd(g["hidden"], g["weight"], g["targets"], g["loss_mask"],
                             w.temperature, w.chunk_size, *out, ws)
    assert rc == 0
    return out


def test_noalloc_forward_matches_regular_forward_on_two_calls():
    ensure_built()
    cases = [
        W.WORKLOADS["tiny"].with_(T=1000, H=256, V=5000, chunk_size=64, temperature=0.7,
                                  seed=31, mask="bernoulli", mask_drop=0.25, hidden_dist="rms"),
        W.WORKLOADS["tiny"].with_(T=777, H=192, V=3001, chunk_size=16, temperature=1.0,
                                  seed=32, hidden_dist="rms"),
    ]
    for w in cases:
        x = W.make_inputs(w, with_grads=False)
        g = to_device(x)
        ref = _regular_forward(g, w)
        got = [torch.full((w.T,), float("nan"), device="cuda") for _ in range(3)]
        rc = lm.lmhead_logps_fwd_noalloc(g["hidden"], g["weight"], g["targets"], g["loss_mask"],
                                         w.temperature, w.chunk_size, *got)
        assert rc == 0, lm.STATUS_NAMES.get(rc)
        torch.cuda.synchronize()
        for name, a, b in zip(("logp", "entropy", "lse"), got, ref):
            a = a.cpu().double().numpy()
            b = b.cpu().double().numpy()
            assert np.array_equal(np.isfinite(a), np.isfinite(b)), name
            assert np.abs(a - b).max() <= LIMITS[name], name
        if x["loss_mask"] is not None:
            m = x["loss_mask"].numpy() == 0
            assert np.all(got[0].cpu().numpy()[m] == 0.0)


def test_noalloc_rejects_sizes_beyond_its_scratch():
    ensure_built()
    lib = lm.library()
    fake = ctypes.c_void_p(1 << 20)
    T, H, V = 20000, 4096, 1000
    assert lm.lmhead_workspace_size(0, T, H, V, 64) > lm.NOALLOC_SCRATCH_BYTES
    rc = lib.lmhead_logps_fwd_noalloc(fake, fake, fake, None, T, H, V, 1.0, 64, fake, fake, fake,
                                      None)
    assert rc == 3   # LMHEAD_ERR_WORKSPACE_TOO_SMALL, nothing launched
