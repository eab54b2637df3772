"""The forward entry point that allocates nothing (lmhead_logps_fwd_noalloc).

Some callers cannot call cudaMalloc: a plugin inside a host program that owns
every device allocation and gives it no allocator, or code on a path where an
allocation would synchronise the device.  For them the library keeps the
forward's scratch in a static per-GPU device array.  These tests call that
entry point through the C ABI twice in a row, on different inputs (so that
anything left in the shared array by the first call would show), and check:
- each result is bit for bit the regular workspace-taking forward's (the same
  kernels run the same plan, only the scratch address differs);
- one case against the fp64 oracle within the parity tolerances;
- that the calls allocate nothing: torch's allocator and the device's free
  memory are unchanged across them;
- that sizes beyond the array are rejected, after the usual argument checks.

The file is named so that pytest collects it last.
"""
import ctypes

import numpy as np
import pytest
import torch

import chunked_lm_head_tcgen05_gb300 as lm
from chunked_lm_head_tcgen05_gb300 import workloads as W

from gpu_helpers import LIMITS, ensure_built, run_oracle, to_device

pytestmark = pytest.mark.gpu


def _cases():
    return [
        W.WORKLOADS["tiny"].with_(T=1000, H=256, V=5000, chunk_size=64, temperature=0.7,
                                  seed=31, mask="bernoulli", mask_drop=0.25, hidden_dist="rms"),
        W.WORKLOADS["tiny"].with_(T=777, H=192, V=3001, chunk_size=16, temperature=1.0,
                                  seed=32, hidden_dist="rms"),
    ]


def _regular_forward(g, w):
    T, H, V = w.T, w.H, w.V
    ws = torch.empty(lm.lmhead_workspace_size(0, T, H, V, w.chunk_size), dtype=torch.uint8,
                     device="cuda")
    out = [torch.empty(T, device="cuda") for _ in range(3)]
    rc = lm.lmhead_logps_fwd(g["hidden"], g["weight"], g["targets"], g["loss_mask"],
                             w.temperature, w.chunk_size, *out, ws)
    assert rc == 0
    torch.cuda.synchronize()
    return out


def test_noalloc_forward_is_bitwise_the_regular_forward_on_two_calls():
    ensure_built()
    cases = _cases()
    data = []
    for w in cases:
        x = W.make_inputs(w, with_grads=False)
        g = to_device(x)
        ref = _regular_forward(g, w)
        got = [torch.full((w.T,), float("nan"), device="cuda") for _ in range(3)]
        data.append((w, x, g, ref, got))
    # warm-up call: the first call on a device does the set-up (symbol lookup)
    w, _, g, _, got = data[0]
    assert lm.lmhead_logps_fwd_noalloc(g["hidden"], g["weight"], g["targets"], g["loss_mask"],
                                       w.temperature, w.chunk_size, *got) == 0
    torch.cuda.synchronize()
    for t in got:
        t.fill_(float("nan"))
    torch.cuda.synchronize()
    alloc0 = torch.cuda.memory_allocated()
    reserved0 = torch.cuda.memory_reserved()
    free0, _ = torch.cuda.mem_get_info()
    for w, x, g, ref, got in data:
        rc = lm.lmhead_logps_fwd_noalloc(g["hidden"], g["weight"], g["targets"],
                                         g["loss_mask"], w.temperature, w.chunk_size, *got)
        assert rc == 0, lm.STATUS_NAMES.get(rc)
    torch.cuda.synchronize()
    free1, _ = torch.cuda.mem_get_info()
    assert torch.cuda.memory_allocated() == alloc0
    assert torch.cuda.memory_reserved() == reserved0
    assert free1 == free0
    for w, x, g, ref, got in data:
        for name, a, b in zip(("logp", "entropy", "lse"), got, ref):
            assert torch.equal(a, b), name
        if x["loss_mask"] is not None:
            m = x["loss_mask"].numpy() == 0
            assert np.all(got[0].cpu().numpy()[m] == 0.0)
    # one case against the oracle on the same inputs
    w, x, g, ref, got = data[0]
    o = run_oracle(x, backward=False, grad_logp=False, grad_entropy=False)
    for name, a in zip(("logp", "entropy", "lse"), got):
        a = a.cpu().double().numpy()
        assert np.abs(a - o[name]).max() <= LIMITS[name], name


def test_noalloc_rejects_sizes_beyond_its_scratch():
    ensure_built()
    lib = lm.library()
    fake = ctypes.c_void_p(1 << 20)
    T, H, V = 20000, 4096, 1000
    assert lm.lmhead_workspace_size(0, T, H, V, 64) > lm.NOALLOC_SCRATCH_BYTES
    rc = lib.lmhead_logps_fwd_noalloc(fake, fake, fake, None, T, H, V, 1.0, 64, fake, fake, fake,
                                      None)
    assert rc == 3   # LMHEAD_ERR_WORKSPACE_TOO_SMALL, nothing launched
    # the regular forward's own checks come first, as in lmhead_logps_fwd
    rc = lib.lmhead_logps_fwd_noalloc(fake, fake, fake, None, T, H, V, 0.0, 64, fake, fake, fake,
                                      None)
    assert rc == 1   # LMHEAD_ERR_INVALID_ARG: temperature
    rc = lib.lmhead_logps_fwd_noalloc(None, fake, fake, None, T, H, V, 1.0, 64, fake, fake, fake,
                                      None)
    assert rc == 1   # LMHEAD_ERR_INVALID_ARG: hidden missing
    rc = lib.lmhead_logps_fwd_noalloc(ctypes.c_void_p((1 << 20) + 2), fake, fake, None, T, H, V,
                                      1.0, 64, fake, fake, fake, None)
    assert rc == 2   # LMHEAD_ERR_UNSUPPORTED: misaligned hidden
