"""Seeded random configurations against the oracle: token counts, hidden and
vocabulary sizes, chunk sizes, temperatures, mask styles, missing
cotangents and d_weight accumulation drawn together, at sizes the oracle
finishes in about a second each.  Each case also runs the single-call path
with kept logits (the fp16 logit store and in-place cotangent pass) against
the oracle, and every fourth case the other backward forms (two launches per
block, launch windows), which must give the default path's bits."""
import os

import numpy as np
import pytest
import torch

import chunked_lm_head_tcgen05_gb300 as lm
from chunked_lm_head_tcgen05_gb300 import workloads as W

from gpu_helpers import assert_parity, run_gpu, run_gpu_fwd_bwd, run_oracle

pytestmark = pytest.mark.gpu

N_CASES = 24


def _case(i):
    r = np.random.default_rng(20261202 + 1000 + i)
    T = int(r.choice([1, 2, 7, 129, 255, 256, 257, int(r.integers(300, 900))]))
    H = int(64 * r.integers(1, 9))
    V = int(r.choice([1, 2, 255, 256, 257, int(r.integers(300, 5000))]))
    chunk = int(r.choice([1, 16, 64, 500, 2048]))
    tau = float(r.choice([0.3, 0.7, 1.0, 2.5]))
    mask = str(r.choice(["none", "bernoulli", "prompt_prefix"]))
    extra = {}
    if mask == "bernoulli":
        extra["mask_drop"] = float(r.uniform(0.05, 0.9))
    if mask == "prompt_prefix":
        extra["rows"] = 1
    opts = dict(grad_entropy=bool(r.random() > 0.25), accumulate=bool(r.random() > 0.7))
    w = W.WORKLOADS["tiny"].with_(T=T, H=H, V=V, chunk_size=chunk, temperature=tau, mask=mask,
                                  hidden_dist="rms", weight_std=float(r.choice([0.02, 0.05, 0.2])),
                                  seed=int(r.integers(1, 1 << 30)), **extra)
    return w, opts


@pytest.mark.parametrize("i", range(N_CASES))
def test_random_configuration(i):
    w, opts = _case(i)
    x = W.make_inputs(w)
    V, H = x["weight"].shape
    init = None
    if opts["accumulate"]:
        init = torch.randn((V, H), generator=torch.Generator().manual_seed(i))
    g = run_gpu(x, grad_entropy=opts["grad_entropy"], accumulate=opts["accumulate"],
                d_weight_init=init)
    assert g["fwd_status"] == 0 and g["bwd_status"] == 0
    o = run_oracle(x, grad_entropy=opts["grad_entropy"])
    if init is not None:
        o["d_weight"] = o["d_weight"] + init.double().numpy()
    e = assert_parity(g, o)
    k = run_gpu_fwd_bwd(x, lm.LMHEAD_STRATEGY_KEEP_LOGITS, grad_entropy=opts["grad_entropy"],
                        accumulate=opts["accumulate"], d_weight_init=init)
    assert k["status"] == 0
    ek = assert_parity(k, o)
    if i % 4 == 0:
        old = os.environ.get("LMHEAD_BWD_PERSISTENT")
        try:
            for mode in ("0", "2"):
                os.environ["LMHEAD_BWD_PERSISTENT"] = mode
                g2 = run_gpu(x, grad_entropy=opts["grad_entropy"], accumulate=opts["accumulate"],
                             d_weight_init=init)
                for k in ("d_hidden", "d_weight"):
                    assert np.array_equal(g2[k], g[k]), (mode, k)
        finally:
            if old is None:
                os.environ.pop("LMHEAD_BWD_PERSISTENT", None)
            else:
                os.environ["LMHEAD_BWD_PERSISTENT"] = old
    print(i, dict(T=w.T, H=w.H, V=w.V, chunk=w.chunk_size, tau=w.temperature, mask=w.mask),
          opts, e, ek)
