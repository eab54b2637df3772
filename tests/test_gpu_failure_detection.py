"""Failure detection without a GPU fault: the bounded mbarrier wait that every
GEMM pipeline stage uses runs out on a barrier nothing arrives on (a short
limit), reports LMHEAD_ERR_DEVICE_TIMEOUT through the status word, frees its
tensor memory, and the context stays usable for a normal call afterwards."""
import time

import numpy as np
import pytest
import torch

import chunked_lm_head_tcgen05_gb300 as lm
from chunked_lm_head_tcgen05_gb300 import workloads as W

from gpu_helpers import assert_parity, ensure_built, run_gpu, run_oracle

pytestmark = pytest.mark.gpu


def test_bounded_wait_times_out_and_context_survives():
    ensure_built()
    ws = torch.empty(256, dtype=torch.uint8, device="cuda")
    t0 = time.perf_counter()
    assert lm.lmhead_selftest_bounded_wait(ws, 50) == 0
    assert lm.lmhead_read_device_status(ws) == 5          # LMHEAD_ERR_DEVICE_TIMEOUT
    assert time.perf_counter() - t0 < 10.0
    assert torch.cuda.synchronize() is None
    x = W.make_inputs(W.WORKLOADS["tiny"])
    g = run_gpu(x)
    assert g["fwd_status"] == 0 and g["bwd_status"] == 0
    assert_parity(g, run_oracle(x))


def test_selftest_argument_errors():
    ensure_built()
    ws = torch.empty(256, dtype=torch.uint8, device="cuda")
    assert lm.lmhead_selftest_bounded_wait(ws, 0) == 1
    assert lm.lmhead_selftest_bounded_wait(ws, 20000) == 1
    big = torch.empty(512, dtype=torch.uint8, device="cuda")
    assert lm.lmhead_selftest_bounded_wait(big[1:], 10) == 2     # not 256-byte aligned
