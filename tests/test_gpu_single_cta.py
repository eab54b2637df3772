"""The single-CTA tile path (128 x 256 tiles, LMHEAD_CTA_PAIR=0) against the
oracle.  The switch is read once per process, so the cases run in a child
process: forward + backward on ragged and masked shapes, the log-prob-only
backward, and the single-call path with kept logits."""
import os
import subprocess
import sys
import textwrap

import pytest

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

CHILD = textwrap.dedent("""
    import sys
    sys.path.insert(0, {tests!r})
    import numpy as np
    import chunked_lm_head_tcgen05_gb300 as lm
    from chunked_lm_head_tcgen05_gb300 import workloads as W
    from gpu_helpers import assert_parity, run_gpu, run_gpu_fwd_bwd, run_oracle
    tiny = W.WORKLOADS["tiny"]
    cases = [
        dict(T=333, H=192, V=3001, chunk_size=64, temperature=0.7, mask="bernoulli", mask_drop=0.3),
        dict(T=700, H=256, V=5000, chunk_size=128, temperature=0.5, mask="prompt_prefix", rows=2),
        dict(T=257, H=320, V=1025, chunk_size=7, temperature=1.3, mask="none"),
    ]
    for c in cases:
        x = W.make_inputs(tiny.with_(hidden_dist="rms", weight_std=0.05, seed=3, **c))
        g = run_gpu(x)
        assert g["fwd_status"] == 0 and g["bwd_status"] == 0
        print(c["T"], assert_parity(g, run_oracle(x)))
    x = W.make_inputs(tiny.with_(T=300, H=128, V=1500, chunk_size=50, temperature=0.7,
                                 mask="bernoulli", mask_drop=0.2, hidden_dist="rms", seed=4))
    assert_parity(run_gpu(x, grad_entropy=False), run_oracle(x, grad_entropy=False))
    g = run_gpu_fwd_bwd(x, strategy=lm.LMHEAD_STRATEGY_KEEP_LOGITS)
    assert_parity(g, run_oracle(x))
    print("OK")
""")


def test_single_cta_tiles_match_the_oracle():
    env = dict(os.environ, LMHEAD_CTA_PAIR="0")
    code = CHILD.format(tests=os.path.join(ROOT, "tests"))
    r = subprocess.run([sys.executable, "-c", code], cwd=ROOT, env=env, capture_output=True,
                       text=True, timeout=900)
    print(r.stdout[-3000:], r.stderr[-3000:])
    assert r.returncode == 0 and r.stdout.strip().endswith("OK")
