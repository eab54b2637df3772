"""Seeded synthetic workloads for the chunked LM-head log-prob + entropy head.

This module only draws random inputs (hidden states, the vocabulary table,
targets, loss masks and per-token cotangents).  It holds none of the head's
arithmetic, imports neither the CUDA binding nor the oracle, and is the one
module that both the GPU path's tests/benchmark and the oracle's tests use.

The shapes and structures follow the workloads the source pages describe:
a Qwen3-4B-shaped head (vocabulary 151,936, hidden 2,560; SkyRL issue #891
"[tx] support long sequence", memory benchmark), batched 4k rows whose prompt
prefix is not scored, a packed 65,536-token row with leading padding and
segment boundaries (tunix PR #2913, pad-first packing on the RL trainer
benchmark), and a 200k-token trace ("Long Sequences (SeCO)" guide).

All draws use a CPU ``torch.Generator`` so that a given seed gives the same
bits wherever it runs on the same software stack.
"""
from dataclasses import dataclass, replace
import math

import torch

SEED_BASE = 20261202


@dataclass(frozen=True)
class Workload:
    name: str
    T: int                      # tokens (rows x sequence, flattened)
    H: int                      # hidden size
    V: int                      # vocabulary size
    temperature: float
    chunk_size: int
    seed: int
    hidden_dist: str = "normal"     # "normal": N(0, 0.02^2); "rms": N(0,1) rows scaled to unit RMS
    weight_std: float = 0.02
    targets: str = "uniform"        # "uniform" or "zipf"
    mask: str = "none"              # "none", "prompt_prefix", "packed_pads", "bernoulli", "all"
    rows: int = 1                   # rows for "prompt_prefix"
    pad_tokens: int = 0             # leading pads for "packed_pads"
    segments: int = 0               # segments for "packed_pads"
    mask_drop: float = 0.0          # P(token unscored) for "bernoulli"
    zipf_s: float = 1.1

    def with_(self, **kw):
        return replace(self, **kw)


WORKLOADS = {
    "tiny": Workload("tiny", T=256, H=128, V=2048, temperature=1.0, chunk_size=64,
                     seed=SEED_BASE + 1),
    "qwen3_4b": Workload("qwen3_4b", T=4096, H=2560, V=151936, temperature=1.0,
                         chunk_size=512, seed=SEED_BASE + 2, hidden_dist="rms"),
    "batched_4k": Workload("batched_4k", T=16 * 4096, H=2560, V=151936, temperature=0.7,
                           chunk_size=512, seed=SEED_BASE + 3, hidden_dist="rms",
                           mask="prompt_prefix", rows=16),
    "packed_long_row": Workload("packed_long_row", T=65536, H=4096, V=151936,
                                temperature=1.0, chunk_size=4096, seed=SEED_BASE + 4,
                                hidden_dist="rms", mask="packed_pads", pad_tokens=4588,
                                segments=8),
    "long_trace": Workload("long_trace", T=200000, H=2048, V=151936, temperature=1.0,
                           chunk_size=4096, seed=SEED_BASE + 5, hidden_dist="rms",
                           targets="zipf", mask="bernoulli", mask_drop=0.2),
}


def _normal_bf16(gen, rows, cols, std, rms_rows=False, block=1 << 24):
    """rows x cols bf16 matrix drawn in fp32 blocks and rounded to nearest even."""
    out = torch.empty((rows, cols), dtype=torch.bfloat16)
    step = max(1, block // max(cols, 1))
    for r0 in range(0, rows, step):
        r1 = min(rows, r0 + step)
        x = torch.randn((r1 - r0, cols), generator=gen, dtype=torch.float32)
        if rms_rows:
            x = x / x.pow(2).mean(dim=1, keepdim=True).sqrt().clamp_min(1e-12)
        elif std != 1.0:
            x = x * std
        out[r0:r1] = x.to(torch.bfloat16)
    return out


def _targets(w, gen):
    if w.targets == "uniform":
        return torch.randint(0, w.V, (w.T,), generator=gen, dtype=torch.int64).to(torch.int32)
    if w.targets == "zipf":
        ranks = torch.arange(1, w.V + 1, dtype=torch.float64)
        weights = ranks.pow(-w.zipf_s)
        cdf = torch.cumsum(weights / weights.sum(), 0)
        u = torch.rand((w.T,), generator=gen, dtype=torch.float64)
        r = torch.searchsorted(cdf, u).clamp_max(w.V - 1)
        perm = torch.randperm(w.V, generator=gen)
        return perm[r].to(torch.int32)
    raise ValueError(w.targets)


def _mask(w, gen, extras):
    """uint8 [T], 1 = scored, or None when every token is scored."""
    if w.mask == "none":
        return None
    m = torch.ones(w.T, dtype=torch.uint8)
    if w.mask == "all":          # every token unscored (degenerate case)
        return torch.zeros(w.T, dtype=torch.uint8)
    if w.mask == "prompt_prefix":
        L = w.T // w.rows
        frac = 0.10 + 0.40 * torch.rand((w.rows,), generator=gen, dtype=torch.float64)
        for r in range(w.rows):
            m[r * L: r * L + int(math.floor(float(frac[r]) * L))] = 0
        return m
    if w.mask == "packed_pads":
        real = w.T - w.pad_tokens
        m[:w.pad_tokens] = 0
        # random composition of `real` into `segments` positive lengths
        cuts = torch.randperm(real - 1, generator=gen)[: w.segments - 1] + 1
        bounds = [0] + sorted(int(c) for c in cuts) + [real]
        seg_ids = torch.zeros(w.T, dtype=torch.int32)
        for s in range(w.segments):
            a, b = w.pad_tokens + bounds[s], w.pad_tokens + bounds[s + 1]
            seg_ids[a:b] = s + 1
            m[b - 1] = 0   # the next token lies in another segment
        extras["segment_ids"] = seg_ids
        return m
    if w.mask == "bernoulli":
        drop = torch.rand((w.T,), generator=gen, dtype=torch.float64) < w.mask_drop
        m[drop] = 0
        return m
    raise ValueError(w.mask)


def make_inputs(w, with_grads=True):
    """Draw one workload.  Returns a dict of CPU tensors:

    hidden [T,H] bf16, weight [V,H] bf16, targets [T] int32, loss_mask [T]
    uint8 or None, grad_logp / grad_entropy [T] fp32 (zero where unscored),
    plus the workload's temperature and chunk_size.
    """
    gen = torch.Generator().manual_seed(w.seed)
    if w.hidden_dist == "rms":
        hidden = _normal_bf16(gen, w.T, w.H, 1.0, rms_rows=True)
    else:
        hidden = _normal_bf16(gen, w.T, w.H, 0.02)
    weight = _normal_bf16(gen, w.V, w.H, w.weight_std)
    targets = _targets(w, gen)
    extras = {}
    mask = _mask(w, gen, extras)
    out = dict(hidden=hidden, weight=weight, targets=targets, loss_mask=mask,
               temperature=w.temperature, chunk_size=w.chunk_size, workload=w, **extras)
    if with_grads:
        gl = torch.randn((w.T,), generator=gen, dtype=torch.float32)
        ge = torch.randn((w.T,), generator=gen, dtype=torch.float32)
        if mask is not None:
            gl = gl * mask.to(torch.float32)
            ge = ge * mask.to(torch.float32)
        out["grad_logp"] = gl
        out["grad_entropy"] = ge
    return out


def scored_count(inputs):
    m = inputs["loss_mask"]
    return int(inputs["hidden"].shape[0]) if m is None else int(m.to(torch.int64).sum())


def bf16_bits(t):
    """Raw bit patterns of a bf16 tensor as a numpy uint16 array (no rounding)."""
    import numpy as np
    return t.contiguous().view(torch.int16).numpy().view(np.uint16)
