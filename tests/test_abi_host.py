"""Host-side checks of the C ABI (CPU only: no kernel is launched).

The library must load, export every entry point include/lmhead.h declares,
size its workspace without any T x V term, and reject bad arguments
synchronously with the documented status codes.
"""
import ctypes
import os
import re

import pytest

import chunked_lm_head_tcgen05_gb300 as lm

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "lmhead.h")


@pytest.fixture(scope="module")
def lib():
    lm.build()
    return lm.library()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(lmhead_[a-z_]+)\s*\(", text)))


def test_every_declared_symbol_is_exported(lib):
    names = declared_functions()
    assert len(names) >= 10
    for n in names:
        assert hasattr(lib, n), n
    assert set(names) == set(lm._SIGNATURES)


def test_status_strings(lib):
    for code, name in lm.STATUS_NAMES.items():
        assert lm.lmhead_status_string(code).startswith(name)
    assert "unknown" in lm.lmhead_status_string(99)


def test_workspace_size_invalid(lib):
    assert lm.lmhead_workspace_size(0, -1, 64, 10, 8) == 0
    assert lm.lmhead_workspace_size(0, 10, 0, 10, 8) == 0
    assert lm.lmhead_workspace_size(0, 10, 64, 0, 8) == 0
    assert lm.lmhead_workspace_size(0, 10, 64, 10, 0) == 0
    assert lm.lmhead_workspace_size(0, 10, 65, 10, 8) == 0     # H % 64 != 0
    assert lm.lmhead_workspace_size(3, 10, 64, 10, 8) == 0     # unknown op
    assert lm.lmhead_workspace_size(-1, 10, 64, 10, 8) == 0


@pytest.mark.parametrize("T,H,V,c", [(4096, 2560, 151936, 512), (65536, 2560, 151936, 512),
                                     (65536, 4096, 151936, 4096), (200000, 2048, 151936, 4096),
                                     (256, 128, 2048, 64), (1, 64, 1, 1)])
def test_workspace_bounded_by_chunk(lib, T, H, V, c):
    """No T x V term: fwd is O(T (H + splits)), bwd adds at most ~chunk*V bf16."""
    Ta = (T + 127) // 128 * 128
    fwd = lm.lmhead_workspace_size(0, T, H, V, c)
    bwd = lm.lmhead_workspace_size(1, T, H, V, c)
    per_token = 4 + 4 + 2 * H
    assert 0 < fwd <= Ta * (per_token + 16 * 32) + 8 * 256
    dz_bound = 2 * max(c * V, 128 * 256) + 2 * 128 * 256 * max(1, V // 256) * 0
    # the scratch block is T_b x V_b bf16 with T_b * V_b <= chunk * V (+ rounding of one tile)
    assert bwd <= Ta * (per_token + 16) + 2 * (c * V + 128 * 256 + 256 * Ta + 128 * V) + 8 * 256
    assert bwd < 2 * T * V or T * V < 1 << 20
    del dz_bound


def _fake(n):
    return ctypes.c_void_p(n)


def test_forward_argument_errors(lib):
    f = lib.lmhead_logps_fwd
    A = _fake(1 << 20)
    ws = _fake(1 << 24)
    ok_args = dict(T=8, H=64, V=10, tau=1.0, c=4)

    def call(h=A, w=A, y=A, m=None, T=8, H=64, V=10, tau=1.0, c=4, lp=A, en=None, ls=A,
             wsp=ws, wsb=1 << 40):
        return f(h, w, y, m, T, H, V, tau, c, lp, en, ls, wsp, wsb, None)

    assert call(T=-1) == 1
    assert call(H=0) == 1
    assert call(V=0) == 1
    assert call(c=0) == 1
    assert call(tau=0.0) == 1
    assert call(tau=float("nan")) == 1
    assert call(tau=float("inf")) == 1
    assert call(tau=-0.5) == 1
    assert call(H=96) == 2
    assert call(T=0, h=None, w=None, y=None, lp=None, ls=None, wsp=None) == 0   # no-op
    assert call(h=None) == 1
    assert call(w=None) == 1
    assert call(y=None) == 1
    assert call(lp=None) == 1
    assert call(ls=None) == 1
    assert call(wsp=None) == 1
    assert call(h=_fake((1 << 20) + 8)) == 2      # misaligned bf16 matrix
    assert call(wsp=_fake((1 << 24) + 16)) == 2   # workspace not 256-aligned
    assert call(wsb=16) == 3
    del ok_args


def test_backward_argument_errors(lib):
    f = lib.lmhead_logps_bwd
    A = _fake(1 << 20)
    ws = _fake(1 << 24)

    def call(h=A, w=A, y=A, m=None, T=8, H=64, V=10, tau=1.0, c=4, gl=A, ge=None, ls=A, en=None,
             dh=A, dw=A, acc=0, wsp=ws, wsb=1 << 40):
        return f(h, w, y, m, T, H, V, tau, c, gl, ge, ls, en, dh, dw, acc, wsp, wsb, None)

    assert call(T=-3) == 1
    assert call(H=-64) == 1
    assert call(tau=0.0) == 1
    assert call(H=32) == 2
    assert call(dw=None) == 1
    assert call(ls=None) == 1
    assert call(dh=None) == 1
    assert call(ge=A, en=None) == 1          # entropy is required with grad_entropy
    assert call(dh=_fake((1 << 20) + 4)) == 2
    assert call(dw=_fake((1 << 20) + 4)) == 2
    assert call(wsb=100) == 3
    assert call(T=0, acc=1, h=None, y=None, ls=None, dh=None, wsp=None) == 0


@pytest.mark.parametrize("T,H,V,c", [(4096, 2560, 151936, 512), (65536, 4096, 151936, 4096),
                                     (200000, 2048, 151936, 4096), (300, 192, 3001, 64)])
def test_fwd_bwd_workspace_and_plan(lib, T, H, V, c):
    """The single-call workspace covers every strategy and stays chunk-bounded."""
    ws = lm.lmhead_workspace_size(2, T, H, V, c)
    assert ws >= lm.lmhead_workspace_size(0, T, H, V, c)
    assert ws >= lm.lmhead_workspace_size(1, T, H, V, c)
    keep, tb = lm.lmhead_fwd_bwd_keeps_logits(T, H, V, c)
    Vp = (V + 255) // 256 * 256
    assert tb % 256 == 0 and (tb * Vp <= c * V or tb == 256)
    Ta = (T + 127) // 128 * 128
    # logits block (2 B) + per-tile maxima (4 B per 256 columns): no T x V term
    assert ws <= Ta * (8 + 2 * H + 16 * 32 + 16) + 2 * tb * Vp + 4 * tb * (Vp // 256) + \
        2 * (c * V + 128 * 256 + 256 * Ta + 128 * V) + 16 * 256


def test_fwd_bwd_argument_errors(lib):
    f = lib.lmhead_logps_fwd_bwd
    A = _fake(1 << 20)
    ws = _fake(1 << 24)

    def call(h=A, w=A, y=A, m=None, T=8, H=64, V=10, tau=1.0, c=4, gl=A, ge=None, lp=A, en=None,
             ls=A, dh=A, dw=A, acc=0, strat=0, wsp=ws, wsb=1 << 40):
        return f(h, w, y, m, T, H, V, tau, c, gl, ge, lp, en, ls, dh, dw, acc, strat, wsp, wsb,
                 None)

    assert call(strat=3) == 1
    assert call(strat=-1) == 1
    assert call(tau=0.0) == 1
    assert call(H=96) == 2
    assert call(ge=A, en=None) == 1
    assert call(lp=None) == 1
    assert call(dh=_fake((1 << 20) + 4)) == 2
    assert call(wsb=64) == 3
    assert call(T=0, acc=1, h=None, y=None, lp=None, ls=None, dh=None, wsp=None) == 0


def test_plan_is_chunk_bounded(lib):
    """T_b * V_b never exceeds chunk_size * V beyond one tile of rounding."""
    for T, V, c in [(4096, 151936, 512), (65536, 151936, 512), (65536, 151936, 4096),
                    (200000, 151936, 4096), (256, 2048, 64), (300, 3001, 16), (5, 7, 1)]:
        _, tb, vb = lm.lmhead_plan_info(T, 128, V, c)
        # token blocks are whole 256-row pair tiles
        assert tb % 256 == 0 and vb % 256 == 0
        assert tb * vb <= max(c * V, 256 * 256) + 256 * 256 + 256 * tb + 256 * vb, (T, V, c, tb, vb)
        assert tb <= (T + 255) // 256 * 256


def test_shard_argument_errors(lib):
    f = lib.lmhead_logps_fwd_shard
    b = lib.lmhead_logps_bwd_shard
    cmb = lib.lmhead_combine_shards
    A = _fake(1 << 20)
    ws = _fake(1 << 24)

    def fwd(h=A, w=A, y=A, m=None, T=8, H=64, Vs=10, v0=0, Vt=30, tau=1.0, c=4, part=A, wsp=ws,
            wsb=1 << 40):
        return f(h, w, y, m, T, H, Vs, v0, Vt, tau, c, part, wsp, wsb, None)

    def bwd(h=A, w=A, y=A, m=None, T=8, H=64, Vs=10, v0=0, Vt=30, tau=1.0, c=4, gl=A, ge=None,
            ls=A, en=None, dh=A, dw=A, acc=0, wsp=ws, wsb=1 << 40):
        return b(h, w, y, m, T, H, Vs, v0, Vt, tau, c, gl, ge, ls, en, dh, dw, acc, wsp, wsb,
                 None)

    assert fwd(Vs=0) == 1
    assert fwd(v0=-1) == 1
    assert fwd(v0=21) == 1                 # rows past the vocabulary
    assert fwd(Vt=0) == 1
    assert fwd(part=None) == 1
    assert fwd(part=_fake((1 << 20) + 8)) == 2   # statistics need 16-byte alignment
    assert fwd(tau=0.0) == 1
    assert fwd(H=96) == 2
    assert fwd(h=None) == 1
    assert fwd(wsb=16) == 3
    assert fwd(T=0, h=None, w=None, y=None, part=None, wsp=None) == 0
    assert bwd(v0=25) == 1
    assert bwd(Vs=-2) == 1
    assert bwd(ge=A, en=None) == 1
    assert bwd(dw=None) == 1
    assert bwd(wsb=100) == 3
    assert bwd(T=0, acc=1, h=None, y=None, ls=None, dh=None, wsp=None) == 0

    def comb(part=A, n=2, y=A, m=None, T=8, Vt=30, lp=A, en=None, ls=A):
        return cmb(part, n, y, m, T, Vt, lp, en, ls, None)

    assert comb(n=0) == 1
    assert comb(T=-1) == 1
    assert comb(Vt=0) == 1
    assert comb(part=None) == 1
    assert comb(lp=None) == 1
    assert comb(ls=None) == 1
    assert comb(y=None) == 1
    assert comb(part=_fake((1 << 20) + 4)) == 2
    assert comb(T=0, part=None, y=None, lp=None, ls=None) == 0
