"""The C-ABI library: it loads, exports every function include/*.h declares, and
rejects bad arguments on the host before touching the GPU (runs without one)."""
import ctypes
import glob
import os
import re

import pytest

import causal_gqa_attention_attn_gb300 as ga
from causal_gqa_attention_attn_gb300 import build as gbuild

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def L():
    gbuild.build()
    return ga.lib()


def _declared_functions():
    names = set()
    for h in glob.glob(os.path.join(ROOT, "include", "*.h")):
        text = re.sub(r"/\*.*?\*/", "", open(h).read(), flags=re.S)
        for m in re.finditer(r"^\s*[A-Za-z_][\w\s\*]*?\b([A-Za-z_]\w*)\s*\(", text, flags=re.M):
            if m.group(1) not in ("if", "defined"):
                names.add(m.group(1))
    return sorted(names)


def test_every_declared_symbol_is_exported(L):
    names = _declared_functions()
    assert "attn_bwd" in names and "attn_fwd_lse" in names and "rope_bwd_inplace" in names
    for n in names:
        assert hasattr(L, n), f"{n} declared in include/ but not exported"


def test_status_strings(L):
    for code, name in ((0, "GQA_OK"), (1, "GQA_ERR_INVALID_ARG"), (2, "GQA_ERR_UNSUPPORTED"),
                       (3, "GQA_ERR_CUDA"), (4, "GQA_ERR_DEVICE_TIMEOUT"),
                       (5, "GQA_ERR_DEVICE_CHECK")):
        assert L.gqa_status_str(code).decode() == name


def test_workspace_size(L):
    a = L.attn_bwd_workspace_bytes(4096, 32, 8, 128)
    b = L.attn_bwd_workspace_bytes(16384, 32, 8, 128)
    assert a % 256 == 0 and b % 256 == 0
    assert b > a >= 4096 * 32 * 4 + 4096 * 8 * 128 * 4     # D + K^T of the tensor-core path
    odd = L.attn_bwd_workspace_bytes(4096, 32, 8, 100)      # CUDA-core only: D and tile minima
    assert 4096 * 32 * 4 <= odd < a
    assert L.attn_bwd_workspace_bytes(0, 4, 2, 32) >= 0


FAKE = 0x10000  # a 16-byte-aligned non-null address; never dereferenced (checks fail first)


def _bwd(L, S=128, H=4, Hk=2, d=32, scale=0.17, ws_bytes=None, ptrs=None, fn="attn_bwd"):
    p = [FAKE] * 10 if ptrs is None else ptrs
    if ws_bytes is None:
        ws_bytes = L.attn_bwd_workspace_bytes(S, H, Hk, d)
    return getattr(L, fn)(*p[:9], S, H, Hk, d, scale, p[9], ws_bytes, None)


@pytest.mark.parametrize("fn", ["attn_bwd", "attn_bwd_simt", "attn_bwd_short"])
def test_bwd_rejects_bad_arguments(L, fn):
    assert _bwd(L, H=6, Hk=4, fn=fn) == 1                       # heads not a multiple
    assert _bwd(L, Hk=0, fn=fn) == 1
    assert _bwd(L, S=-1, fn=fn) == 1
    assert _bwd(L, d=30, fn=fn) == 1                            # not a multiple of 4
    assert _bwd(L, d=132, fn=fn) == 2                           # no kernel above 128
    assert _bwd(L, scale=float("nan"), fn=fn) == 1
    assert _bwd(L, ws_bytes=16, fn=fn) == 1                     # workspace too small
    assert "workspace" in L.gqa_last_error().decode()
    for k in range(10):
        p = [FAKE] * 10
        p[k] = None
        assert _bwd(L, ptrs=p, fn=fn) == 1
        p[k] = FAKE + 4                                         # misaligned
        assert _bwd(L, ptrs=p, fn=fn) == 1
    assert _bwd(L, S=1 << 20, H=64, Hk=8, d=128, fn=fn) == 2   # 2^33 elements
    assert _bwd(L, S=0, fn=fn) == 0                             # empty: no-op


def test_short_path_limits_and_switch(L):
    """attn_bwd_short takes seq_len <= 2048 with bounded tile work and refuses
    the rest before any launch; the workspace query covers its partial sums;
    gqa_set_short_path returns the previous setting."""
    assert _bwd(L, S=4096, H=4, Hk=2, d=32, fn="attn_bwd_short") == 2
    assert _bwd(L, S=1024, H=32, Hk=8, d=128, fn="attn_bwd_short") == 2
    assert "short path" in L.gqa_last_error().decode()
    # 16 x 17 / 2 tiles x 1024 x 4 heads x 32: partial dQ, dK, dV of every cell
    cells = 16 * 17 // 2 * 4
    assert L.attn_bwd_workspace_bytes(512, 4, 2, 32) >= 3 * cells * 32 * 32 * 4 + cells * 32 * 4
    # head_dim 100 is padded to 128 (8 x 9 / 2 tiles x 4 heads)
    assert L.attn_bwd_workspace_bytes(256, 4, 2, 100) >= 3 * 144 * 32 * 128 * 4
    assert L.gqa_set_short_path(0) == 1
    assert L.gqa_set_short_path(1) == 0
    assert L.gqa_set_short_path(1) == 1


def test_workspace_reserves_key_major_parts(L):
    """Where the key-major grid is under one wave (one CTA per SM) its walk
    is split into up to four parts whose partial dK / dV live in the
    workspace: [2][parts][S][Hk*d] fp32, sized for devices of up to 192 SMs,
    so the size depends on the shape alone. Deep grids (the 16k workload)
    reserve nothing for them, only the operand copies."""
    S, H, Hk, d = 2048, 16, 4, 64           # 64 key-major CTAs: four parts
    parts = 2 * 4 * S * Hk * d * 4
    qt = Hk * d * (S * (H // Hk)) * 4       # Q^T (and dO^T) copies
    assert L.attn_bwd_workspace_bytes(S, H, Hk, d) >= parts + 2 * qt
    S, H, Hk, d = 16384, 32, 8, 128         # 1024 key-major CTAs: no split
    # Q^T, dO^T, K^T, and at d = 128 K' (K's rows permuted within 64-key chunks)
    copies = 2 * Hk * d * (S * (H // Hk)) * 4 + 2 * Hk * d * S * 4
    one_part = 2 * S * Hk * d * 4                                # what a single part would add
    assert copies <= L.attn_bwd_workspace_bytes(S, H, Hk, d) < copies + one_part // 2


def test_fwd_and_rope_reject_bad_arguments(L):
    fwd = lambda S=64, H=4, Hk=2, d=32, s=0.2: L.attn_fwd_lse(  # noqa: E731
        FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, S, H, Hk, d, s, None)
    assert fwd(H=5) == 1 and fwd(d=136) == 2 and fwd(S=-3) == 1 and fwd(S=0) == 0
    assert L.attn_fwd_lse(FAKE, None, FAKE, FAKE, FAKE, FAKE, 64, 4, 2, 32, 0.2, None) == 1
    rope = L.rope_bwd_inplace
    assert rope(FAKE, 16, 4, 6, 0, 10000.0, None) == 1          # head_dim not a multiple of 4
    assert rope(FAKE, 16, 4, 8, -1, 10000.0, None) == 1
    assert rope(FAKE, 16, 4, 8, 0, 0.0, None) == 1
    assert rope(None, 16, 4, 8, 0, 10000.0, None) == 1
    assert rope(FAKE + 8, 16, 4, 8, 0, 10000.0, None) == 1
    assert rope(FAKE, 0, 4, 8, 0, 10000.0, None) == 0


def test_fused_rope_rejects_bad_arguments(L):
    def call(S=128, H=4, Hk=2, d=32, pos=0, base=10000.0, ws_bytes=None, ptrs=None):
        p = [FAKE] * 10 if ptrs is None else ptrs
        if ws_bytes is None:
            ws_bytes = L.attn_bwd_workspace_bytes(S, H, Hk, d)
        return L.attn_bwd_rope(*p[:9], S, H, Hk, d, 0.17, pos, base, p[9], ws_bytes, None)
    assert call(pos=-1) == 1
    assert call(base=0.0) == 1 and call(base=-2.0) == 1 and call(base=float("inf")) == 1
    assert call(H=6, Hk=4) == 1 and call(d=30) == 1 and call(d=132) == 2
    assert call(ws_bytes=16) == 1
    p = [FAKE] * 10
    p[6] = None                                                  # dQ
    assert call(ptrs=p) == 1
    assert call(S=0) == 0


def test_given_o_rejects_bad_arguments(L):
    def call(S=128, H=4, Hk=2, d=32, ptrs=None, ws_bytes=None):
        p = [FAKE] * 11 if ptrs is None else ptrs
        if ws_bytes is None:
            ws_bytes = L.attn_bwd_workspace_bytes(S, H, Hk, d)
        return L.attn_bwd_o(*p[:10], S, H, Hk, d, 0.17, p[10], ws_bytes, None)
    for k in range(11):
        p = [FAKE] * 11
        p[k] = None
        assert call(ptrs=p) == 1
        p[k] = FAKE + 4
        assert call(ptrs=p) == 1
    assert call(H=6, Hk=4) == 1 and call(d=132) == 2 and call(ws_bytes=16) == 1
    assert call(S=0) == 0


def test_tensor_core_forward_rejects_bad_arguments(L):
    def call(S=128, H=4, Hk=2, d=32, s=0.2, ptrs=None, ws_bytes=None):
        p = [FAKE] * 7 if ptrs is None else ptrs
        if ws_bytes is None:
            ws_bytes = L.attn_fwd_workspace_bytes(S, H, Hk, d)
        return L.attn_fwd(*p[:6], S, H, Hk, d, s, p[6], ws_bytes, None)
    assert call(H=5) == 1 and call(d=136) == 2 and call(S=-3) == 1 and call(S=0) == 0
    assert call(s=float("inf")) == 1 and call(ws_bytes=16) == 1
    for k in range(7):
        p = [FAKE] * 7
        p[k] = None
        assert call(ptrs=p) == 1
    # tensor-core shapes need the V^T copy; other head dims only the header
    assert L.attn_fwd_workspace_bytes(4096, 32, 8, 128) >= 256 + 8 * 128 * 4096 * 4
    assert L.attn_fwd_workspace_bytes(4096, 32, 8, 100) == 256


def test_decode_backward_rejects_bad_arguments(L):
    def call(Lh=64, H=4, Hk=2, d=32, s=0.2, ptrs=None, ws_bytes=None):
        p = [FAKE] * 10 if ptrs is None else ptrs
        if ws_bytes is None:
            ws_bytes = L.attn_decode_bwd_workspace_bytes(Lh, H, Hk, d)
        return L.attn_decode_bwd(*p[:9], Lh, H, Hk, d, s, p[9], ws_bytes, None)
    assert call(H=5) == 1 and call(Hk=0) == 1 and call(Lh=-1) == 1 and call(Lh=0) == 0
    assert call(d=30) == 1 and call(d=36) == 2 and call(d=160) == 2 and call(s=float("nan")) == 1
    assert call(ws_bytes=16) == 1
    for k in range(10):
        p = [FAKE] * 10
        p[k] = None
        assert call(ptrs=p) == 1
    p = [FAKE] * 10
    p[3] = FAKE + 4                                   # probs not 16-byte aligned
    assert call(ptrs=p) == 1
    # per-block partial sums of D and of d_q, after the status header
    assert L.attn_decode_bwd_workspace_bytes(16384, 32, 8, 128) >= 256 + 512 * 32 * 128 * 4


def test_binding_fails_loudly_without_library(monkeypatch, tmp_path):
    monkeypatch.setattr(ga, "_libs", {})
    monkeypatch.setattr(ga, "_LIB_PATHS", {"release": str(tmp_path / "missing.so"),
                                            "checks": str(tmp_path / "missing_checks.so")})
    with pytest.raises(ga.GqaError):
        ga.lib()
    with pytest.raises(ga.GqaError):
        ga.lib("checks")


def test_checks_library_exports_every_symbol():
    """The debug build (-DGQA_CHECKS) exports the same C ABI as the release
    build, and both name the debug-only status code."""
    gbuild.build()
    for variant in ("release", "checks"):
        L = ga.lib(variant)
        for name in _declared_functions():
            assert hasattr(L, name), (variant, name)
        assert L.gqa_status_str(5) == b"GQA_ERR_DEVICE_CHECK"
