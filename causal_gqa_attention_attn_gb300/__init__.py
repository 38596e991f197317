"""Causal grouped-query attention backward from a saved log-sum-exp on GB300.

Thin ctypes binding over ``libgqa_attn.so`` (C ABI in ``include/gqa_attn.h``).
The functions here only check tensor metadata and pass device pointers and the
current CUDA stream through; every step of the computation runs in the
library's CUDA kernels. PyTorch provides device memory and streams.

If the shared library has not been built, importing works but the first call
raises :class:`GqaError`; build it with ``__graft_entry__.build()`` (or
``python -m causal_gqa_attention_attn_gb300.build``). There is no fallback.

``checks_build()`` routes the calls made inside its ``with`` block through
``libgqa_attn_checks.so``, the debug build of the same sources with
device-side checks (seg precondition, kernel indices) that report through
the workspace status word (``read_device_status`` raises GQA_ERR_DEVICE_CHECK).
"""
from __future__ import annotations

import contextlib
import ctypes
import os

__all__ = ["GqaError", "lib", "lib_path", "attn_fwd_lse", "attn_bwd", "attn_bwd_simt",
           "rope_bwd_inplace", "workspace_bytes", "read_device_status", "n_pairs_from_seg",
           "profile_events", "profile_stage_name", "launch_count", "attn_bwd_noalloc",
           "attn_fwd", "attn_bwd_rope", "attn_bwd_o", "attn_decode_bwd", "attn_bwd_short",
           "set_short_path", "checks_build"]

_HERE = os.path.dirname(os.path.abspath(__file__))
_LIB_PATH = os.path.join(_HERE, "libgqa_attn.so")
_LIB_PATHS = {"release": _LIB_PATH, "checks": os.path.join(_HERE, "libgqa_attn_checks.so")}
_libs: dict = {}
_active = "release"

GQA_OK = 0
_STATUS = {0: "GQA_OK", 1: "GQA_ERR_INVALID_ARG", 2: "GQA_ERR_UNSUPPORTED", 3: "GQA_ERR_CUDA",
           4: "GQA_ERR_DEVICE_TIMEOUT", 5: "GQA_ERR_DEVICE_CHECK"}


class GqaError(RuntimeError):
    def __init__(self, status: int, message: str):
        super().__init__(f"{_STATUS.get(status, status)}: {message}")
        self.status = status


def lib_path() -> str:
    return _LIB_PATH


def lib(variant: str | None = None) -> ctypes.CDLL:
    """The loaded library (declares the argument types of every entry point):
    the release build, or inside ``checks_build()`` the debug build; an
    explicit ``variant`` ("release" or "checks") picks one."""
    variant = _active if variant is None else variant
    if variant in _libs:
        return _libs[variant]
    path = _LIB_PATHS[variant]
    if not os.path.exists(path):
        raise GqaError(3, f"{path} is missing: build it first (__graft_entry__.build())")
    L = ctypes.CDLL(path)
    P, I, F, Z = ctypes.c_void_p, ctypes.c_int, ctypes.c_float, ctypes.c_size_t
    L.attn_fwd_lse.argtypes = [P, P, P, P, P, P, I, I, I, I, F, P]
    L.attn_fwd.argtypes = [P, P, P, P, P, P, I, I, I, I, F, P, Z, P]
    L.attn_fwd_workspace_bytes.argtypes = [I, I, I, I]
    L.attn_fwd_workspace_bytes.restype = Z
    L.attn_decode_bwd.argtypes = [P, P, P, P, P, P, P, P, P, I, I, I, I, F, P, Z, P]
    L.attn_decode_bwd_workspace_bytes.argtypes = [I, I, I, I]
    L.attn_decode_bwd_workspace_bytes.restype = Z
    bwd_args = [P, P, P, P, P, P, P, P, P, I, I, I, I, F, P, Z, P]
    L.attn_bwd.argtypes = bwd_args
    L.attn_bwd_simt.argtypes = bwd_args
    L.attn_bwd_short.argtypes = bwd_args
    L.gqa_set_short_path.argtypes = [I]
    L.gqa_set_short_path.restype = ctypes.c_int
    L.attn_bwd_rope.argtypes = [P, P, P, P, P, P, P, P, P, I, I, I, I, F, I, F, P, Z, P]
    L.attn_bwd_o.argtypes = [P, P, P, P, P, P, P, P, P, P, I, I, I, I, F, P, Z, P]
    L.attn_bwd_noalloc.argtypes = [P, P, P, P, P, P, P, P, P, I, I, I, I, F, P]
    L.attn_bwd_noalloc.restype = ctypes.c_int
    L.rope_bwd_inplace.argtypes = [P, I, I, I, I, F, P]
    L.attn_bwd_workspace_bytes.argtypes = [I, I, I, I]
    L.attn_bwd_workspace_bytes.restype = Z
    L.attn_read_device_status.argtypes = [P, P]
    L.gqa_status_str.argtypes = [I]
    L.gqa_status_str.restype = ctypes.c_char_p
    L.gqa_profile_events.argtypes = [P, P]
    L.gqa_profile_events.restype = None
    L.gqa_profile_stage_name.argtypes = []
    L.gqa_profile_stage_name.restype = ctypes.c_char_p
    L.gqa_wait_selftest.argtypes = [P, Z, ctypes.c_longlong, P]
    L.gqa_wait_selftest.restype = ctypes.c_int
    L.gqa_grid_barrier_selftest.argtypes = [P, Z, ctypes.c_longlong, P]
    L.gqa_grid_barrier_selftest.restype = ctypes.c_int
    L.gqa_launch_count.argtypes = []
    L.gqa_launch_count.restype = ctypes.c_ulonglong
    L.gqa_last_error.argtypes = []
    L.gqa_last_error.restype = ctypes.c_char_p
    for name in ("attn_fwd_lse", "attn_fwd", "attn_bwd", "attn_bwd_simt", "attn_bwd_short",
                 "attn_bwd_rope", "attn_bwd_o",
                 "attn_decode_bwd", "rope_bwd_inplace", "attn_read_device_status"):
        getattr(L, name).restype = ctypes.c_int
    _libs[variant] = L
    return L


@contextlib.contextmanager
def checks_build():
    """Inside the block, this module's calls go to libgqa_attn_checks.so (the
    -DGQA_CHECKS debug build); yields that library. Not thread-safe: switch
    only between calls."""
    global _active
    prev = _active
    L = lib("checks")
    _active = "checks"
    try:
        yield L
    finally:
        _active = prev


def _check(status: int):
    if status != GQA_OK:
        raise GqaError(status, lib().gqa_last_error().decode())


def _torch():
    import torch
    return torch


def _ptr(t, name, dtypes):
    if t is None:
        return None
    torch = _torch()
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if t.device.type != "cuda":
        raise ValueError(f"{name} must be a CUDA tensor")
    if t.dtype not in dtypes:
        raise TypeError(f"{name} has dtype {t.dtype}, expected one of {dtypes}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    return t.data_ptr()


def _stream(stream):
    torch = _torch()
    s = torch.cuda.current_stream() if stream is None else stream
    return s.cuda_stream


def _f32(t, name):
    return _ptr(t, name, (_torch().float32,))


def _seg(t):
    torch = _torch()
    return _ptr(t, "seg", tuple(x for x in (torch.int32, getattr(torch, "uint32", None)) if x))


def workspace_bytes(seq_len, n_heads, n_kv_heads, head_dim) -> int:
    return int(lib().attn_bwd_workspace_bytes(seq_len, n_heads, n_kv_heads, head_dim))


def attn_fwd_lse(Q, K, V, seg, n_heads, n_kv_heads, head_dim, scale, O=None, LSE=None,
                 stream=None):
    """Forward attention: returns (O, LSE); O [S, H*d], LSE [S, H] fp32."""
    torch = _torch()
    S = Q.shape[0]
    O = torch.empty((S, n_heads * head_dim), device=Q.device, dtype=torch.float32) if O is None else O
    LSE = torch.empty((S, n_heads), device=Q.device, dtype=torch.float32) if LSE is None else LSE
    _check(lib().attn_fwd_lse(_f32(Q, "Q"), _f32(K, "K"), _f32(V, "V"), _seg(seg), _f32(O, "O"),
                              _f32(LSE, "LSE"), S, n_heads, n_kv_heads, head_dim, float(scale),
                              _stream(stream)))
    return O, LSE


def attn_fwd(Q, K, V, seg, n_heads, n_kv_heads, head_dim, scale, O=None, LSE=None,
             workspace=None, stream=None):
    """Forward attention on tensor cores where the shape allows: returns (O, LSE).
    Pass `workspace` (attn_fwd_workspace_bytes) to reuse it or to read the
    device status afterwards (read_device_status)."""
    torch = _torch()
    S = Q.shape[0]
    if O is None:
        O = torch.empty(S, n_heads * head_dim, device=Q.device, dtype=torch.float32)
    if LSE is None:
        LSE = torch.empty(S, n_heads, device=Q.device, dtype=torch.float32)
    need = int(lib().attn_fwd_workspace_bytes(S, n_heads, n_kv_heads, head_dim))
    if workspace is None:
        workspace = torch.empty(need, device=Q.device, dtype=torch.uint8)
    _check(lib().attn_fwd(_f32(Q, "Q"), _f32(K, "K"), _f32(V, "V"), _seg(seg), _f32(O, "O"),
                          _f32(LSE, "LSE"), S, n_heads, n_kv_heads, head_dim, float(scale),
                          _ptr(workspace, "workspace", (torch.uint8,)), workspace.numel(),
                          _stream(stream)))
    return O, LSE


def attn_decode_bwd(q, k_hist, v_hist, probs, d_out, n_heads, n_kv_heads, head_dim, scale,
                    d_q=None, d_k_hist=None, d_v_hist=None, d_scores=None, workspace=None,
                    stream=None):
    """Decode-style backward from saved probabilities (one query per head vs the
    key history): returns (d_scores, d_q, d_k_hist, d_v_hist). d_q, d_k_hist,
    d_v_hist accumulate into the tensors passed (zeros when omitted); d_scores
    is overwritten. q, d_out [n_heads*head_dim]; k_hist, v_hist
    [history_len, n_kv_heads*head_dim]; probs [n_heads, history_len]."""
    torch = _torch()
    L = k_hist.shape[0]
    dev = k_hist.device
    if d_q is None:
        d_q = torch.zeros(n_heads * head_dim, device=dev, dtype=torch.float32)
    if d_k_hist is None:
        d_k_hist = torch.zeros(L, n_kv_heads * head_dim, device=dev, dtype=torch.float32)
    if d_v_hist is None:
        d_v_hist = torch.zeros(L, n_kv_heads * head_dim, device=dev, dtype=torch.float32)
    if d_scores is None:
        d_scores = torch.empty(n_heads, L, device=dev, dtype=torch.float32)
    need = int(lib().attn_decode_bwd_workspace_bytes(L, n_heads, n_kv_heads, head_dim))
    if workspace is None:
        workspace = torch.empty(need, device=dev, dtype=torch.uint8)
    _check(lib().attn_decode_bwd(_f32(q, "q"), _f32(k_hist, "k_hist"), _f32(v_hist, "v_hist"),
                                 _f32(probs, "probs"), _f32(d_out, "d_out"),
                                 _f32(d_scores, "d_scores"), _f32(d_q, "d_q"),
                                 _f32(d_k_hist, "d_k_hist"), _f32(d_v_hist, "d_v_hist"), L,
                                 n_heads, n_kv_heads, head_dim, float(scale),
                                 _ptr(workspace, "workspace", (torch.uint8,)), workspace.numel(),
                                 _stream(stream)))
    return d_scores, d_q, d_k_hist, d_v_hist


def _bwd(fn, Q, K, V, dO, LSE, seg, dQ, dK, dV, n_heads, n_kv_heads, head_dim, scale,
         workspace, stream):
    torch = _torch()
    S = Q.shape[0]
    need = workspace_bytes(S, n_heads, n_kv_heads, head_dim)
    if workspace is None:
        workspace = torch.empty(need, device=Q.device, dtype=torch.uint8)
    _check(fn(_f32(Q, "Q"), _f32(K, "K"), _f32(V, "V"), _f32(dO, "dO"), _f32(LSE, "LSE"),
              _seg(seg), _f32(dQ, "dQ"), _f32(dK, "dK"), _f32(dV, "dV"), S, n_heads, n_kv_heads,
              head_dim, float(scale), _ptr(workspace, "workspace", (torch.uint8,)),
              workspace.numel(), _stream(stream)))
    return workspace


def attn_bwd(Q, K, V, dO, LSE, seg, dQ, dK, dV, n_heads, n_kv_heads, head_dim, scale,
             workspace=None, stream=None):
    """Backward from a saved LSE; accumulates into dQ, dK, dV (+=). Returns the
    workspace used (a uint8 device tensor; pass it back in to reuse it)."""
    return _bwd(lib().attn_bwd, Q, K, V, dO, LSE, seg, dQ, dK, dV, n_heads, n_kv_heads,
                head_dim, scale, workspace, stream)


def attn_bwd_o(Q, K, V, dO, O, LSE, seg, dQ, dK, dV, n_heads, n_kv_heads, head_dim, scale,
               workspace=None, stream=None):
    """:func:`attn_bwd` given the forward output O: D = rowsum(dO * O) replaces
    the D pass. Returns the workspace used."""
    torch = _torch()
    S = Q.shape[0]
    if workspace is None:
        workspace = torch.empty(workspace_bytes(S, n_heads, n_kv_heads, head_dim),
                                device=Q.device, dtype=torch.uint8)
    _check(lib().attn_bwd_o(
        _f32(Q, "Q"), _f32(K, "K"), _f32(V, "V"), _f32(dO, "dO"), _f32(O, "O"), _f32(LSE, "LSE"),
        _seg(seg), _f32(dQ, "dQ"), _f32(dK, "dK"), _f32(dV, "dV"), S, n_heads, n_kv_heads,
        head_dim, float(scale), _ptr(workspace, "workspace", (torch.uint8,)), workspace.numel(),
        _stream(stream)))
    return workspace


def attn_bwd_rope(Q, K, V, dO, LSE, seg, dQ, dK, dV, n_heads, n_kv_heads, head_dim, scale,
                  pos_offset=0, base=10000.0, workspace=None, stream=None):
    """:func:`attn_bwd` with the interleaved RoPE backward fused into the final
    writes: dQ += R^T(attention dQ), dK += R^T(attention dK), dV += attention dV.
    Returns the workspace used."""
    torch = _torch()
    S = Q.shape[0]
    if workspace is None:
        workspace = torch.empty(workspace_bytes(S, n_heads, n_kv_heads, head_dim),
                                device=Q.device, dtype=torch.uint8)
    _check(lib().attn_bwd_rope(
        _f32(Q, "Q"), _f32(K, "K"), _f32(V, "V"), _f32(dO, "dO"), _f32(LSE, "LSE"), _seg(seg),
        _f32(dQ, "dQ"), _f32(dK, "dK"), _f32(dV, "dV"), S, n_heads, n_kv_heads, head_dim,
        float(scale), int(pos_offset), float(base), _ptr(workspace, "workspace", (torch.uint8,)),
        workspace.numel(), _stream(stream)))
    return workspace


def attn_bwd_simt(Q, K, V, dO, LSE, seg, dQ, dK, dV, n_heads, n_kv_heads, head_dim, scale,
                  workspace=None, stream=None):
    """Same as :func:`attn_bwd`, on CUDA cores only (exact fp32 products)."""
    return _bwd(lib().attn_bwd_simt, Q, K, V, dO, LSE, seg, dQ, dK, dV, n_heads, n_kv_heads,
                head_dim, scale, workspace, stream)


def attn_bwd_short(Q, K, V, dO, LSE, seg, dQ, dK, dV, n_heads, n_kv_heads, head_dim, scale,
                   workspace=None, stream=None):
    """Same as :func:`attn_bwd`, as one cooperative launch on CUDA cores for
    short sequences (seq_len <= 2048 and bounded tile work; GqaError with
    GQA_ERR_UNSUPPORTED beyond). Returns the workspace used."""
    return _bwd(lib().attn_bwd_short, Q, K, V, dO, LSE, seg, dQ, dK, dV, n_heads, n_kv_heads,
                head_dim, scale, workspace, stream)


def set_short_path(enable: bool) -> bool:
    """Process-wide: let attn_bwd / attn_bwd_o / attn_bwd_rope use the
    single-launch short path for the shapes it accepts (default True).
    Returns the previous setting."""
    return bool(lib().gqa_set_short_path(1 if enable else 0))


def attn_bwd_noalloc(Q, K, V, dO, LSE, seg, dQ, dK, dV, n_heads, n_kv_heads, head_dim, scale,
                     stream=None):
    """Same as :func:`attn_bwd_simt`, for callers that cannot allocate device
    memory: no workspace argument; the library's fixed 4 MiB scratch array is
    used instead (seq_len * n_heads up to about 1M; overlapping calls race)."""
    _check(lib().attn_bwd_noalloc(_f32(Q, "Q"), _f32(K, "K"), _f32(V, "V"), _f32(dO, "dO"),
                                  _f32(LSE, "LSE"), _seg(seg), _f32(dQ, "dQ"), _f32(dK, "dK"),
                                  _f32(dV, "dV"), Q.shape[0], n_heads, n_kv_heads, head_dim,
                                  float(scale), _stream(stream)))


def rope_bwd_inplace(dX, n_heads, head_dim, pos_offset=0, base=10000.0, stream=None):
    """Interleaved RoPE backward in place on dX [S, n_heads*head_dim]."""
    _check(lib().rope_bwd_inplace(_f32(dX, "dX"), dX.shape[0], n_heads, head_dim, pos_offset,
                                  float(base), _stream(stream)))
    return dX


def profile_events(before, after):
    """Arm the one-shot measurement hook with two torch.cuda.Event objects: the
    next backward call records them around its dominant kernel stage."""
    lib().gqa_profile_events(before.cuda_event, after.cuda_event)


def profile_stage_name() -> str:
    return lib().gqa_profile_stage_name().decode()


def launch_count() -> int:
    """Kernels launched by the library so far in this process."""
    return int(lib().gqa_launch_count())


def read_device_status(workspace, stream=None):
    """Synchronise and raise if a bounded device wait gave up during the last call."""
    _check(lib().attn_read_device_status(workspace.data_ptr(), _stream(stream)))


def n_pairs_from_seg(seg_host) -> int:
    """Unmasked (query, key) pairs: sum over i of i - seg[i] + 1 (host-side count)."""
    import numpy as np
    s = np.arange(len(seg_host), dtype=np.int64)
    return int(np.sum(s - np.asarray(seg_host, dtype=np.int64) + 1))
