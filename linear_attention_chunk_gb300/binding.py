"""ctypes binding of libgla (include/gla.h), with the C ABI's names.

Argument marshalling only: every step of the mixer runs in libgla's CUDA
kernels. PyTorch supplies device memory and the current stream; the
functions below read shapes from the tensors, allocate outputs that the
caller did not pass, and forward raw device pointers. There is no CPU path:
if libgla.so is missing or a call fails, a GlaError is raised.

Functions:
  gla_chunk_fwd(q, k, v, log_lambda, h0=None, scale=None, chunk=128, ...) -> (o, hT)
  gla_chunk_fwd_noalloc(...)                                              -> (o, hT)
  gla_chunk_fwd_varlen(q, k, v, log_lambda, cu_seqlens, state_pool, ...)  -> o  (pool updated)
  gla_chunk_fwd_varlen_gated(q, k, v, g, cu_seqlens, state_pool, ...)     -> o  (pool updated) per-token decay
  gla_chunk_fwd_mixer(q, k, v, g, log_lambda, ...)                        -> (z, hT)
  gla_chunk_fwd_gated(q, k, v, g, h0=None, scale=None, chunk=128, ...)    -> (o, hT)  per-token decay
  gla_chunk_bwd(q, k, v, log_lambda, do, h0=None, dhT=None, ...)          -> (dq, dk, dv, dh0)
  gla_chunk_bwd_gated(q, k, v, g, do, h0=None, dhT=None, ...)             -> (dq, dk, dv, dh0, dg)
  gla_decode_step(q, k, v, log_lambda, S, scale=None, ...)                -> o  (S updated in place)
  gla_decode_step_mixer(q, k, v, log_lambda, S, g, ...)                   -> z  (S updated in place)
  gla_decode_step_gated(q, k, v, g, S, scale=None, ...)                   -> o  (S updated in place)
  gla_mixer_epilogue(o, q, k, v, g, aug=None, norm_w=None, eps=1e-6)      -> z
  gla_conv1d_fwd(x, w, b=None, win_in=None, ...)                          -> (y, win_out)
  gla_conv1d_varlen(x, w, b, cu_seqlens, win_pool, slots=None)            -> y  (pool updated)
  gla_conv1d_step(x, w, b, win)                                           -> y  (window updated)
  gla_check(stream=None), gla_status_string(code), gla_version()
  gla_chunk_fwd_workspace_size(...), gla_chunk_bwd_workspace_size(...)
`lib()` returns the loaded ctypes library for callers that hold raw pointers.
"""
from __future__ import annotations

import ctypes
import math
import os
import threading

PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(PKG, "_lib", "libgla.so")

GLA_OK, GLA_ERR_INVALID_ARG, GLA_ERR_UNSUPPORTED, GLA_ERR_CUDA, GLA_ERR_TIMEOUT, GLA_ERR_WORKSPACE = range(6)
GLA_BF16, GLA_FP32 = 0, 1

# The public entry points declared in include/gla.h.
ABI_FUNCTIONS = ("gla_chunk_fwd", "gla_chunk_fwd_workspace_size", "gla_chunk_fwd_noalloc", "gla_chunk_fwd_varlen", "gla_chunk_fwd_varlen_gated",
                 "gla_chunk_fwd_mixer", "gla_chunk_fwd_gated", "gla_chunk_fwd_gated_workspace_size", "gla_decode_step_gated", "gla_chunk_bwd",
                 "gla_chunk_bwd_workspace_size", "gla_chunk_bwd_gated", "gla_chunk_bwd_gated_workspace_size", "gla_decode_step", "gla_decode_step_mixer", "gla_mixer_epilogue",
                 "gla_conv1d_fwd", "gla_conv1d_varlen", "gla_conv1d_step", "gla_selftest_wait_timeout", "gla_check",
                 "gla_status_string", "gla_last_error", "gla_last_launch_count", "gla_version")


class GlaError(RuntimeError):
    def __init__(self, status: int, func: str, detail: str = ""):
        self.status = status
        name = _status_name(status)
        super().__init__(f"{func} failed: {name}" + (f" -- {detail}" if detail else ""))


_lock = threading.Lock()
_lib = None
_vp = ctypes.c_void_p
_i = ctypes.c_int
_f = ctypes.c_float
_sz = ctypes.c_size_t


def lib():
    """Load libgla.so (built in-tree by linear_attention_chunk_gb300.build)."""
    global _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(LIB_PATH):
                raise GlaError(GLA_ERR_CUDA, "load",
                               f"{LIB_PATH} is not built; run `python -m linear_attention_chunk_gb300.build`")
            L = ctypes.CDLL(LIB_PATH)
            L.gla_chunk_fwd.argtypes = [_vp, _vp, _vp, _vp, _vp, _f, _i, _i, _i, _i, _i, _i, _i,
                                        _vp, _vp, _vp, _sz, _vp]
            L.gla_chunk_fwd.restype = _i
            L.gla_chunk_fwd_noalloc.argtypes = [_vp, _vp, _vp, _vp, _vp, _f, _i, _i, _i, _i, _i, _i, _i,
                                                _vp, _vp, _vp]
            L.gla_chunk_fwd_noalloc.restype = _i
            L.gla_chunk_fwd_varlen.argtypes = [_vp, _vp, _vp, _vp, _f, _vp, _vp, _vp, _i, _i, _i, _i, _i, _i,
                                               _i, _i, _vp, _vp]
            L.gla_chunk_fwd_varlen.restype = _i
            L.gla_chunk_fwd_mixer.argtypes = [_vp, _vp, _vp, _vp, _vp, _vp, _f, _vp, _vp, _f, _i, _i, _i, _i, _i, _i,
                                              _i, _vp, _vp, _vp, _sz, _vp]
            L.gla_chunk_fwd_mixer.restype = _i
            L.gla_chunk_fwd_varlen_gated.argtypes = [_vp, _vp, _vp, _vp, _f, _vp, _vp, _vp, _i, _i, _i, _i, _i,
                                                     _i, _i, _i, _vp, _vp]
            L.gla_chunk_fwd_varlen_gated.restype = _i
            L.gla_chunk_fwd_gated.argtypes = [_vp, _vp, _vp, _vp, _vp, _f, _i, _i, _i, _i, _i, _i, _i, _vp, _vp,
                                              _vp, _sz, _vp]
            L.gla_chunk_fwd_gated.restype = _i
            L.gla_chunk_fwd_gated_workspace_size.argtypes = [_i, _i, _i, _i, _i, _i, _i]
            L.gla_chunk_fwd_gated_workspace_size.restype = _sz
            L.gla_decode_step_gated.argtypes = [_vp, _vp, _vp, _vp, _vp, _f, _i, _i, _i, _i, _i, _vp, _vp]
            L.gla_decode_step_gated.restype = _i
            L.gla_chunk_fwd_workspace_size.argtypes = [_i, _i, _i, _i, _i, _i, _i]
            L.gla_chunk_fwd_workspace_size.restype = _sz
            L.gla_chunk_bwd.argtypes = [_vp, _vp, _vp, _vp, _vp, _f, _vp, _vp, _i, _i, _i, _i, _i, _i, _i,
                                        _vp, _vp, _vp, _vp, _vp, _sz, _vp]
            L.gla_chunk_bwd.restype = _i
            L.gla_chunk_bwd_workspace_size.argtypes = [_i, _i, _i, _i, _i, _i, _i]
            L.gla_chunk_bwd_workspace_size.restype = _sz
            L.gla_chunk_bwd_gated.argtypes = [_vp, _vp, _vp, _vp, _vp, _f, _vp, _vp, _i, _i, _i, _i, _i, _i, _i,
                                              _vp, _vp, _vp, _vp, _vp, _vp, _sz, _vp]
            L.gla_chunk_bwd_gated.restype = _i
            L.gla_chunk_bwd_gated_workspace_size.argtypes = [_i, _i, _i, _i, _i, _i, _i]
            L.gla_chunk_bwd_gated_workspace_size.restype = _sz
            L.gla_decode_step.argtypes = [_vp, _vp, _vp, _vp, _vp, _f, _i, _i, _i, _i, _i, _vp, _vp]
            L.gla_decode_step.restype = _i
            L.gla_decode_step_mixer.argtypes = [_vp, _vp, _vp, _vp, _vp, _f, _vp, _vp, _vp, _f, _i, _i, _i, _i, _i,
                                                _vp, _vp]
            L.gla_decode_step_mixer.restype = _i
            L.gla_mixer_epilogue.argtypes = [_vp, _vp, _vp, _vp, _vp, _vp, _vp, _f, _i, _i, _i, _i, _i, _vp, _vp]
            L.gla_mixer_epilogue.restype = _i
            L.gla_conv1d_fwd.argtypes = [_vp, _vp, _vp, _vp, _i, _i, _i, _i, _vp, _vp, _vp]
            L.gla_conv1d_fwd.restype = _i
            L.gla_conv1d_varlen.argtypes = [_vp, _vp, _vp, _vp, _vp, _vp, _i, _i, _i, _i, _i, _vp, _vp]
            L.gla_conv1d_varlen.restype = _i
            L.gla_conv1d_step.argtypes = [_vp, _vp, _vp, _vp, _i, _i, _i, _vp, _vp]
            L.gla_conv1d_step.restype = _i
            L.gla_selftest_wait_timeout.argtypes = [ctypes.c_uint, _vp, _vp]
            L.gla_selftest_wait_timeout.restype = _i
            L.gla_check.argtypes = [_vp]
            L.gla_check.restype = _i
            L.gla_status_string.argtypes = [_i]
            L.gla_status_string.restype = ctypes.c_char_p
            L.gla_last_error.argtypes = []
            L.gla_last_error.restype = ctypes.c_char_p
            L.gla_last_launch_count.argtypes = []
            L.gla_last_launch_count.restype = _i
            L.gla_version.argtypes = []
            L.gla_version.restype = ctypes.c_char_p
            _lib = L
    return _lib


def _status_name(status: int) -> str:
    try:
        return lib().gla_status_string(int(status)).decode()
    except Exception:
        return f"status {status}"


def _raise_on(status: int, func: str):
    if status != GLA_OK:
        raise GlaError(status, func, lib().gla_last_error().decode(errors="replace"))


def gla_status_string(status: int) -> str:
    return lib().gla_status_string(int(status)).decode()


def gla_version() -> str:
    return lib().gla_version().decode()


def gla_last_launch_count() -> int:
    """Kernels launched by the last entry-point call on this thread."""
    return int(lib().gla_last_launch_count())


# ------------------------------------------------------------------ helpers
def _torch():
    import torch
    return torch


def _dtype_code(t) -> int:
    torch = _torch()
    if t.dtype == torch.bfloat16:
        return GLA_BF16
    if t.dtype == torch.float32:
        return GLA_FP32
    raise GlaError(GLA_ERR_INVALID_ARG, "dtype", f"unsupported tensor dtype {t.dtype}")


def _ptr(t):
    if t is None:
        return None
    if not t.is_cuda:
        raise GlaError(GLA_ERR_INVALID_ARG, "argument", "tensors must live on a CUDA device")
    if not t.is_contiguous():
        raise GlaError(GLA_ERR_INVALID_ARG, "argument", "tensors must be contiguous")
    return t.data_ptr()


def _f32(t, shape, name):
    """Pointer of an fp32 argument (decays, states), after checking its dtype
    and shape: the C ABI reads these buffers as float without knowing them."""
    if t is None:
        return None
    torch = _torch()
    if t.dtype != torch.float32:
        raise GlaError(GLA_ERR_INVALID_ARG, "argument", f"{name} must be float32, got {t.dtype}")
    if tuple(t.shape) != tuple(shape):
        raise GlaError(GLA_ERR_INVALID_ARG, "argument", f"{name} has shape {tuple(t.shape)}, expected {tuple(shape)}")
    return _ptr(t)


def _stream(stream):
    torch = _torch()
    if stream is None:
        stream = torch.cuda.current_stream()
    return stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)


# --------------------------------------------------------------- entry points
def gla_chunk_fwd_workspace_size(B, T, H, dk, dv, chunk=128, dtype=GLA_BF16) -> int:
    return int(lib().gla_chunk_fwd_workspace_size(B, T, H, dk, dv, chunk, dtype))


def gla_chunk_bwd_workspace_size(B, T, H, dk, dv, chunk=128, dtype=GLA_BF16) -> int:
    return int(lib().gla_chunk_bwd_workspace_size(B, T, H, dk, dv, chunk, dtype))


def gla_chunk_fwd(q, k, v, log_lambda, h0=None, scale=None, chunk=128, *, o=None, hT=None,
                  want_hT=True, workspace=None, stream=None):
    """Chunked forward. q, k [B,T,H,dk], v [B,T,H,dv] (bf16 or fp32, CUDA),
    log_lambda [H] fp32, h0 [B,H,dk,dv] fp32 or None. Returns (o, hT)."""
    torch = _torch()
    B, T, H, dk = q.shape
    dv = v.shape[-1]
    dt = _dtype_code(q)
    if scale is None:
        scale = 1.0 / math.sqrt(dk)
    if o is None:
        o = torch.empty((B, T, H, dv), dtype=q.dtype, device=q.device)
    if hT is None and want_hT:
        hT = torch.empty((B, H, dk, dv), dtype=torch.float32, device=q.device)
    ws_need = gla_chunk_fwd_workspace_size(B, T, H, dk, dv, chunk, dt)
    if workspace is None and ws_need > 0:
        workspace = torch.empty(ws_need, dtype=torch.uint8, device=q.device)
    ws_bytes = workspace.numel() * workspace.element_size() if workspace is not None else 0
    st = lib().gla_chunk_fwd(_ptr(q), _ptr(k), _ptr(v), _f32(log_lambda, (H,), "log_lambda"),
                             _f32(h0, (B, H, dk, dv), "h0"), float(scale),
                             B, T, H, dk, dv, int(chunk), dt, _ptr(o), _ptr(hT),
                             _ptr(workspace), ws_bytes, _stream(stream))
    _raise_on(st, "gla_chunk_fwd")
    return o, hT


def gla_chunk_fwd_noalloc(q, k, v, log_lambda, h0=None, scale=None, chunk=128, *, o, hT=None, stream=None):
    """The forward without any device allocation by the library: for callers
    that may not allocate device memory, the segmentation scratch comes from
    a fixed array inside the library. The caller passes the output tensors.
    Returns (o, hT)."""
    B, T, H, dk = q.shape
    dv = v.shape[-1]
    if scale is None:
        scale = 1.0 / math.sqrt(dk)
    st = lib().gla_chunk_fwd_noalloc(_ptr(q), _ptr(k), _ptr(v), _ptr(log_lambda), _ptr(h0), float(scale),
                                     B, T, H, dk, dv, int(chunk), _dtype_code(q), _ptr(o), _ptr(hT),
                                     _stream(stream))
    _raise_on(st, "gla_chunk_fwd_noalloc")
    return o, hT


def gla_chunk_fwd_varlen(q, k, v, log_lambda, cu_seqlens, state_pool, slots=None, scale=None, chunk=128, *,
                         o=None, stream=None):
    """Variable-length forward: q, k [total_T,H,dk], v [total_T,H,dv] bf16
    packed, sequence n = tokens [cu_seqlens[n], cu_seqlens[n+1]) (int32 CUDA
    tensor), state_pool [n_slots,H,dk,dv] fp32 updated in place at slots[n]
    (int32 CUDA tensor, or None for slot n). Returns o [total_T,H,dv]."""
    torch = _torch()
    total_T, H, dk = q.shape
    dv = v.shape[-1]
    if scale is None:
        scale = 1.0 / math.sqrt(dk)
    if o is None:
        o = torch.empty((total_T, H, dv), dtype=q.dtype, device=q.device)
    nseq = cu_seqlens.numel() - 1
    st = lib().gla_chunk_fwd_varlen(_ptr(q), _ptr(k), _ptr(v), _ptr(log_lambda), float(scale), _ptr(cu_seqlens),
                                    _ptr(slots), _ptr(state_pool), int(state_pool.shape[0]), nseq, total_T, H,
                                    dk, dv, int(chunk), _dtype_code(q), _ptr(o), _stream(stream))
    _raise_on(st, "gla_chunk_fwd_varlen")
    return o


def gla_chunk_fwd_gated_workspace_size(B, T, H, dk, dv, chunk=128, dtype=GLA_BF16) -> int:
    return int(lib().gla_chunk_fwd_gated_workspace_size(B, T, H, dk, dv, chunk, dtype))


def gla_chunk_fwd_gated(q, k, v, g, h0=None, scale=None, chunk=128, *, o=None, hT=None, want_hT=True,
                        workspace=None, stream=None):
    """Chunked forward with a per-token decay: g [B,T,H] fp32 natural-log
    decays (<= 0, -inf clears the state); q, k, v, h0 as gla_chunk_fwd.
    Returns (o, hT)."""
    torch = _torch()
    B, T, H, dk = q.shape
    dv = v.shape[-1]
    if scale is None:
        scale = 1.0 / math.sqrt(dk)
    if o is None:
        o = torch.empty((B, T, H, dv), dtype=q.dtype, device=q.device)
    if hT is None and want_hT:
        hT = torch.empty((B, H, dk, dv), dtype=torch.float32, device=q.device)
    dt = _dtype_code(q)
    ws_need = gla_chunk_fwd_gated_workspace_size(B, T, H, dk, dv, chunk, dt)
    if workspace is None and ws_need > 0:
        workspace = torch.empty(ws_need, dtype=torch.uint8, device=q.device)
    ws_bytes = workspace.numel() * workspace.element_size() if workspace is not None else 0
    st = lib().gla_chunk_fwd_gated(_ptr(q), _ptr(k), _ptr(v), _f32(g, (B, T, H), "g"), _f32(h0, (B, H, dk, dv), "h0"),
                                   float(scale), B, T, H, dk, dv,
                                   int(chunk), dt, _ptr(o), _ptr(hT), _ptr(workspace), ws_bytes, _stream(stream))
    _raise_on(st, "gla_chunk_fwd_gated")
    return o, hT


def gla_chunk_fwd_varlen_gated(q, k, v, g, cu_seqlens, state_pool, slots=None, scale=None, chunk=128, *,
                               o=None, stream=None):
    """Variable-length forward with a per-token decay: g [total_T,H] fp32
    natural-log decays, packed like q; otherwise as gla_chunk_fwd_varlen.
    Returns o [total_T,H,dv]."""
    torch = _torch()
    total_T, H, dk = q.shape
    dv = v.shape[-1]
    if scale is None:
        scale = 1.0 / math.sqrt(dk)
    if o is None:
        o = torch.empty((total_T, H, dv), dtype=q.dtype, device=q.device)
    nseq = cu_seqlens.numel() - 1
    st = lib().gla_chunk_fwd_varlen_gated(_ptr(q), _ptr(k), _ptr(v), _f32(g, (total_T, H), "g"), float(scale),
                                          _ptr(cu_seqlens),
                                          _ptr(slots), _ptr(state_pool), int(state_pool.shape[0]), nseq, total_T, H,
                                          dk, dv, int(chunk), _dtype_code(q), _ptr(o), _stream(stream))
    _raise_on(st, "gla_chunk_fwd_varlen_gated")
    return o


def gla_chunk_fwd_mixer(q, k, v, g, log_lambda, h0=None, scale=None, chunk=128, aug=None, norm_w=None, eps=1e-6,
                        *, z=None, hT=None, want_hT=True, workspace=None, stream=None):
    """The chunked forward followed by the mixer epilogue, z in place of o
    (bf16): returns (z, hT), z [B,T,H,dv] = Head RMSNorm(o + sigmoid(q.(aug*k)) v)
    * norm_w * SiLU(g)."""
    torch = _torch()
    B, T, H, dk = q.shape
    dv = v.shape[-1]
    if scale is None:
        scale = 1.0 / math.sqrt(dk)
    if z is None:
        z = torch.empty((B, T, H, dv), dtype=q.dtype, device=q.device)
    if hT is None and want_hT:
        hT = torch.empty((B, H, dk, dv), dtype=torch.float32, device=q.device)
    if workspace is None:
        n = gla_chunk_fwd_workspace_size(B, T, H, dk, dv, chunk)
        workspace = torch.empty(max(n, 16), dtype=torch.uint8, device=q.device) if n else None
    ws_bytes = workspace.numel() * workspace.element_size() if workspace is not None else 0
    st = lib().gla_chunk_fwd_mixer(_ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(log_lambda), _ptr(h0), float(scale),
                                   _ptr(aug), _ptr(norm_w), float(eps), B, T, H, dk, dv, int(chunk), _dtype_code(q),
                                   _ptr(z), _ptr(hT), _ptr(workspace), ws_bytes, _stream(stream))
    _raise_on(st, "gla_chunk_fwd_mixer")
    return z, hT


def gla_chunk_bwd(q, k, v, log_lambda, do, h0=None, dhT=None, scale=None, chunk=128, *,
                  dq=None, dk=None, dv=None, dh0=None, want_dh0=True, workspace=None, stream=None):
    """Chunked backward. Returns (dq, dk, dv, dh0)."""
    torch = _torch()
    B, T, H, dk_ = q.shape
    dv_ = v.shape[-1]
    dt = _dtype_code(q)
    if scale is None:
        scale = 1.0 / math.sqrt(dk_)
    dq = torch.empty_like(q) if dq is None else dq
    dk = torch.empty_like(k) if dk is None else dk
    dv = torch.empty_like(v) if dv is None else dv
    if dh0 is None and want_dh0:
        dh0 = torch.empty((B, H, dk_, dv_), dtype=torch.float32, device=q.device)
    ws_need = gla_chunk_bwd_workspace_size(B, T, H, dk_, dv_, chunk, dt)
    if workspace is None and ws_need > 0:
        workspace = torch.empty(ws_need, dtype=torch.uint8, device=q.device)
    ws_bytes = workspace.numel() * workspace.element_size() if workspace is not None else 0
    st = lib().gla_chunk_bwd(_ptr(q), _ptr(k), _ptr(v), _ptr(log_lambda), _ptr(h0), float(scale),
                             _ptr(do), _ptr(dhT), B, T, H, dk_, dv_, int(chunk), dt,
                             _ptr(dq), _ptr(dk), _ptr(dv), _ptr(dh0), _ptr(workspace), ws_bytes,
                             _stream(stream))
    _raise_on(st, "gla_chunk_bwd")
    return dq, dk, dv, dh0


def gla_chunk_bwd_gated_workspace_size(B, T, H, dk, dv, chunk=128, dtype=GLA_BF16) -> int:
    return int(lib().gla_chunk_bwd_gated_workspace_size(B, T, H, dk, dv, chunk, dtype))


def gla_chunk_bwd_gated(q, k, v, g, do, h0=None, dhT=None, scale=None, chunk=128, *,
                        dq=None, dk=None, dv=None, dh0=None, dg=None, want_dh0=True, workspace=None, stream=None):
    """Chunked backward with a per-token decay: g [B,T,H] fp32 natural-log
    decays as gla_chunk_fwd_gated; otherwise as gla_chunk_bwd. Returns
    (dq, dk, dv, dh0, dg), dg [B,T,H] fp32."""
    torch = _torch()
    B, T, H, dk_ = q.shape
    dv_ = v.shape[-1]
    dt = _dtype_code(q)
    if scale is None:
        scale = 1.0 / math.sqrt(dk_)
    dq = torch.empty_like(q) if dq is None else dq
    dk = torch.empty_like(k) if dk is None else dk
    dv = torch.empty_like(v) if dv is None else dv
    if dh0 is None and want_dh0:
        dh0 = torch.empty((B, H, dk_, dv_), dtype=torch.float32, device=q.device)
    if dg is None:
        dg = torch.empty((B, T, H), dtype=torch.float32, device=q.device)
    ws_need = gla_chunk_bwd_gated_workspace_size(B, T, H, dk_, dv_, chunk, dt)
    if workspace is None and ws_need > 0:
        workspace = torch.empty(ws_need, dtype=torch.uint8, device=q.device)
    ws_bytes = workspace.numel() * workspace.element_size() if workspace is not None else 0
    st = lib().gla_chunk_bwd_gated(_ptr(q), _ptr(k), _ptr(v), _f32(g, (B, T, H), "g"),
                                   _f32(h0, (B, H, dk_, dv_), "h0"), float(scale), _ptr(do),
                                   _f32(dhT, (B, H, dk_, dv_), "dhT"), B, T, H, dk_, dv_, int(chunk), dt,
                                   _ptr(dq), _ptr(dk), _ptr(dv), _f32(dh0, (B, H, dk_, dv_), "dh0"),
                                   _f32(dg, (B, T, H), "dg"), _ptr(workspace), ws_bytes, _stream(stream))
    _raise_on(st, "gla_chunk_bwd_gated")
    return dq, dk, dv, dh0, dg


def gla_decode_step(q, k, v, log_lambda, S, scale=None, *, o=None, stream=None):
    """One recurrent step. q, k [N,H,dk], v [N,H,dv], S [N,H,dk,dv] fp32
    (updated in place). Returns o [N,H,dv]."""
    torch = _torch()
    N, H, dk = q.shape
    dv = v.shape[-1]
    dt = _dtype_code(q)
    if scale is None:
        scale = 1.0 / math.sqrt(dk)
    if o is None:
        o = torch.empty((N, H, dv), dtype=q.dtype, device=q.device)
    st = lib().gla_decode_step(_ptr(q), _ptr(k), _ptr(v), _f32(log_lambda, (H,), "log_lambda"),
                               _f32(S, (N, H, dk, dv), "S"), float(scale),
                               N, H, dk, dv, dt, _ptr(o), _stream(stream))
    _raise_on(st, "gla_decode_step")
    return o


def gla_decode_step_gated(q, k, v, g, S, scale=None, *, o=None, stream=None):
    """One recurrent step with a per-token decay g [N,H] fp32 (natural log).
    S [N,H,dk,dv] fp32 is updated in place. Returns o [N,H,dv]."""
    torch = _torch()
    N, H, dk = q.shape
    dv = v.shape[-1]
    if scale is None:
        scale = 1.0 / math.sqrt(dk)
    if o is None:
        o = torch.empty((N, H, dv), dtype=q.dtype, device=q.device)
    st = lib().gla_decode_step_gated(_ptr(q), _ptr(k), _ptr(v), _f32(g, (N, H), "g"), _f32(S, (N, H, dk, dv), "S"),
                                     float(scale), N, H, dk, dv,
                                     _dtype_code(q), _ptr(o), _stream(stream))
    _raise_on(st, "gla_decode_step_gated")
    return o


def gla_decode_step_mixer(q, k, v, log_lambda, S, g, aug=None, norm_w=None, eps=1e-6, scale=None, *, z=None,
                          stream=None):
    """Decode step plus the mixer epilogue in one kernel. Returns z [N,H,dv]."""
    torch = _torch()
    N, H, dk = q.shape
    dv = v.shape[-1]
    if scale is None:
        scale = 1.0 / math.sqrt(dk)
    if z is None:
        z = torch.empty((N, H, dv), dtype=q.dtype, device=q.device)
    st = lib().gla_decode_step_mixer(_ptr(q), _ptr(k), _ptr(v), _ptr(log_lambda), _ptr(S), float(scale), _ptr(g),
                                     _ptr(aug), _ptr(norm_w), float(eps), N, H, dk, dv, _dtype_code(q), _ptr(z),
                                     _stream(stream))
    _raise_on(st, "gla_decode_step_mixer")
    return z


def gla_mixer_epilogue(o, q, k, v, g, aug=None, norm_w=None, eps=1e-6, *, z=None, stream=None):
    """The mixer epilogue over [..., H, d] rows (any leading dims). Returns z like o."""
    torch = _torch()
    H, dv = o.shape[-2], o.shape[-1]
    dk = q.shape[-1]
    NT = o.numel() // (H * dv)
    if z is None:
        z = torch.empty_like(o)
    st = lib().gla_mixer_epilogue(_ptr(o), _ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(aug), _ptr(norm_w), float(eps),
                                  NT, H, dk, dv, _dtype_code(o), _ptr(z), _stream(stream))
    _raise_on(st, "gla_mixer_epilogue")
    return z


def gla_conv1d_fwd(x, w, b=None, win_in=None, *, y=None, win_out=None, want_window=True, stream=None):
    """Causal depthwise Conv1d (width 4) + SiLU over x [B,T,D]; w [D,4], b [D]
    fp32; win_in [B,4,D] fp32 or None (zeros). Returns (y, win_out); win_out
    may be win_in (in place), or None with want_window=False."""
    torch = _torch()
    B, T, D = x.shape
    if y is None:
        y = torch.empty_like(x)
    if win_out is None and want_window:
        win_out = torch.empty((B, 4, D), dtype=torch.float32, device=x.device)
    st = lib().gla_conv1d_fwd(_ptr(x), _ptr(w), _ptr(b), _ptr(win_in), B, T, D, _dtype_code(x), _ptr(y),
                              _ptr(win_out), _stream(stream))
    _raise_on(st, "gla_conv1d_fwd")
    return y, win_out


def gla_conv1d_varlen(x, w, b, cu_seqlens, win_pool, slots=None, *, y=None, stream=None):
    """The Conv1d over packed sequences x [total_T,D] (cu_seqlens int32 CUDA
    tensor), windows in win_pool [n_slots,4,D] fp32 at slots[n] (int32 CUDA
    tensor, or None for slot n), updated in place. Returns y [total_T,D]."""
    torch = _torch()
    total_T, D = x.shape
    if y is None:
        y = torch.empty_like(x)
    nseq = cu_seqlens.numel() - 1
    st = lib().gla_conv1d_varlen(_ptr(x), _ptr(w), _ptr(b), _ptr(cu_seqlens), _ptr(slots), _ptr(win_pool),
                                 int(win_pool.shape[0]), nseq, total_T, D, _dtype_code(x), _ptr(y), _stream(stream))
    _raise_on(st, "gla_conv1d_varlen")
    return y


def gla_conv1d_step(x, w, b, win, *, y=None, stream=None):
    """One serving step of the Conv1d: x [N,D], win [N,4,D] fp32 updated in
    place. Returns y [N,D]."""
    torch = _torch()
    N, D = x.shape
    if y is None:
        y = torch.empty_like(x)
    st = lib().gla_conv1d_step(_ptr(x), _ptr(w), _ptr(b), _ptr(win), N, D, _dtype_code(x), _ptr(y), _stream(stream))
    _raise_on(st, "gla_conv1d_step")
    return y


def gla_selftest_wait_timeout(limit_us=20000, *, stream=None):
    """Diagnostic: make the device-side bounded waits run out (no fault, no
    hang). Returns the int32 CUDA tensor [completed0, completed1, us_waited1];
    the next gla_check() raises GlaError(GLA_ERR_TIMEOUT)."""
    torch = _torch()
    result = torch.full((4,), -1, dtype=torch.int32, device="cuda")
    st = lib().gla_selftest_wait_timeout(int(limit_us), _ptr(result), _stream(stream))
    _raise_on(st, "gla_selftest_wait_timeout")
    return result[:3]


def gla_check(stream=None):
    """Synchronise the stream; raise GlaError on a CUDA error or a device-side timeout."""
    st = lib().gla_check(_stream(stream))
    _raise_on(st, "gla_check")
