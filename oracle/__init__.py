"""Double-precision CPU oracle for the Simple GLA mixer (ctypes wrapper).

TEST INFRASTRUCTURE ONLY: the test suite, the entry module's smoke check and
the benchmark's CPU-baseline / reference leg are the only users. The CUDA
library never imports, links or calls it, and it shares no code with it.

The arithmetic lives in gla_oracle.c; this file compiles it with gcc (no
fast-math, no FMA contraction) and marshals numpy arrays. Every array is
promoted to float64 before the call, so the oracle sees exactly the values
the GPU receives (bf16-rounded inputs stay bf16 values).

Functions (all layouts token-major, see gla_oracle.c):
  fwd_recurrent  -- the token recurrence (O2)
  fwd_quadratic  -- brute-force unrolled form, tiny inputs only (O1)
  fwd_chunked    -- the chunked form in double (O5)
  bwd            -- analytic two-pass backward (O3)
  bwd_chunked    -- the chunk-level backward equations in double (O6)
  decode         -- one recurrent step per (sequence, head) (O4)
  mixer_epilogue -- self-augmentation, Head RMSNorm and the SiLU(g) gate (O7)
  conv1d         -- causal depthwise Conv1d (width 4) with SiLU and its window (O8)
  fwd_gated      -- per-token (data-dependent) decay: recurrence, unrolled and
                    chunked forms (O9)
  decode_gated   -- one recurrent step with a per-token decay (O10)
  bwd_gated      -- gradients of the per-token decay form, the gate's included (O11)
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "gla_oracle.c")
_LIB = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_lib = None

_D = ctypes.POINTER(ctypes.c_double)
_L = ctypes.c_long


def build(force: bool = False) -> str:
    """Compile gla_oracle.c into liboracle.so next to it (gcc, -O2, no fast-math)."""
    if not force and os.path.exists(_LIB) and os.path.getmtime(_LIB) >= os.path.getmtime(_SRC):
        return _LIB
    tmp = _LIB + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-pthread", "-ffp-contract=off",
           "-fno-fast-math", _SRC, "-o", tmp, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    with _lock:
        if _lib is None:
            build()
            lib = ctypes.CDLL(_LIB)
            fwd_sig = [_D, _D, _D, _D, _D, ctypes.c_double, _L, _L, _L, _L, _L, _D, _D, ctypes.c_int]
            lib.gla_oracle_fwd_recurrent.argtypes = fwd_sig
            lib.gla_oracle_fwd_quadratic.argtypes = fwd_sig
            lib.gla_oracle_fwd_chunked.argtypes = fwd_sig[:11] + [_L] + fwd_sig[11:]
            bwd_sig = [_D, _D, _D, _D, _D, ctypes.c_double, _D, _D, _L, _L, _L, _L, _L,
                       _D, _D, _D, _D, ctypes.c_int]
            lib.gla_oracle_bwd.argtypes = bwd_sig
            lib.gla_oracle_bwd_chunked.argtypes = bwd_sig[:13] + [_L] + bwd_sig[13:]
            lib.gla_oracle_decode.argtypes = [_D, _D, _D, _D, _D, ctypes.c_double, _L, _L, _L, _L,
                                              _D, ctypes.c_int]
            lib.gla_oracle_threads.argtypes = [ctypes.c_int]
            lib.gla_oracle_mixer_epilogue.argtypes = [_D, _D, _D, _D, _D, _D, _D, ctypes.c_double, _L, _L, _L,
                                                      _L, _D, ctypes.c_int]
            lib.gla_oracle_conv1d.argtypes = [_D, _D, _D, _D, _L, _L, _L, _D, _D, ctypes.c_int]
            gsig = [_D, _D, _D, _D, _D, ctypes.c_double, _L, _L, _L, _L, _L, _D, _D, ctypes.c_int]
            lib.gla_oracle_fwd_gated.argtypes = gsig
            lib.gla_oracle_fwd_gated_quadratic.argtypes = gsig
            lib.gla_oracle_fwd_gated_chunked.argtypes = gsig[:11] + [_L] + gsig[11:]
            lib.gla_oracle_decode_gated.argtypes = [_D, _D, _D, _D, _D, ctypes.c_double, _L, _L, _L, _L,
                                                    _D, ctypes.c_int]
            lib.gla_oracle_bwd_gated.argtypes = [_D, _D, _D, _D, _D, ctypes.c_double, _D, _D, _L, _L, _L, _L, _L,
                                                 _D, _D, _D, _D, _D, ctypes.c_int]
            for f in ("gla_oracle_fwd_recurrent", "gla_oracle_fwd_quadratic", "gla_oracle_fwd_chunked",
                      "gla_oracle_bwd", "gla_oracle_bwd_chunked", "gla_oracle_decode",
                      "gla_oracle_threads", "gla_oracle_mixer_epilogue", "gla_oracle_conv1d",
                      "gla_oracle_fwd_gated", "gla_oracle_fwd_gated_quadratic", "gla_oracle_fwd_gated_chunked",
                      "gla_oracle_decode_gated", "gla_oracle_bwd_gated"):
                getattr(lib, f).restype = ctypes.c_int
            _lib = lib
    return _lib


def threads(nthreads: int = 0) -> int:
    """Number of host threads the oracle uses for `nthreads` (0 = all online cores)."""
    return int(_load().gla_oracle_threads(int(nthreads)))


def _f64(x):
    if x is None:
        return None
    return np.ascontiguousarray(x, dtype=np.float64)


def _p(x):
    return None if x is None else x.ctypes.data_as(_D)


def _dims(q, v):
    B, T, H, dk = q.shape
    dv = v.shape[-1]
    return B, T, H, dk, dv


def _check(rc, name):
    if rc != 0:
        raise ValueError(f"oracle {name}: invalid arguments")


def _fwd(fn_name, q, k, v, log_lambda, h0, scale, nthreads, chunk=None, want_o=True, want_hT=True):
    lib = _load()
    q, k, v, ll, h0 = _f64(q), _f64(k), _f64(v), _f64(log_lambda), _f64(h0)
    B, T, H, dk, dv = _dims(q, v)
    o = np.zeros((B, T, H, dv)) if want_o else None
    hT = np.zeros((B, H, dk, dv)) if want_hT else None
    args = [_p(q), _p(k), _p(v), _p(ll), _p(h0), float(scale), B, T, H, dk, dv]
    if chunk is not None:
        args.append(int(chunk))
    args += [_p(o), _p(hT), int(nthreads)]
    _check(getattr(lib, fn_name)(*args), fn_name)
    return o, hT


def fwd_recurrent(q, k, v, log_lambda, h0=None, scale=1.0, nthreads=0, want_o=True):
    """O2: o_t = scale * S_t^T q_t with S_t = lambda S_{t-1} + k_t v_t^T. Returns (o, hT)."""
    return _fwd("gla_oracle_fwd_recurrent", q, k, v, log_lambda, h0, scale, nthreads, want_o=want_o)


def fwd_quadratic(q, k, v, log_lambda, h0=None, scale=1.0, nthreads=0):
    """O1: brute-force unrolled sum (O(T^2)). Returns (o, hT)."""
    return _fwd("gla_oracle_fwd_quadratic", q, k, v, log_lambda, h0, scale, nthreads)


def fwd_chunked(q, k, v, log_lambda, h0=None, scale=1.0, chunk=128, nthreads=0):
    """O5: the chunked form in double with chunk length `chunk`. Returns (o, hT)."""
    return _fwd("gla_oracle_fwd_chunked", q, k, v, log_lambda, h0, scale, nthreads, chunk=chunk)


def _bwd(fn_name, q, k, v, log_lambda, h0, scale, do, dhT, nthreads, chunk=None):
    lib = _load()
    q, k, v, ll, h0, do, dhT = map(_f64, (q, k, v, log_lambda, h0, do, dhT))
    B, T, H, dk, dv = _dims(q, v)
    dq = np.zeros((B, T, H, dk))
    dk_ = np.zeros((B, T, H, dk))
    dv_ = np.zeros((B, T, H, dv))
    dh0 = np.zeros((B, H, dk, dv))
    args = [_p(q), _p(k), _p(v), _p(ll), _p(h0), float(scale), _p(do), _p(dhT), B, T, H, dk, dv]
    if chunk is not None:
        args.append(int(chunk))
    args += [_p(dq), _p(dk_), _p(dv_), _p(dh0), int(nthreads)]
    _check(getattr(lib, fn_name)(*args), fn_name)
    return dq, dk_, dv_, dh0


def bwd(q, k, v, log_lambda, h0, scale, do, dhT=None, nthreads=0):
    """O3: gradients of sum<do, o> + <dhT, hT>. Returns (dq, dk, dv, dh0)."""
    return _bwd("gla_oracle_bwd", q, k, v, log_lambda, h0, scale, do, dhT, nthreads)


def bwd_chunked(q, k, v, log_lambda, h0, scale, do, dhT=None, chunk=128, nthreads=0):
    """O6: the chunk-level backward equations in double. Returns (dq, dk, dv, dh0)."""
    return _bwd("gla_oracle_bwd_chunked", q, k, v, log_lambda, h0, scale, do, dhT, nthreads, chunk)


def decode(q, k, v, log_lambda, S, scale=1.0, nthreads=0):
    """O4: one recurrent step per (n, h). q, k [N,H,dk], v [N,H,dv], S [N,H,dk,dv].
    Returns (o, S_new); the input S is not modified."""
    lib = _load()
    q, k, v, ll = map(_f64, (q, k, v, log_lambda))
    S_new = np.array(S, dtype=np.float64, copy=True, order="C")
    N, H, dk = q.shape
    dv = v.shape[-1]
    o = np.zeros((N, H, dv))
    _check(lib.gla_oracle_decode(_p(q), _p(k), _p(v), _p(ll), _p(S_new), float(scale), N, H, dk, dv,
                                 _p(o), int(nthreads)), "decode")
    return o, S_new


def mixer_epilogue(o, q, k, v, g, aug=None, norm_w=None, eps=1e-6, nthreads=0):
    """O7: z = w * u / sqrt(mean(u^2) + eps) * SiLU(g) with u = o + sigmoid(q.(a*k)) v,
    per (token, head). o, v, g [..., H, dv]; q, k [..., H, dk]; aug [H, dk] or None
    (zero); norm_w [H, dv] or None (one). Returns z with o's shape."""
    lib = _load()
    o, q, k, v, g = map(_f64, (o, q, k, v, g))
    H, dv = o.shape[-2], o.shape[-1]
    dk = q.shape[-1]
    NT = int(np.prod(o.shape[:-2]))
    a = _f64(aug) if aug is not None else None
    w = _f64(norm_w) if norm_w is not None else None
    z = np.zeros_like(o)
    _check(lib.gla_oracle_mixer_epilogue(_p(o), _p(q), _p(k), _p(v), _p(g), _p(a), _p(w), float(eps), NT, H, dk,
                                         dv, _p(z), int(nthreads)), "mixer_epilogue")
    return z


def conv1d(x, w, b=None, window=None, nthreads=0):
    """O8: y_t = SiLU(sum_i w[:, i] x_{t-3+i} + b) per channel. x [B,T,D], w [D,4],
    b [D] or None, window [B,4,D] (the sequence's last four inputs before x,
    oldest first) or None (zeros). Returns (y, window_out)."""
    lib = _load()
    x, w = _f64(x), _f64(w)
    b = _f64(b)
    win = _f64(window)
    B, T, D = x.shape
    y = np.zeros_like(x)
    win_out = np.zeros((B, 4, D))
    _check(lib.gla_oracle_conv1d(_p(x), _p(w), _p(b), _p(win), B, T, D, _p(y), _p(win_out), int(nthreads)),
           "conv1d")
    return y, win_out


def fwd_gated(q, k, v, g, h0=None, scale=1.0, form="recurrent", chunk=128, nthreads=0, want_o=True):
    """O9: the forward with a per-token log-decay g [B, T, H] (natural log,
    <= 0, -inf allowed). form = "recurrent" (the token recurrence),
    "quadratic" (unrolled sums, tiny inputs only) or "chunked" (the chunk
    equations at `chunk`). Returns (o [B,T,H,dv], hT [B,H,dk,dv])."""
    lib = _load()
    q, k, v, g, h0 = _f64(q), _f64(k), _f64(v), _f64(g), _f64(h0)
    B, T, H, dk, dv = _dims(q, v)
    if g.shape != (B, T, H):
        raise ValueError(f"oracle fwd_gated: g has shape {g.shape}, expected {(B, T, H)}")
    o = np.zeros((B, T, H, dv)) if (want_o or form == "quadratic") else None
    hT = np.zeros((B, H, dk, dv))
    args = [_p(q), _p(k), _p(v), _p(g), _p(h0), float(scale), B, T, H, dk, dv]
    name = {"recurrent": "gla_oracle_fwd_gated", "quadratic": "gla_oracle_fwd_gated_quadratic",
            "chunked": "gla_oracle_fwd_gated_chunked"}[form]
    if form == "chunked":
        args.append(int(chunk))
    args += [_p(o), _p(hT), int(nthreads)]
    _check(getattr(lib, name)(*args), name)
    return o, hT


def decode_gated(q, k, v, g, S, scale=1.0, nthreads=0):
    """O10: one step S <- exp(g) S + k v^T, o = scale S^T q per (n, h), with a
    per-sequence, per-head log-decay g [N, H]. Returns (o [N,H,dv], S_new)."""
    lib = _load()
    q, k, v, g = _f64(q), _f64(k), _f64(v), _f64(g)
    S = np.array(S, dtype=np.float64, copy=True, order="C")
    N, H, dk = q.shape
    dv = v.shape[-1]
    if g.shape != (N, H):
        raise ValueError(f"oracle decode_gated: g has shape {g.shape}, expected {(N, H)}")
    o = np.zeros((N, H, dv))
    _check(lib.gla_oracle_decode_gated(_p(q), _p(k), _p(v), _p(g), _p(S), float(scale), N, H, dk, dv, _p(o),
                                       int(nthreads)), "decode_gated")
    return o, S


def bwd_gated(q, k, v, g, h0, scale, do, dhT=None, nthreads=0):
    """O11: gradients of L = sum <do, o> + <dhT, hT> for the per-token decay
    exp(g), g [B,T,H]. Returns (dq, dk, dv, dh0, dg)."""
    lib = _load()
    q, k, v, g, h0, do, dhT = map(_f64, (q, k, v, g, h0, do, dhT))
    B, T, H, dk, dv = _dims(q, v)
    dq, dk_, dv_ = np.zeros_like(q), np.zeros_like(k), np.zeros_like(v)
    dh0 = np.zeros((B, H, dk, dv))
    dg = np.zeros((B, T, H))
    _check(lib.gla_oracle_bwd_gated(_p(q), _p(k), _p(v), _p(g), _p(h0), float(scale), _p(do), _p(dhT),
                                    B, T, H, dk, dv, _p(dq), _p(dk_), _p(dv_), _p(dh0), _p(dg), int(nthreads)),
           "bwd_gated")
    return dq, dk_, dv_, dh0, dg
