"""Seeded synthetic inputs for the Simple GLA mixer.

This module is shared by the oracle-side tests and the CUDA-side tests and
benchmarks. It draws random numbers and rounds them to the storage type; it
holds none of the mixer's arithmetic (no recurrence, no decay powers, no
readout). Every tensor is built on the host with numpy's PCG64 generator,
so the same seed yields the same bytes on x86 and on Arm.

Layouts (token-major, as a fused per-token QKV projection emits them):
  q, k, do, dq, dk : [B, T, H, dk]
  v, o, dv         : [B, T, H, dv]
  h0, hT, dhT, dh0 : [B, H, dk, dv] fp32, dv contiguous
  decode state S   : [N, H, dk, dv] fp32; decode q, k: [N, H, dk]; v, o: [N, H, dv]
  log_lambda       : [H] fp32 (natural log of the per-head decay, <= 0)

Draw order within one case is fixed: q, k, v, do, h0 (or S), dhT, then the
decay draw when the decay is random.

The five named workloads are the mixer shapes of the Laplace 3B layer
("Beyond the KV cache: Training and serving i14's Laplace 3B linear
attention model on AWS Trainium2 with native PyTorch", section "i14 and the
Laplace 3B architecture": H = 16 heads, dk = 96, dv = 192, sequence 2,048,
chunk C = 128 from "Challenge 1"; 1,280 concurrent sequences from
"Inference optimization on Trainium2").
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field
from typing import Optional

import numpy as np

BF16 = "bf16"
FP32 = "fp32"


# ----------------------------------------------------------------------------
# bf16 storage helpers (round-to-nearest-even, the rounding a GPU store uses)
# ----------------------------------------------------------------------------
def bf16_bits(x: np.ndarray) -> np.ndarray:
    """fp32 -> bf16 bit patterns (uint16), round to nearest, ties to even."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    u = x.view(np.uint32).astype(np.uint64)
    rounded = (u + 0x7FFF + ((u >> 16) & 1)) >> 16
    return rounded.astype(np.uint16)


def bf16_to_f32(bits: np.ndarray) -> np.ndarray:
    """bf16 bit patterns (uint16) -> fp32 values (exact)."""
    bits = np.ascontiguousarray(bits, dtype=np.uint16)
    return (bits.astype(np.uint32) << 16).view(np.float32)


def bf16_round(x: np.ndarray) -> np.ndarray:
    """Round fp32 values to the nearest bf16 value, returned as fp32."""
    return bf16_to_f32(bf16_bits(x))


# ----------------------------------------------------------------------------
# decay schedules (inputs of the method, not part of its arithmetic)
# ----------------------------------------------------------------------------
def decay_layer_schedule(H: int) -> np.ndarray:
    """Per-head decay lambda_h = 1 - 2^(-5 - 7h/(H-1)) used by the layer
    workloads (0.96875 for head 0 up to 1 - 2^-12 for the last head)."""
    h = np.arange(H, dtype=np.float64)
    den = max(H - 1, 1)
    return 1.0 - np.exp2(-5.0 - 7.0 * h / den)


def decay_page_schedule(H: int = 16, t_min: float = 1.0, t_max: float = 2048.0) -> np.ndarray:
    """Geometric half-life schedule: head h has a half-life of
    T_h = t_min * (t_max/t_min)^(h/(H-1)) tokens, so lambda_h = 2^(-1/T_h).

    Reading of the "Decay schedule" paragraph (the equation itself is an
    image that did not survive): with T_min = 1 and T_max = 2,048 it gives
    lambda_0 = 0.5 and lambda_15 = 0.99966, the two values the text prints.
    """
    h = np.arange(H, dtype=np.float64)
    den = max(H - 1, 1)
    half_life = t_min * (t_max / t_min) ** (h / den)
    return np.exp2(-1.0 / half_life)


def decay_log_uniform(rng: np.random.Generator, H: int, lo: float = 0.9, hi: float = 0.9999) -> np.ndarray:
    """ln(lambda_h) drawn uniformly in [ln lo, ln hi], independently per head."""
    return np.exp(rng.uniform(math.log(lo), math.log(hi), size=H))


def log_gates(rng: np.random.Generator, shape, kind: str = "gla") -> np.ndarray:
    """Per-token log-decays g <= 0 as fp32 (natural log; the decay is exp(g)).
    kind "gla": log(sigmoid(x)) / 16 with x ~ N(0, 1), the gate-logit
    normaliser of gated linear attention (about -0.045 per token, a decay of
    about e^-5.8 across a 128-token chunk); "wide": uniform in [-3, 0], strong
    decays whose products underflow inside a chunk."""
    if kind == "gla":
        x = rng.standard_normal(shape)
        g = -np.logaddexp(0.0, -x) / 16.0
    elif kind == "wide":
        g = -rng.uniform(0.0, 3.0, size=shape)
    else:
        raise ValueError(f"unknown gate kind {kind!r}")
    return np.minimum(g, 0.0).astype(np.float32)


def log_lambda_of(lam: np.ndarray) -> np.ndarray:
    """Natural log of the decay, as the fp32 value the library receives.
    lambda = 0 maps to -inf."""
    lam = np.asarray(lam, dtype=np.float64)
    with np.errstate(divide="ignore"):
        return np.log(lam).astype(np.float32)


# ----------------------------------------------------------------------------
# a generated case
# ----------------------------------------------------------------------------
@dataclass
class Case:
    """One seeded input set. Float arrays are fp32 holding exactly the values
    the GPU receives (already bf16-rounded when dtype == 'bf16')."""
    B: int
    T: int
    H: int
    dk: int
    dv: int
    dtype: str
    scale: float
    log_lambda: np.ndarray
    q: np.ndarray
    k: np.ndarray
    v: np.ndarray
    h0: Optional[np.ndarray] = None
    do: Optional[np.ndarray] = None
    dhT: Optional[np.ndarray] = None
    chunk: int = 128
    name: str = ""
    extra: dict = field(default_factory=dict)

    def storage(self, x: np.ndarray) -> np.ndarray:
        """The array in the library's storage dtype: uint16 bf16 bits or fp32."""
        if self.dtype == BF16:
            return bf16_bits(x)
        return np.ascontiguousarray(x, dtype=np.float32)


def _normal(rng: np.random.Generator, shape, std: float = 1.0) -> np.ndarray:
    return (rng.standard_normal(size=shape, dtype=np.float64) * std).astype(np.float32)


def _store(x: np.ndarray, dtype: str) -> np.ndarray:
    return bf16_round(x) if dtype == BF16 else np.ascontiguousarray(x, dtype=np.float32)


def _l2_normalise_last(x: np.ndarray) -> np.ndarray:
    x64 = x.astype(np.float64)
    n = np.sqrt(np.sum(x64 * x64, axis=-1, keepdims=True))
    n[n == 0] = 1.0
    return (x64 / n).astype(np.float32)


def make_case(B: int, T: int, H: int, dk: int, dv: int, *, seed: int, dtype: str = BF16,
              lam: Optional[np.ndarray] = None, lam_random: bool = False,
              lam_range=(0.9, 0.9999), normalise_k: bool = False,
              h0_std: Optional[float] = None, with_grad: bool = False,
              dhT_std: Optional[float] = None, do_std: float = 1.0,
              scale: Optional[float] = None, chunk: int = 128, name: str = "",
              gate: Optional[str] = None) -> Case:
    """Draw one case. `lam` fixes the per-head decay (array of H, or a scalar);
    `lam_random` draws it log-uniformly in `lam_range` after the tensors.
    `gate` (a log_gates kind) also draws per-token log-decays g [B, T, H]
    last, into extra["g"]."""
    rng = np.random.default_rng(seed)
    q = _normal(rng, (B, T, H, dk))
    k = _normal(rng, (B, T, H, dk))
    v = _normal(rng, (B, T, H, dv))
    do = _normal(rng, (B, T, H, dv), do_std) if with_grad else None
    h0 = _normal(rng, (B, H, dk, dv), h0_std) if h0_std is not None else None
    dhT = _normal(rng, (B, H, dk, dv), dhT_std) if (with_grad and dhT_std is not None) else None
    if lam_random:
        lam_arr = decay_log_uniform(rng, H, *lam_range)
    elif lam is None:
        lam_arr = decay_layer_schedule(H)
    else:
        lam_arr = np.broadcast_to(np.asarray(lam, dtype=np.float64), (H,)).copy()
    g = log_gates(rng, (B, T, H), gate) if gate is not None else None
    if normalise_k:
        k = _l2_normalise_last(k)
    q, k, v = _store(q, dtype), _store(k, dtype), _store(v, dtype)
    if do is not None:
        do = _store(do, dtype)
    if scale is None:
        scale = 1.0 / math.sqrt(dk)
    return Case(B=B, T=T, H=H, dk=dk, dv=dv, dtype=dtype, scale=float(np.float32(scale)),
                log_lambda=log_lambda_of(lam_arr), q=q, k=k, v=v, h0=h0, do=do, dhT=dhT,
                chunk=chunk, name=name, extra={} if g is None else {"g": g})


# ----------------------------------------------------------------------------
# the five named workloads
# ----------------------------------------------------------------------------
LAYER_H, LAYER_DK, LAYER_DV = 16, 96, 192


def tiny_fp32(seed: int = 0) -> Case:
    """Tiny forward, fp32: B=H=1, T=256 (two 128-token chunks), lambda=0.95, h0=0."""
    return make_case(1, 256, 1, LAYER_DK, LAYER_DV, seed=seed, dtype=FP32, lam=0.95,
                     chunk=128, name="tiny_fwd_fp32_B1_H1_T256")


def layer_fwd(seed: int = 1, B: int = 8, T: int = 2048) -> Case:
    """Laplace-layer forward, bf16: B=8, H=16, T=2048, k L2-normalised per token."""
    return make_case(B, T, LAYER_H, LAYER_DK, LAYER_DV, seed=seed, dtype=BF16,
                     normalise_k=True, chunk=128, name=f"layer_fwd_bf16_B{B}_H16_T{T}")


def train_fwd_bwd(seed: int = 2, B: int = 16, T: int = 2048) -> Case:
    """Training forward+backward, bf16: B=16, H=16, T=2048; do ~ N(0,1),
    h0 ~ N(0, 0.02), dhT = 0."""
    return make_case(B, T, LAYER_H, LAYER_DK, LAYER_DV, seed=seed, dtype=BF16,
                     normalise_k=True, h0_std=0.02, with_grad=True, chunk=128,
                     name=f"train_fwd_bwd_bf16_B{B}_H16_T{T}")


def long_prefill(seed: int = 4, T: int = 65536, chunk: int = 128) -> Case:
    """Long-context prefill, bf16: B=1, H=16, T=65,536, decay log-uniform in
    [0.9, 0.9999], h0 ~ N(0, 0.1), k not normalised."""
    return make_case(1, T, LAYER_H, LAYER_DK, LAYER_DV, seed=seed, dtype=BF16,
                     lam_random=True, h0_std=0.1, chunk=chunk,
                     name=f"long_prefill_bf16_B1_H16_T{T}_C{chunk}")


@dataclass
class DecodeCase:
    N: int
    H: int
    dk: int
    dv: int
    dtype: str
    scale: float
    log_lambda: np.ndarray
    q: np.ndarray   # [N, H, dk]
    k: np.ndarray   # [N, H, dk]
    v: np.ndarray   # [N, H, dv]
    S: np.ndarray   # [N, H, dk, dv] fp32
    name: str = ""

    def storage(self, x: np.ndarray) -> np.ndarray:
        if self.dtype == BF16:
            return bf16_bits(x)
        return np.ascontiguousarray(x, dtype=np.float32)


def make_decode_case(N: int, H: int, dk: int, dv: int, *, seed: int, dtype: str = BF16,
                     lam: Optional[np.ndarray] = None, S_std: float = 0.1,
                     scale: Optional[float] = None, name: str = "") -> DecodeCase:
    rng = np.random.default_rng(seed)
    q = _store(_normal(rng, (N, H, dk)), dtype)
    k = _store(_normal(rng, (N, H, dk)), dtype)
    v = _store(_normal(rng, (N, H, dv)), dtype)
    S = _normal(rng, (N, H, dk, dv), S_std)
    lam_arr = decay_layer_schedule(H) if lam is None else np.broadcast_to(
        np.asarray(lam, dtype=np.float64), (H,)).copy()
    if scale is None:
        scale = 1.0 / math.sqrt(dk)
    return DecodeCase(N=N, H=H, dk=dk, dv=dv, dtype=dtype, scale=float(np.float32(scale)),
                      log_lambda=log_lambda_of(lam_arr), q=q, k=k, v=v, S=S, name=name)


def serving_decode(seed: int = 3, N: int = 1280, layer: int = 0) -> DecodeCase:
    """Serving decode step: N=1,280 sequences x H=16 heads, one token each,
    state S ~ N(0, 0.1) fp32; each layer of the 24 draws from seed + 1000*layer."""
    return make_decode_case(N, LAYER_H, LAYER_DK, LAYER_DV, seed=seed + 1000 * layer,
                            dtype=BF16, name=f"serving_decode_bf16_N{N}_H16_layer{layer}")


def decode_tokens(N: int, H: int, dk: int, dv: int, *, seed: int, dtype: str = BF16) -> dict:
    """Only the per-token q, k, v of a decode step (same draw order and
    distribution as make_decode_case, without drawing the state)."""
    rng = np.random.default_rng(seed)
    q = _store(_normal(rng, (N, H, dk)), dtype)
    k = _store(_normal(rng, (N, H, dk)), dtype)
    v = _store(_normal(rng, (N, H, dv)), dtype)
    return {"q": q, "k": k, "v": v}


# ------------------------------------------------- variable-length prefill
@dataclass
class VarlenCase:
    """Sequences of different lengths packed token-major ([total_T, H, d]),
    with their states in a pool of n_slots fp32 states [n_slots, H, dk, dv]."""
    lengths: np.ndarray      # [nseq] int
    cu_seqlens: np.ndarray   # [nseq + 1] int32
    slots: np.ndarray        # [nseq] int32, distinct
    H: int
    dk: int
    dv: int
    scale: float
    log_lambda: np.ndarray   # [H] fp32
    q: np.ndarray            # [total_T, H, dk]
    k: np.ndarray
    v: np.ndarray            # [total_T, H, dv]
    pool: np.ndarray         # [n_slots, H, dk, dv] fp32


def make_varlen_case(lengths, H: int, *, seed: int, n_slots: Optional[int] = None, dk: int = 96, dv: int = 192,
                     pool_std: float = 0.1, lam_range=(0.9, 0.9999), dtype: str = BF16) -> VarlenCase:
    """Given lengths, draw packed q, k, v ~ N(0, 1), a pool of states
    ~ N(0, pool_std), distinct slots (a random subset of the pool, in random
    order) and log-uniform per-head decays, in that order."""
    rng = np.random.default_rng(seed)
    lengths = np.asarray(lengths, dtype=np.int64)
    nseq = len(lengths)
    n_slots = nseq if n_slots is None else n_slots
    cu = np.zeros(nseq + 1, dtype=np.int32)
    cu[1:] = np.cumsum(lengths)
    total = int(cu[-1])
    q = _normal(rng, (total, H, dk))
    k = _normal(rng, (total, H, dk))
    v = _normal(rng, (total, H, dv))
    pool = _normal(rng, (n_slots, H, dk, dv), pool_std)
    slots = rng.permutation(n_slots)[:nseq].astype(np.int32)
    lam = decay_log_uniform(rng, H, *lam_range)
    return VarlenCase(lengths=lengths, cu_seqlens=cu, slots=slots, H=H, dk=dk, dv=dv,
                      scale=float(np.float32(1.0 / math.sqrt(dk))), log_lambda=log_lambda_of(lam),
                      q=_store(q, dtype), k=_store(k, dtype), v=_store(v, dtype), pool=pool)


def serving_prefill_lengths(seed: int = 5, nseq: int = 64, lo: int = 64, hi: int = 4096) -> np.ndarray:
    """Prompt lengths of a batch of staggered requests: log-uniform integers in [lo, hi]."""
    rng = np.random.default_rng(seed)
    return np.floor(np.exp(rng.uniform(math.log(lo), math.log(hi + 1), size=nseq))).astype(np.int64)


# ------------------------------------------------------- the token Conv1d
D_MODEL = 3072   # the residual width D of the Laplace 3B layer


@dataclass
class ConvCase:
    """Inputs of the causal depthwise Conv1d: x [B, T, D] (LayerNorm output,
    N(0, 1)), taps w [D, 4] and bias b [D] ~ U(-1/2, 1/2) (PyTorch's default
    bound for a depthwise width-4 Conv1d, 1/sqrt(fan_in = 4)), and fp32 conv
    windows [B, 4, D] ~ N(0, 1) (the previous inputs of each sequence)."""
    x: np.ndarray
    w: np.ndarray
    b: np.ndarray
    window: np.ndarray
    dtype: str


def make_conv_case(B: int, T: int, D: int = D_MODEL, *, seed: int, dtype: str = BF16) -> ConvCase:
    """Draw x, w, b, window in that order. The window holds previous inputs,
    so it is drawn on the same grid as x (bf16 values for bf16 x)."""
    rng = np.random.default_rng(seed)
    x = _store(_normal(rng, (B, T, D)), dtype)
    w = rng.uniform(-0.5, 0.5, size=(D, 4)).astype(np.float32)
    b = rng.uniform(-0.5, 0.5, size=D).astype(np.float32)
    window = _store(_normal(rng, (B, 4, D)), dtype).astype(np.float32)
    return ConvCase(x=x, w=w, b=b, window=window, dtype=dtype)
