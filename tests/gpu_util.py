"""Helpers for the GPU parity tests: move generator cases to the device in
the library's storage types and measure the parity error.

Parity metric (per output tensor): max |gpu - ref| / max |ref|, against the
double-precision oracle run on exactly the values the GPU received.
Bars: 2e-2 for bf16 inputs, 1e-4 for the fp32 validation mode."""
import numpy as np

import gla_gen as gen

TOL = {"bf16": 2e-2, "fp32": 1e-4}


def torch_mod():
    import torch
    return torch


def to_dev(x, dtype):
    """fp32 numpy array (bf16-exact values when dtype == 'bf16') -> CUDA tensor."""
    torch = torch_mod()
    if x is None:
        return None
    if dtype == "bf16":
        bits = gen.bf16_bits(x)
        return torch.from_numpy(bits.view(np.int16)).cuda().view(torch.bfloat16)
    return torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32)).cuda()


def f32_dev(x):
    torch = torch_mod()
    if x is None:
        return None
    return torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32)).cuda()


def to_host(t):
    if t is None:
        return None
    return t.float().cpu().numpy().astype(np.float64)


def relerr(got, ref):
    got = np.asarray(got, np.float64)
    ref = np.asarray(ref, np.float64)
    assert got.shape == ref.shape, (got.shape, ref.shape)
    assert np.all(np.isfinite(got)), "non-finite GPU output"
    den = np.max(np.abs(ref)) if ref.size else 0.0
    if den == 0.0:
        return float(np.max(np.abs(got))) if got.size else 0.0
    return float(np.max(np.abs(got - ref)) / den)


def case_to_dev(c):
    return dict(q=to_dev(c.q, c.dtype), k=to_dev(c.k, c.dtype), v=to_dev(c.v, c.dtype),
                ll=f32_dev(c.log_lambda), h0=f32_dev(c.h0),
                do=to_dev(c.do, c.dtype) if c.do is not None else None, dhT=f32_dev(c.dhT))
