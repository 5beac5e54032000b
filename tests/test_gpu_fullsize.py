"""Parity at the full sizes of the five named workloads, in the launch
configuration the benchmark times, against the double-precision oracle on
sampled outputs (whole batch rows or heads the oracle computes one by one).

  tiny fp32     B=1  H=1  T=256     lambda=0.95             (all outputs)
  layer fwd     B=8  H=16 T=2048    k L2-normalised         (all outputs)
  train f+b     B=16 H=16 T=2048    h0 ~ N(0,0.02)          (batch rows 0 and 15)
  decode        N=1280 H=16         S ~ N(0,0.1), 1 layer   (all outputs)
  long prefill  B=1  H=16 T=65536   C=64 and C=128          (heads 0, 7, 15; C=64 vs C=128 all)
"""
import numpy as np
import pytest

import gla_gen as gen
import oracle
from gpu_util import TOL, case_to_dev, f32_dev, relerr, to_dev, to_host

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def gla():
    import linear_attention_chunk_gb300 as m
    from linear_attention_chunk_gb300.build import build
    build()
    return m


def test_tiny_fp32(gla):
    c = gen.tiny_fp32()
    d = case_to_dev(c)
    o, hT = gla.gla_chunk_fwd(d["q"], d["k"], d["v"], d["ll"], None, c.scale, 128)
    gla.gla_check()
    ro, rh = oracle.fwd_recurrent(c.q, c.k, c.v, c.log_lambda, None, c.scale)
    assert relerr(to_host(o), ro) <= TOL["fp32"]
    assert relerr(to_host(hT), rh) <= TOL["fp32"]


def test_layer_forward_full(gla):
    c = gen.layer_fwd()
    d = case_to_dev(c)
    o, hT = gla.gla_chunk_fwd(d["q"], d["k"], d["v"], d["ll"], None, c.scale, 128)
    gla.gla_check()
    ro, rh = oracle.fwd_recurrent(c.q, c.k, c.v, c.log_lambda, None, c.scale)
    assert relerr(to_host(o), ro) <= TOL["bf16"]
    assert relerr(to_host(hT), rh) <= TOL["bf16"]


def test_train_forward_backward_full(gla):
    c = gen.train_fwd_bwd()
    d = case_to_dev(c)
    o, hT = gla.gla_chunk_fwd(d["q"], d["k"], d["v"], d["ll"], d["h0"], c.scale, 128)
    dq, dk, dv, dh0 = gla.gla_chunk_bwd(d["q"], d["k"], d["v"], d["ll"], d["do"], d["h0"], None, c.scale, 128)
    gla.gla_check()
    rows = [0, c.B - 1]
    sl = lambda x: x[rows]
    ro, rh = oracle.fwd_recurrent(sl(c.q), sl(c.k), sl(c.v), c.log_lambda, sl(c.h0), c.scale)
    assert relerr(to_host(o)[rows], ro) <= TOL["bf16"]
    assert relerr(to_host(hT)[rows], rh) <= TOL["bf16"]
    ref = oracle.bwd(sl(c.q), sl(c.k), sl(c.v), c.log_lambda, sl(c.h0), c.scale, sl(c.do), None)
    for name, g, r in zip(("dq", "dk", "dv", "dh0"), (dq, dk, dv, dh0), ref):
        e = relerr(to_host(g)[rows], r)
        assert e <= TOL["bf16"], f"{name} {e:.3g}"
    # every row is finite and the unsampled rows are not left unwritten
    for g in (dq, dk, dv, dh0):
        assert bool(g.isfinite().all())


def test_serving_decode_full(gla):
    dc = gen.serving_decode()
    S = f32_dev(dc.S)
    o = gla.gla_decode_step(to_dev(dc.q, "bf16"), to_dev(dc.k, "bf16"), to_dev(dc.v, "bf16"),
                            f32_dev(dc.log_lambda), S, dc.scale)
    gla.gla_check()
    ro, rS = oracle.decode(dc.q, dc.k, dc.v, dc.log_lambda, dc.S, dc.scale)
    assert relerr(to_host(o), ro) <= TOL["bf16"]
    assert relerr(to_host(S), rS) <= 1e-5


def test_long_prefill_full(gla):
    c128 = gen.long_prefill(chunk=128)
    d = case_to_dev(c128)
    outs = {}
    for C in (64, 128):
        o, hT = gla.gla_chunk_fwd(d["q"], d["k"], d["v"], d["ll"], d["h0"], c128.scale, C)
        gla.gla_check()
        outs[C] = (to_host(o), to_host(hT))
    # C=64 and C=128 agree with each other over every output
    assert relerr(outs[64][0], outs[128][0]) <= TOL["bf16"]
    assert relerr(outs[64][1], outs[128][1]) <= TOL["bf16"]
    heads = [0, 7, 15]
    sl = lambda x: np.ascontiguousarray(x[:, :, heads])
    ro, rh = oracle.fwd_recurrent(sl(c128.q), sl(c128.k), sl(c128.v), c128.log_lambda[heads],
                                  np.ascontiguousarray(c128.h0[:, heads]), c128.scale)
    for C in (64, 128):
        assert relerr(outs[C][0][:, :, heads], ro) <= TOL["bf16"], C
        assert relerr(outs[C][1][:, heads], rh) <= TOL["bf16"], C
