"""GPU parity of libgla against the double-precision oracle, through the C
ABI (ctypes binding), on seeded inputs that span several chunks and a ragged
tail, plus the degenerate cases of the method (lambda = 0, lambda = 1, T = 1,
T = 0, no initial state, no final state wanted).

Bars (max |gpu - ref| / max |ref| per output tensor): 2e-2 for bf16 inputs,
1e-4 for the fp32 validation mode."""
import math

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


def run_fwd(gla, c, chunk=None, want_hT=True):
    d = case_to_dev(c)
    o, hT = gla.gla_chunk_fwd(d["q"], d["k"], d["v"], d["ll"], d["h0"], c.scale, chunk or c.chunk,
                              want_hT=want_hT)
    gla.gla_check()
    return to_host(o), to_host(hT)


def check_fwd(gla, c, chunk=None):
    o, hT = run_fwd(gla, c, chunk)
    ro, rhT = oracle.fwd_recurrent(c.q, c.k, c.v, c.log_lambda, c.h0, c.scale)
    eo, eh = relerr(o, ro), relerr(hT, rhT)
    assert eo <= TOL[c.dtype], f"o rel err {eo:.3g}"
    assert eh <= TOL[c.dtype], f"hT rel err {eh:.3g}"
    return eo, eh


def check_bwd(gla, c, chunk=None):
    d = case_to_dev(c)
    dq, dk, dv, dh0 = gla.gla_chunk_bwd(d["q"], d["k"], d["v"], d["ll"], d["do"], d["h0"], d["dhT"],
                                        c.scale, chunk or c.chunk)
    gla.gla_check()
    ref = oracle.bwd(c.q, c.k, c.v, c.log_lambda, c.h0, c.scale, c.do, c.dhT)
    errs = [relerr(to_host(g), r) for g, r in zip((dq, dk, dv, dh0), ref)]
    for name, e in zip(("dq", "dk", "dv", "dh0"), errs):
        assert e <= TOL[c.dtype], f"{name} rel err {e:.3g}"
    return errs


# --------------------------------------------------------------- fp32 mode
def test_tiny_fwd_fp32_workload():
    """B=H=1, T=256 (two chunks of 128), lambda = 0.95, h0 = 0."""
    import linear_attention_chunk_gb300 as m
    c = gen.tiny_fp32()
    check_fwd(m, c)


@pytest.mark.parametrize("dk,dv,T,C", [(5, 7, 200, 64), (3, 1, 65, 64), (1, 4, 129, 128),
                                       (96, 192, 300, 128), (17, 33, 1, 64), (128, 256, 130, 128)])
def test_fwd_fp32_shapes(gla, dk, dv, T, C):
    c = gen.make_case(2, T, 3, dk, dv, seed=11 + dk, dtype="fp32", lam_random=True, lam_range=(0.5, 0.999),
                      h0_std=0.5, chunk=C)
    check_fwd(gla, c)


@pytest.mark.parametrize("lam", [0.0, 1.0])
def test_fwd_fp32_lambda_extremes(gla, lam):
    c = gen.make_case(1, 150, 2, 8, 12, seed=21, dtype="fp32", lam=lam, h0_std=0.3, chunk=64)
    check_fwd(gla, c)


@pytest.mark.parametrize("dk,dv,T,C", [(5, 7, 150, 64), (96, 192, 260, 128), (2, 3, 1, 64)])
def test_bwd_fp32(gla, dk, dv, T, C):
    c = gen.make_case(2, T, 2, dk, dv, seed=31 + T, dtype="fp32", lam_random=True, lam_range=(0.3, 0.999),
                      h0_std=0.5, with_grad=True, dhT_std=0.3, chunk=C)
    check_bwd(gla, c)


def test_decode_fp32(gla):
    dc = gen.make_decode_case(7, 3, 96, 192, seed=41, dtype="fp32")
    q, k, v = to_dev(dc.q, "fp32"), to_dev(dc.k, "fp32"), to_dev(dc.v, "fp32")
    S = f32_dev(dc.S)
    o = gla.gla_decode_step(q, k, v, f32_dev(dc.log_lambda), S, dc.scale)
    gla.gla_check()
    ro, rS = oracle.decode(dc.q, dc.k, dc.v, dc.log_lambda, dc.S, dc.scale)
    assert relerr(to_host(o), ro) <= TOL["fp32"]
    assert relerr(to_host(S), rS) <= TOL["fp32"]


def test_decode_fp32_generic_dims(gla):
    dc = gen.make_decode_case(5, 2, 7, 11, seed=42, dtype="fp32")
    S = f32_dev(dc.S)
    o = gla.gla_decode_step(to_dev(dc.q, "fp32"), to_dev(dc.k, "fp32"), to_dev(dc.v, "fp32"),
                            f32_dev(dc.log_lambda), S, dc.scale)
    gla.gla_check()
    ro, rS = oracle.decode(dc.q, dc.k, dc.v, dc.log_lambda, dc.S, dc.scale)
    assert relerr(to_host(o), ro) <= TOL["fp32"] and relerr(to_host(S), rS) <= TOL["fp32"]


# --------------------------------------------------------------- bf16 path
@pytest.mark.parametrize("T,C", [(300, 128), (300, 64), (128, 128), (1, 128), (129, 64), (700, 128)])
def test_fwd_bf16_ragged(gla, T, C):
    c = gen.make_case(2, T, 3, 96, 192, seed=51 + T + C, dtype="bf16", normalise_k=True, h0_std=0.1, chunk=C)
    check_fwd(gla, c)


@pytest.mark.parametrize("T,C", [(300, 128), (260, 64), (1, 128), (129, 64)])
def test_fwd_bf16_one_cta_per_chain(gla, T, C):
    """More chains than half the SMs run one CTA per (b, h), which holds the
    whole state; fewer chains run two CTAs each (the cases above). Ragged T,
    both chunk lengths, the page schedule with lambda = 0 and lambda = 1 among
    the 80 heads, h0 and hT."""
    lam = np.tile(gen.decay_page_schedule(16), 5)
    lam[3] = 0.0
    lam[21] = 1.0
    c = gen.make_case(1, T, 80, 96, 192, seed=57 + T + C, dtype="bf16", lam=lam, normalise_k=True, h0_std=0.1,
                      chunk=C)
    check_fwd(gla, c)


def test_fwd_bf16_page_schedule_and_lambda_zero(gla):
    lam = gen.decay_page_schedule(16)
    lam[3] = 0.0                      # lambda = 0: o_t = scale (q_t.k_t) v_t
    lam[5] = 1.0                      # lambda = 1: causal linear attention
    c = gen.make_case(1, 400, 16, 96, 192, seed=61, dtype="bf16", lam=lam, h0_std=0.1, chunk=128)
    check_fwd(gla, c)


def test_fwd_bf16_unnormalised_long_decay(gla):
    c = gen.make_case(1, 1000, 4, 96, 192, seed=62, dtype="bf16", lam_random=True, h0_std=0.1, chunk=64)
    check_fwd(gla, c)


def test_fwd_without_state_outputs(gla):
    c = gen.make_case(1, 200, 2, 96, 192, seed=63, dtype="bf16", normalise_k=True, chunk=128)
    o, hT = run_fwd(gla, c, want_hT=False)
    assert hT is None
    ro, _ = oracle.fwd_recurrent(c.q, c.k, c.v, c.log_lambda, None, c.scale)
    assert relerr(o, ro) <= TOL["bf16"]


def test_fwd_empty_sequence_copies_state(gla):
    import torch
    h0 = torch.randn(2, 3, 96, 192, device="cuda")
    q = torch.empty(2, 0, 3, 96, device="cuda", dtype=torch.bfloat16)
    v = torch.empty(2, 0, 3, 192, device="cuda", dtype=torch.bfloat16)
    ll = torch.full((3,), math.log(0.9), device="cuda")
    o, hT = gla.gla_chunk_fwd(q, q, v, ll, h0)
    gla.gla_check()
    assert torch.equal(hT, h0)


def test_fwd_split_call_matches_single_call(gla):
    c = gen.make_case(2, 500, 2, 96, 192, seed=64, dtype="bf16", normalise_k=True, h0_std=0.1, chunk=128)
    d = case_to_dev(c)
    o, hT = gla.gla_chunk_fwd(d["q"], d["k"], d["v"], d["ll"], d["h0"], c.scale, 128)
    t1 = 200
    sl = lambda x: x[:, :t1].contiguous()
    sr = lambda x: x[:, t1:].contiguous()
    oa, ha = gla.gla_chunk_fwd(sl(d["q"]), sl(d["k"]), sl(d["v"]), d["ll"], d["h0"], c.scale, 128)
    ob, hb = gla.gla_chunk_fwd(sr(d["q"]), sr(d["k"]), sr(d["v"]), d["ll"], ha, c.scale, 128)
    gla.gla_check()
    import torch
    assert relerr(to_host(torch.cat([oa, ob], 1)), to_host(o)) <= TOL["bf16"]
    assert relerr(to_host(hb), to_host(hT)) <= TOL["bf16"]


@pytest.mark.parametrize("T,C", [(300, 128), (260, 64), (1, 128)])
def test_bwd_bf16(gla, T, C):
    c = gen.make_case(2, T, 2, 96, 192, seed=71 + T, dtype="bf16", normalise_k=True, h0_std=0.02,
                      with_grad=True, dhT_std=0.02, chunk=C)
    check_bwd(gla, c)


@pytest.mark.parametrize("B,H", [(1, 1), (1, 3), (3, 5)])
def test_bwd_bf16_odd_head_count(gla, B, H):
    """dk and dv run in one launch whose CTAs come in groups of four (two
    (b, h) chains each); an odd number of chains ends in a group of two."""
    c = gen.make_case(B, 200, H, 96, 192, seed=73 + B * H, dtype="bf16", normalise_k=True, h0_std=0.05,
                      with_grad=True, dhT_std=0.05, lam_random=True, chunk=128)
    check_bwd(gla, c)


def test_bwd_bf16_page_schedule(gla):
    lam = gen.decay_page_schedule(16)
    lam[2] = 0.0
    c = gen.make_case(1, 333, 16, 96, 192, seed=72, dtype="bf16", lam=lam, h0_std=0.1,
                      with_grad=True, dhT_std=0.1, chunk=128)
    check_bwd(gla, c)


def test_decode_bf16(gla):
    dc = gen.make_decode_case(33, 16, 96, 192, seed=81, dtype="bf16")
    S = f32_dev(dc.S)
    o = gla.gla_decode_step(to_dev(dc.q, "bf16"), to_dev(dc.k, "bf16"), to_dev(dc.v, "bf16"),
                            f32_dev(dc.log_lambda), S, dc.scale)
    gla.gla_check()
    ro, rS = oracle.decode(dc.q, dc.k, dc.v, dc.log_lambda, dc.S, dc.scale)
    assert relerr(to_host(o), ro) <= TOL["bf16"]
    assert relerr(to_host(S), rS) <= 1e-5   # the state itself stays fp32


def test_prefill_then_decode_matches_longer_prefill(gla):
    """Serving hand-off: hT of a prefill feeds the decode state page."""
    import torch
    c = gen.make_case(3, 260, 16, 96, 192, seed=82, dtype="bf16", normalise_k=True, chunk=128)
    d = case_to_dev(c)
    t1 = 256
    sl = lambda x: x[:, :t1].contiguous()
    _, S = gla.gla_chunk_fwd(sl(d["q"]), sl(d["k"]), sl(d["v"]), d["ll"], None, c.scale, 128)
    ro, rhT = oracle.fwd_recurrent(c.q, c.k, c.v, c.log_lambda, None, c.scale)
    for t in range(t1, 260):
        o = gla.gla_decode_step(d["q"][:, t].contiguous(), d["k"][:, t].contiguous(),
                                d["v"][:, t].contiguous(), d["ll"], S, c.scale)
        assert relerr(to_host(o), ro[:, t]) <= TOL["bf16"]
    gla.gla_check()
    assert relerr(to_host(S), rhT) <= TOL["bf16"]


# ------------------------------------------------ long sequences, segmented
@pytest.mark.parametrize("T,C", [(5120, 128), (5000, 128), (2600, 64)])
def test_fwd_segmented_matches_oracle_and_single_chain(gla, T, C):
    """Few (b, h) pairs and a long sequence: the forward splits each sequence
    into segments (state-only pass, scan, then all segments at once). The
    result must match the oracle and the one-chain-per-(b, h) path."""
    import torch
    c = gen.make_case(1, T, 2, 96, 192, seed=91 + T, dtype="bf16", lam_random=True, h0_std=0.1, chunk=C)
    assert gla.gla_chunk_fwd_workspace_size(1, T, 2, 96, 192, C) > 0
    d = case_to_dev(c)
    o, hT = gla.gla_chunk_fwd(d["q"], d["k"], d["v"], d["ll"], d["h0"], c.scale, C)
    launches_seg = gla.gla_last_launch_count()
    empty = torch.empty(0, dtype=torch.uint8, device="cuda")
    o1, hT1 = gla.gla_chunk_fwd(d["q"], d["k"], d["v"], d["ll"], d["h0"], c.scale, C, workspace=empty)
    launches_one = gla.gla_last_launch_count()
    gla.gla_check()
    assert launches_seg == 3 and launches_one == 1
    ro, rh = oracle.fwd_recurrent(c.q, c.k, c.v, c.log_lambda, c.h0, c.scale)
    assert relerr(to_host(o), ro) <= TOL["bf16"]
    assert relerr(to_host(hT), rh) <= TOL["bf16"]
    assert relerr(to_host(o), to_host(o1)) <= TOL["bf16"]
    assert relerr(to_host(hT), to_host(hT1)) <= TOL["bf16"]
