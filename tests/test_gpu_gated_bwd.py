"""GPU parity of the backward of the per-token (data-dependent) decay against
the oracle's O11 (gradients of L = sum <do, o> + <dhT, hT>, the gate's own
dg included), through the C ABI: gla_chunk_bwd_gated on the tensor-core path
(bf16: dq, dk, dv, dh0 from the three chunk kernels in gated mode, dg from
the chunk-local kernel over their saved states) and on the validation path
(fp32).

Cases span several chunks and a ragged tail at both chunk lengths, h0 and
dhT nonzero, gates that clear the state on either side of the kernels'
32-column block edges and on a chunk's first and last token, strong decays
whose products underflow inside a chunk, a constant gate (which must give
the fixed-decay backward), and the training shape sampled.
Bars (max |gpu - ref| / max |ref| per output tensor): 2e-2 for bf16 inputs,
1e-4 for the fp32 validation mode."""
import numpy as np
import pytest

import gla_gen as gen
import oracle
from gpu_util import TOL, case_to_dev, f32_dev, relerr, to_host

pytestmark = pytest.mark.gpu

NAMES = ("dq", "dk", "dv", "dh0", "dg")


@pytest.fixture(scope="module")
def gla():
    import linear_attention_chunk_gb300 as m
    from linear_attention_chunk_gb300.build import build
    build()
    return m


def run_bwd(gla, c, g, chunk=None):
    d = case_to_dev(c)
    out = gla.gla_chunk_bwd_gated(d["q"], d["k"], d["v"], f32_dev(g), d["do"], d["h0"], d["dhT"], c.scale,
                                  chunk or c.chunk)
    gla.gla_check()
    return [to_host(x) for x in out]


def check_bwd(gla, c, g, chunk=None, tol=None):
    got = run_bwd(gla, c, g, chunk)
    ref = oracle.bwd_gated(c.q, c.k, c.v, g, c.h0, c.scale, c.do, c.dhT)
    tol = tol or TOL[c.dtype]
    errs = {n: relerr(x, r) for n, x, r in zip(NAMES, got, ref)}
    bad = {n: e for n, e in errs.items() if not e <= tol}
    assert not bad, f"rel err above {tol}: {bad} (all: {errs})"
    return got, ref, errs


def case(B, T, H, seed, C, gate="gla", dtype="bf16", dk=96, dv=192, **kw):
    return gen.make_case(B, T, H, dk, dv, seed=seed, dtype=dtype, normalise_k=(dtype == "bf16"), h0_std=0.1,
                         with_grad=True, dhT_std=0.05, chunk=C, gate=gate, **kw)


# --------------------------------------------------------------- bf16 path
@pytest.mark.parametrize("T,C", [(300, 128), (300, 64), (129, 64), (128, 128), (1, 128), (700, 128)])
def test_gated_bwd_bf16_ragged(gla, T, C):
    c = case(2, T, 3, 700 + T + C, C)
    check_bwd(gla, c, c.extra["g"])


@pytest.mark.parametrize("C", [128, 64])
def test_gated_bwd_bf16_clears_on_block_edges(gla, C):
    """P is built in 32-column blocks with the weights walked along the gates,
    leftwards (dq) and rightwards (dk, dv); dg's pair sums walk the same way.
    Clearing gates on either side of a block edge, two in one block, on a
    chunk's last and the next chunk's first token, on the first and the last
    token of the sequence; gates at and just above the clearing threshold."""
    c = case(1, 552, 7, 740 + C, C)
    g = c.extra["g"].copy()
    g[0, 31, 0] = -np.inf                  # a block's last column
    g[0, 32, 1] = -np.inf                  # the next block's first column
    g[0, 191:193, 2] = -np.inf             # both sides of an edge
    g[0, 352, 3] = -80.0                   # at the threshold
    g[0, 356, 3] = -79.0                   # just above it: a strong decay
    g[0, 389, 4] = -np.inf                 # two clears in one block
    g[0, 404, 4] = -np.inf
    g[0, 511:513, 5] = -np.inf             # a chunk's last and the next one's first token
    g[0, 0, 6] = -np.inf                   # the first token: h0 is cleared
    g[0, 551, 6] = -np.inf                 # the last token
    got, ref, _ = check_bwd(gla, c, g)
    # a clearing gate's own gradient is 0 (its decay does not depend on it)
    cleared = ~(g > -80.0)
    assert np.all(got[4][cleared] == 0.0)


def test_gated_bwd_bf16_strong_decays(gla):
    c = case(1, 400, 4, 760, 64, gate="wide")
    check_bwd(gla, c, c.extra["g"])


def test_gated_bwd_without_h0_and_dhT(gla):
    c = gen.make_case(2, 260, 4, 96, 192, seed=765, dtype="bf16", normalise_k=True, with_grad=True, chunk=128,
                      gate="gla")
    assert c.h0 is None and c.dhT is None
    got, ref, _ = check_bwd(gla, c, c.extra["g"])


def test_constant_gate_matches_fixed_decay_backward(gla):
    """g_t = ln lambda_h for every token: dq, dk, dv, dh0 are those of
    gla_chunk_bwd, and the gate gradients of a head sum to its log-lambda
    gradient (the oracle's O3 with the decay's own gradient written out)."""
    c = gen.make_case(2, 333, 16, 96, 192, seed=770, dtype="bf16", normalise_k=True, h0_std=0.1, with_grad=True,
                      dhT_std=0.05, chunk=128)
    g = np.broadcast_to(c.log_lambda.astype(np.float32), (c.B, c.T, c.H)).copy()
    got = run_bwd(gla, c, g)
    d = case_to_dev(c)
    fixed = gla.gla_chunk_bwd(d["q"], d["k"], d["v"], d["ll"], d["do"], d["h0"], d["dhT"], c.scale, 128)
    gla.gla_check()
    ref3 = oracle.bwd(c.q, c.k, c.v, c.log_lambda, c.h0, c.scale, c.do, c.dhT)
    for n, x, f, r in zip(NAMES, got, fixed, ref3):
        assert relerr(x, r) <= TOL["bf16"], n
        assert relerr(x, to_host(f)) <= TOL["bf16"], n
    ref11 = oracle.bwd_gated(c.q, c.k, c.v, g, c.h0, c.scale, c.do, c.dhT)
    assert relerr(got[4], ref11[4]) <= TOL["bf16"]
    assert relerr(got[4].sum(1), ref11[4].sum(1)) <= TOL["bf16"]


def test_gated_bwd_training_shape_sampled(gla):
    """The training workload's shape (16 x 2048 x 16, chunk 128) with gated
    linear attention's gates, in one launch set as the benchmark times it:
    every token of a sample of (b, h) pairs against the oracle."""
    c = gen.make_case(16, 2048, 16, 96, 192, seed=780, dtype="bf16", normalise_k=True, h0_std=0.02,
                      with_grad=True, chunk=128, gate="gla")
    got = run_bwd(gla, c, c.extra["g"])
    for b, h in ((0, 0), (7, 9), (15, 15), (3, 4)):
        sl = lambda x: x[b:b + 1, :, h:h + 1]
        ref = oracle.bwd_gated(sl(c.q), sl(c.k), sl(c.v), sl(c.extra["g"]), c.h0[b:b + 1, h:h + 1], c.scale,
                               sl(c.do), None)
        for n, x, r in zip(NAMES, got, ref):
            part = x[b:b + 1, h:h + 1] if n == "dh0" else sl(x)
            assert relerr(part, r) <= TOL["bf16"], (n, b, h, relerr(part, r))


def test_gated_bwd_repeatable(gla):
    """Two calls on the same inputs give the same bits (no atomics, no stale
    workspace: every saved state is written before it is read)."""
    import torch
    c = case(2, 300, 3, 790, 128)
    d = case_to_dev(c)
    g = f32_dev(c.extra["g"])
    ws = torch.full((gla.gla_chunk_bwd_gated_workspace_size(2, 300, 3, 96, 192, 128),), 0x7f, dtype=torch.uint8,
                    device="cuda")
    a = gla.gla_chunk_bwd_gated(d["q"], d["k"], d["v"], g, d["do"], d["h0"], d["dhT"], c.scale, 128, workspace=ws)
    b = gla.gla_chunk_bwd_gated(d["q"], d["k"], d["v"], g, d["do"], d["h0"], d["dhT"], c.scale, 128, workspace=ws)
    gla.gla_check()
    for x, y in zip(a, b):
        assert torch.equal(x, y)


# --------------------------------------------------------------- fp32 mode
@pytest.mark.parametrize("dk,dv,T,C", [(5, 7, 150, 64), (96, 192, 300, 128), (3, 2, 1, 64), (8, 16, 260, 128)])
def test_gated_bwd_fp32(gla, dk, dv, T, C):
    c = case(2, T, 3, 800 + T + dk, C, dtype="fp32", dk=dk, dv=dv)
    g = c.extra["g"].copy()
    if T > 100:
        g[0, 70, 1] = -np.inf
        g[1, 64, 2] = -np.inf
    check_bwd(gla, c, g)


def test_gated_bwd_fp32_wide_gates(gla):
    c = case(1, 260, 2, 810, 128, gate="wide", dtype="fp32", dk=8, dv=16)
    check_bwd(gla, c, c.extra["g"])
