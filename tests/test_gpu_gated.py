"""GPU parity of the per-token (data-dependent) decay against the oracle's
gated recurrence (O9, O10), through the C ABI: gla_chunk_fwd_gated on the
tensor-core path (bf16) and the validation path (fp32), and
gla_decode_step_gated, and the packed variable-length prefill
gla_chunk_fwd_varlen_gated.

Cases span several chunks and a ragged tail, both chunk lengths, gates that
clear the state (-inf) inside a chunk and on a chunk's first token, strong
decays whose products underflow inside a chunk, a constant gate (which must
agree with the fixed-decay forward), and the layer-forward shape sampled.
Bars (max |gpu - ref| / max |ref| per output tensor): 2e-2 for bf16 inputs,
1e-4 for the fp32 validation mode."""
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


def run_gated(gla, c, g, chunk=None):
    d = case_to_dev(c)
    o, hT = gla.gla_chunk_fwd_gated(d["q"], d["k"], d["v"], f32_dev(g), d["h0"], c.scale, chunk or c.chunk)
    gla.gla_check()
    return to_host(o), to_host(hT)


def check_gated(gla, c, g, chunk=None):
    o, hT = run_gated(gla, c, g, chunk)
    ro, rhT = oracle.fwd_gated(c.q, c.k, c.v, g, c.h0, c.scale)
    eo, eh = relerr(o, ro), relerr(hT, rhT)
    assert eo <= TOL[c.dtype], f"o rel err {eo:.3g}"
    assert eh <= TOL[c.dtype], f"hT rel err {eh:.3g}"
    return eo, eh


# --------------------------------------------------------------- fp32 mode
@pytest.mark.parametrize("dk,dv,T,C", [(5, 7, 150, 64), (96, 192, 300, 128), (3, 2, 1, 64)])
def test_gated_fwd_fp32(gla, dk, dv, T, C):
    c = gen.make_case(2, T, 3, dk, dv, seed=300 + T, dtype="fp32", h0_std=0.3, chunk=C, gate="gla")
    g = c.extra["g"].copy()
    if T > 100:
        g[0, 70, 1] = -np.inf
    check_gated(gla, c, g)


def test_gated_fwd_fp32_wide_gates(gla):
    c = gen.make_case(1, 260, 2, 8, 16, seed=311, dtype="fp32", h0_std=0.3, chunk=128, gate="wide")
    check_gated(gla, c, c.extra["g"])


# --------------------------------------------------------------- bf16 path
@pytest.mark.parametrize("T,C", [(300, 128), (300, 64), (128, 128), (1, 128), (129, 64), (700, 128)])
def test_gated_fwd_bf16_ragged(gla, T, C):
    c = gen.make_case(2, T, 3, 96, 192, seed=320 + T + C, dtype="bf16", normalise_k=True, h0_std=0.1, chunk=C,
                      gate="gla")
    check_gated(gla, c, c.extra["g"])


def test_gated_fwd_bf16_clearing_gates(gla):
    c = gen.make_case(2, 520, 4, 96, 192, seed=331, dtype="bf16", normalise_k=True, h0_std=0.1, chunk=128,
                      gate="gla")
    g = c.extra["g"].copy()
    g[0, 45, 0] = -np.inf          # inside a chunk
    g[0, 128, 1] = -np.inf         # a chunk's first token: S_prev is cleared
    g[1, 127, 2] = -np.inf         # a chunk's last token
    g[1, 300:303, 3] = -np.inf     # a run of them
    g[1, 519, 0] = -np.inf         # the last token: hT = k v^T
    check_gated(gla, c, g)


@pytest.mark.parametrize("C", [128, 64])
@pytest.mark.parametrize("H", [6, 80])
def test_gated_fwd_bf16_clears_on_block_edges(gla, C, H):
    """The tensor-core kernels build P in 32-column blocks, walking each row's
    weights leftwards from the block's last column: clearing gates on either
    side of a block edge, two in one block, on a chunk's last and the next
    chunk's first token, and gates at and just above the kernel's clearing
    threshold (a log-decay of -80, whose exp is below 1e-34). 6 chains run two
    CTAs each (half the state each), 80 chains one CTA each (the whole state)."""
    c = gen.make_case(1, 552, H, 96, 192, seed=334 + C + H, dtype="bf16", normalise_k=True, h0_std=0.1, chunk=C,
                      gate="gla")
    g = c.extra["g"].copy()
    g[0, 31, 0] = -np.inf                  # a block's last column
    g[0, 32, 1] = -np.inf                  # the next block's first column
    g[0, 191:193, 2] = -np.inf             # both sides of an edge
    g[0, 352, 3] = -80.0                   # at the threshold
    g[0, 356, 3] = -79.0                   # just above it: a strong decay
    g[0, 389, 4] = -np.inf                 # two clears in one block
    g[0, 404, 4] = -np.inf
    g[0, 511:513, 5] = -np.inf             # a chunk's last and the next one's first token
    check_gated(gla, c, g)


def test_gated_fwd_bf16_strong_decays(gla):
    c = gen.make_case(1, 400, 4, 96, 192, seed=332, dtype="bf16", h0_std=0.1, chunk=64, gate="wide")
    check_gated(gla, c, c.extra["g"])


def test_constant_gate_matches_fixed_decay_forward(gla):
    c = gen.make_case(2, 333, 16, 96, 192, seed=333, dtype="bf16", normalise_k=True, h0_std=0.1, chunk=128)
    g = np.broadcast_to(c.log_lambda.astype(np.float32), (c.B, c.T, c.H)).copy()
    og, hg = run_gated(gla, c, g)
    d = case_to_dev(c)
    o, hT = gla.gla_chunk_fwd(d["q"], d["k"], d["v"], d["ll"], d["h0"], c.scale, 128)
    gla.gla_check()
    ro, rhT = oracle.fwd_recurrent(c.q, c.k, c.v, c.log_lambda, c.h0, c.scale)
    assert relerr(og, ro) <= TOL["bf16"] and relerr(hg, rhT) <= TOL["bf16"]
    # two kernels (decay tables against per-element exponentials) of one result
    assert relerr(og, to_host(o)) <= TOL["bf16"] and relerr(hg, to_host(hT)) <= TOL["bf16"]


def test_gated_layer_forward_sampled(gla):
    """The layer-forward shape (8 x 2048 x 16) with GLA-style gates; the
    oracle checks two batch rows, all heads."""
    c = gen.make_case(8, 2048, 16, 96, 192, seed=334, dtype="bf16", normalise_k=True, chunk=128, gate="gla")
    g = c.extra["g"]
    o, hT = run_gated(gla, c, g)
    for b in (0, 7):
        ro, rhT = oracle.fwd_gated(c.q[b:b + 1], c.k[b:b + 1], c.v[b:b + 1], g[b:b + 1], None, c.scale)
        assert relerr(o[b:b + 1], ro) <= TOL["bf16"], b
        assert relerr(hT[b:b + 1], rhT) <= TOL["bf16"], b


def test_gated_prefill_then_decode(gla):
    """hT of a gated prefill feeds gated decode steps; the result equals one
    longer gated prefill."""
    import torch
    c = gen.make_case(3, 261, 16, 96, 192, seed=335, dtype="bf16", normalise_k=True, chunk=128, gate="gla")
    g = c.extra["g"]
    d = case_to_dev(c)
    t1 = 257
    _, S = gla.gla_chunk_fwd_gated(d["q"][:, :t1].contiguous(), d["k"][:, :t1].contiguous(),
                                   d["v"][:, :t1].contiguous(), f32_dev(g[:, :t1]), None, c.scale, 128)
    outs = []
    for t in range(t1, c.T):
        outs.append(gla.gla_decode_step_gated(d["q"][:, t].contiguous(), d["k"][:, t].contiguous(),
                                              d["v"][:, t].contiguous(), f32_dev(g[:, t]), S, c.scale))
    gla.gla_check()
    ro, rhT = oracle.fwd_gated(c.q, c.k, c.v, g, None, c.scale)
    got = np.stack([to_host(x) for x in outs], axis=1)
    assert relerr(got, ro[:, t1:]) <= TOL["bf16"]
    assert relerr(to_host(S), rhT) <= TOL["bf16"]


# ------------------------------------------------------------------ decode
@pytest.mark.parametrize("dtype", ["bf16", "fp32"])
def test_gated_decode(gla, dtype):
    dc = gen.make_decode_case(37, 16, 96, 192, seed=340, dtype=dtype)
    rng = np.random.default_rng(341)
    g = gen.log_gates(rng, (37, 16), "wide")
    g[3, 5] = -np.inf
    S = f32_dev(dc.S)
    o = gla.gla_decode_step_gated(to_dev(dc.q, dtype), to_dev(dc.k, dtype), to_dev(dc.v, dtype), f32_dev(g), S,
                                  dc.scale)
    gla.gla_check()
    ro, rS = oracle.decode_gated(dc.q, dc.k, dc.v, g, dc.S, dc.scale)
    assert relerr(to_host(o), ro) <= TOL[dtype]
    assert relerr(to_host(S), rS) <= 1e-5   # the state itself stays fp32


# ------------------------------------------------------- variable-length prefill
@pytest.mark.parametrize("C", [128, 64])
@pytest.mark.parametrize("H", [4, 12])
def test_gated_varlen_matches_oracle_per_sequence(gla, C, H):
    """Packed prompts of mixed lengths with per-token gates, each from and
    into its slot of a state pool; an empty prompt leaves its slot as it is.
    32 (sequence, head) chains run two CTAs each, 96 chains one CTA each."""
    import torch
    lengths = [0, 1, 63, 65, 128, 129, 300, 700]
    c = gen.make_varlen_case(lengths, H, seed=600 + C + H, n_slots=11)
    rng = np.random.default_rng(601 + C + H)
    g = gen.log_gates(rng, (c.q.shape[0], H), "gla")
    g[5, 2] = -np.inf                     # clears the state of sequence 2's head 2 inside its prompt
    d = dict(q=to_dev(c.q, "bf16"), k=to_dev(c.k, "bf16"), v=to_dev(c.v, "bf16"),
             cu=torch.from_numpy(c.cu_seqlens).cuda(), slots=torch.from_numpy(c.slots).cuda(), pool=f32_dev(c.pool))
    o = gla.gla_chunk_fwd_varlen_gated(d["q"], d["k"], d["v"], f32_dev(g), d["cu"], d["pool"], d["slots"], c.scale, C)
    gla.gla_check()
    oh, pool = to_host(o), to_host(d["pool"])
    for n in range(len(lengths)):
        a, b = int(c.cu_seqlens[n]), int(c.cu_seqlens[n + 1])
        if b == a:
            assert np.array_equal(pool[c.slots[n]], c.pool[c.slots[n]].astype(np.float32).astype(np.float64))
            continue
        h0 = c.pool[c.slots[n]][None].astype(np.float32)
        ro, rh = oracle.fwd_gated(c.q[None, a:b], c.k[None, a:b], c.v[None, a:b], g[None, a:b], h0, c.scale)
        assert relerr(oh[a:b], ro[0]) <= TOL["bf16"], f"o of sequence {n} (length {b - a})"
        assert relerr(pool[c.slots[n]], rh[0]) <= TOL["bf16"], f"state of sequence {n}"


# ---------------------------------------------------- long sequences, segmented
@pytest.mark.parametrize("T,C", [(5120, 128), (5000, 128), (2600, 64)])
def test_gated_segmented_matches_oracle_and_single_chain(gla, T, C):
    """Few (b, h) and a long sequence: the forward splits it into segments
    whose decays are the exp of their summed gates. Clearing gates sit inside
    a segment and on a segment's first token. The result matches the oracle
    and the single-chain run (workspace too small to split)."""
    import torch
    c = gen.make_case(1, T, 2, 96, 192, seed=350 + T + C, dtype="bf16", normalise_k=True, h0_std=0.1, chunk=C,
                      gate="gla")
    assert gla.gla_chunk_fwd_gated_workspace_size(1, T, 2, 96, 192, C) > 0
    g = c.extra["g"].copy()
    g[0, 1500, 0] = -np.inf
    g[0, 8 * C, 1] = -np.inf          # the first token of the second segment when segments are 8 chunks long
    g[0, 9 * C, 0] = -np.inf          # ... and when they are 9 chunks long
    og, hg = run_gated(gla, c, g)
    ro, rhT = oracle.fwd_gated(c.q, c.k, c.v, g, c.h0, c.scale)
    assert relerr(og, ro) <= TOL["bf16"] and relerr(hg, rhT) <= TOL["bf16"]
    d = case_to_dev(c)
    small = torch.empty(16, dtype=torch.uint8, device="cuda")
    o1, h1 = gla.gla_chunk_fwd_gated(d["q"], d["k"], d["v"], f32_dev(g), d["h0"], c.scale, C, workspace=small)
    gla.gla_check()
    assert relerr(og, to_host(o1)) <= TOL["bf16"] and relerr(hg, to_host(h1)) <= TOL["bf16"]


def test_gated_calls_capture_and_replay_bit_exact(gla):
    """The gated forward (split into segments), the gated packed prefill and
    the gated serving step inside a CUDA graph replay to the bits of the same
    calls launched eagerly."""
    import torch
    c = gen.make_case(1, 4096, 2, 96, 192, seed=360, normalise_k=True, h0_std=0.1, chunk=128, gate="gla")
    d = case_to_dev(c)
    g = f32_dev(c.extra["g"])
    ws = torch.empty(max(gla.gla_chunk_fwd_gated_workspace_size(1, 4096, 2, 96, 192, 128), 16), dtype=torch.uint8,
                     device="cuda")
    vc = gen.make_varlen_case([70, 300, 5], 2, seed=361, n_slots=4)
    vd = dict(q=to_dev(vc.q, "bf16"), k=to_dev(vc.k, "bf16"), v=to_dev(vc.v, "bf16"),
              cu=torch.from_numpy(vc.cu_seqlens).cuda(), slots=torch.from_numpy(vc.slots).cuda())
    vg = f32_dev(gen.log_gates(np.random.default_rng(362), (vc.q.shape[0], 2), "gla"))
    dc = gen.make_decode_case(8, 2, 96, 192, seed=363)
    dg = f32_dev(gen.log_gates(np.random.default_rng(364), (8, 2), "wide"))
    dq_, dk_, dv_ = to_dev(dc.q, "bf16"), to_dev(dc.k, "bf16"), to_dev(dc.v, "bf16")

    def buffers():
        return dict(o=torch.empty_like(d["v"]), hT=torch.empty((1, 2, 96, 192), device="cuda"),
                    vo=torch.empty_like(vd["v"]), pool=f32_dev(vc.pool), S=f32_dev(dc.S),
                    od=torch.empty((8, 2, 192), dtype=torch.bfloat16, device="cuda"))

    def step(bf, s):
        gla.gla_chunk_fwd_gated(d["q"], d["k"], d["v"], g, d["h0"], c.scale, 128, o=bf["o"], hT=bf["hT"],
                                workspace=ws, stream=s)
        gla.gla_chunk_fwd_varlen_gated(vd["q"], vd["k"], vd["v"], vg, vd["cu"], bf["pool"], vd["slots"], vc.scale,
                                       128, o=bf["vo"], stream=s)
        gla.gla_decode_step_gated(dq_, dk_, dv_, dg, bf["S"], dc.scale, o=bf["od"], stream=s)

    s = torch.cuda.Stream()
    eager = buffers()
    with torch.cuda.stream(s):
        step(eager, s)
    torch.cuda.synchronize()
    gla.gla_check()
    with torch.cuda.stream(s):
        step(buffers(), s)            # warm-up outside the capture
    torch.cuda.synchronize()
    graphed = buffers()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=s):
        step(graphed, s)
    torch.cuda.synchronize()
    with torch.cuda.stream(s):
        graph.replay()
    torch.cuda.synchronize()
    gla.gla_check()
    for name in eager:
        assert torch.equal(eager[name], graphed[name]), name


def test_gated_varlen_bad_device_offsets_are_reported(gla):
    """A decreasing packed offset is skipped on the device and reported by
    gla_check, as in the fixed-decay prefill; the other sequences complete."""
    import torch
    vc = gen.make_varlen_case([100, 50, 80], 2, seed=365, n_slots=3)
    vc.slots[:] = np.arange(3, dtype=np.int32)
    g = gen.log_gates(np.random.default_rng(366), (vc.q.shape[0], 2), "gla")
    bad = vc.cu_seqlens.copy()
    bad[2] = bad[1] - 1
    pool = f32_dev(vc.pool)
    gla.gla_chunk_fwd_varlen_gated(to_dev(vc.q, "bf16"), to_dev(vc.k, "bf16"), to_dev(vc.v, "bf16"), f32_dev(g),
                                   torch.from_numpy(bad).cuda(), pool, None, vc.scale, 128)
    with pytest.raises(gla.GlaError) as ei:
        gla.gla_check()
    assert ei.value.status == gla.GLA_ERR_INVALID_ARG
    ph = to_host(pool)
    assert np.array_equal(ph[1], vc.pool[1].astype(np.float32).astype(np.float64))
    a, b = int(bad[0]), int(bad[1])
    _, rh = oracle.fwd_gated(vc.q[None, a:b], vc.k[None, a:b], vc.v[None, a:b], g[None, a:b],
                             vc.pool[0][None].astype(np.float32), vc.scale)
    assert relerr(ph[0], rh[0]) <= TOL["bf16"]
    gla.gla_check()
