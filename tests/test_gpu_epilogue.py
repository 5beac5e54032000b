"""GPU parity of the mixer epilogue (self-augmentation, Head RMSNorm, SiLU(g)
gate) against the oracle: the standalone kernel over forward outputs, the
decode step with the epilogue fused, in bf16 and in the fp32 validation mode,
and the chunked forward followed by the epilogue in place (gla_chunk_fwd_mixer)."""
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


def weights(H, dk, dv, seed):
    """Random-init epilogue weights (none are trained here): aug ~ N(0, 0.3), norm_w ~ 1 + N(0, 0.1)."""
    rng = np.random.default_rng(seed)
    return (rng.normal(0, 0.3, size=(H, dk)).astype(np.float32),
            (1.0 + rng.normal(0, 0.1, size=(H, dv))).astype(np.float32))


@pytest.mark.parametrize("dtype,dk,dv", [("bf16", 96, 192), ("fp32", 96, 192), ("fp32", 40, 72)])
def test_epilogue_over_forward_output(gla, dtype, dk, dv):
    """gla_chunk_fwd then gla_mixer_epilogue; the oracle takes the GPU's o
    (the forward's own parity is tested elsewhere) and the same q, k, v, g."""
    c = gen.make_case(2, 300, 3, dk, dv, seed=600 + dk, dtype=dtype, lam_random=True, h0_std=0.1)
    d = case_to_dev(c)
    o, _ = gla.gla_chunk_fwd(d["q"], d["k"], d["v"], d["ll"], d["h0"], c.scale, 128)
    rng = np.random.default_rng(601)
    g = rng.normal(size=(2, 300, 3, dv))
    g = gen.bf16_round(g) if dtype == "bf16" else g.astype(np.float32)
    aug, nw = weights(3, dk, dv, 602)
    for a, w in ((aug, nw), (None, None)):
        z = gla.gla_mixer_epilogue(o, d["q"], d["k"], d["v"], to_dev(g, dtype), f32_dev(a), f32_dev(w), 1e-6)
        gla.gla_check()
        ref = oracle.mixer_epilogue(to_host(o), c.q, c.k, c.v, g, a, w, 1e-6)
        assert relerr(to_host(z), ref) <= TOL[dtype]


@pytest.mark.parametrize("dtype,dk,dv", [("bf16", 96, 192), ("fp32", 96, 192), ("fp32", 24, 160)])
def test_decode_step_with_fused_epilogue(gla, dtype, dk, dv):
    dc = gen.make_decode_case(37, 4, dk, dv, seed=610 + dv, dtype=dtype)
    S = f32_dev(dc.S)
    rng = np.random.default_rng(611)
    g = rng.normal(size=(37, 4, dv))
    g = gen.bf16_round(g) if dtype == "bf16" else g.astype(np.float32)
    aug, nw = weights(4, dk, dv, 612)
    z = gla.gla_decode_step_mixer(to_dev(dc.q, dtype), to_dev(dc.k, dtype), to_dev(dc.v, dtype),
                                  f32_dev(dc.log_lambda), S, to_dev(g, dtype), f32_dev(aug), f32_dev(nw), 1e-6,
                                  dc.scale)
    gla.gla_check()
    o_ref, S_ref = oracle.decode(dc.q, dc.k, dc.v, dc.log_lambda, dc.S.astype(np.float32), dc.scale)
    z_ref = oracle.mixer_epilogue(o_ref, dc.q, dc.k, dc.v, g, aug, nw, 1e-6)
    assert relerr(to_host(z), z_ref) <= TOL[dtype]
    assert relerr(to_host(S), S_ref) <= TOL[dtype]


def fused_case(B, T, H, seed, **kw):
    c = gen.make_case(B, T, H, 96, 192, seed=seed, **kw)
    rng = np.random.default_rng(seed + 1)
    g = gen.bf16_round(rng.normal(size=(B, T, H, 192)))
    aug, nw = weights(H, 96, 192, seed + 2)
    return c, g, aug, nw


def fused_reference(c, g, aug, nw, eps):
    """The oracle's forward in double, then its epilogue: no rounding of o.
    Also returns each row's conditioning kappa = (rms(o) + rms(gate v)) / rms(u):
    where o and the gated value nearly cancel, the Head RMSNorm divides by a
    small rms(u) and magnifies the forward's own bf16 error (P is rounded to
    bf16 on the tensor core) by kappa."""
    o, hT = oracle.fwd_recurrent(c.q, c.k, c.v, c.log_lambda, c.h0, c.scale)
    z = oracle.mixer_epilogue(o, c.q, c.k, c.v, g, aug, nw, eps)
    q, k, v = (np.asarray(x, np.float64) for x in (c.q, c.k, c.v))
    a = np.zeros(q.shape[-2:]) if aug is None else np.asarray(aug, np.float64)
    gv = v / (1.0 + np.exp(-(q * a * k).sum(-1)))[..., None]
    rms = lambda x: np.sqrt((x * x).mean(-1))
    kappa = (rms(o) + rms(gv)) / np.maximum(rms(o + gv), 1e-30)
    return z, hT, kappa


def check_fused(z, ref, kappa, tol=TOL["bf16"]):
    """Every row within tol * max|ref| times its conditioning (at least 1); the
    rows with kappa <= 4 -- all but a few degenerate ones in a large case --
    meet the plain bar."""
    err = np.abs(np.asarray(z, np.float64) - ref).max(-1)
    den = np.abs(ref).max()
    assert np.all(err <= tol * den * np.maximum(kappa, 1.0)), float((err / (den * np.maximum(kappa, 1.0))).max())
    good = kappa <= 4.0
    assert good.any() and (good.size < 1000 or good.mean() > 0.99)
    assert err[good].max() <= tol * den


@pytest.mark.parametrize("C", [128, 64])
@pytest.mark.parametrize("T", [300, 128, 1])
def test_forward_with_epilogue(gla, C, T):
    """gla_chunk_fwd_mixer against the oracle's forward + epilogue: ragged tail,
    exact chunks and a single token, with h0 and random decays; its hT is the
    plain forward's bit for bit (the state path is the same)."""
    import torch
    c, g, aug, nw = fused_case(2, T, 4, 620 + T + C, lam_random=True, h0_std=0.1)
    d = case_to_dev(c)
    gd = to_dev(g, "bf16")
    for a, w in ((aug, nw), (None, None)):
        z, hT = gla.gla_chunk_fwd_mixer(d["q"], d["k"], d["v"], gd, d["ll"], d["h0"], c.scale, C, f32_dev(a),
                                        f32_dev(w), 1e-6)
        gla.gla_check()
        ref, hT_ref, kappa = fused_reference(c, g, a, w, 1e-6)
        check_fused(to_host(z), ref, kappa)
        _, hT_plain = gla.gla_chunk_fwd(d["q"], d["k"], d["v"], d["ll"], d["h0"], c.scale, C)
        gla.gla_check()
        assert torch.equal(hT, hT_plain)


@pytest.mark.parametrize("T", [300, 128, 1])
def test_forward_with_epilogue_fused(gla, T):
    """With more chains than half the SMs (80 here) and 128-token chunks the
    forward's output stage normalises each row (u = o + sigmoid(q.(aug k)) v
    over its rms, o never stored) and a light second pass applies the norm
    weight and the SiLU gate: ragged tail, exact chunks and a single token,
    with h0, random decays, and with and without aug and norm_w. Its hT is
    the plain forward's bit for bit."""
    import torch
    c, g, aug, nw = fused_case(1, T, 80, 660 + T, lam_random=True, h0_std=0.1)
    d = case_to_dev(c)
    gd = to_dev(g, "bf16")
    for a, w in ((aug, nw), (None, None)):
        z, hT = gla.gla_chunk_fwd_mixer(d["q"], d["k"], d["v"], gd, d["ll"], d["h0"], c.scale, 128, f32_dev(a),
                                        f32_dev(w), 1e-6)
        assert gla.gla_last_launch_count() == 2
        gla.gla_check()
        ref, hT_ref, kappa = fused_reference(c, g, a, w, 1e-6)
        check_fused(to_host(z), ref, kappa)
        _, hT_plain = gla.gla_chunk_fwd(d["q"], d["k"], d["v"], d["ll"], d["h0"], c.scale, 128)
        gla.gla_check()
        assert torch.equal(hT, hT_plain)


def test_forward_epilogue_page_schedule(gla):
    """The page decay schedule (lambda_0 = 0.5 underflows inside a chunk); the
    separate calls (forward, then the standalone epilogue into a new buffer)
    meet the same bar. This case holds a row with kappa = 106 (token 1 of
    head 13: o is within 2 % of minus the gated value), where the result is
    off by 2-3 % of max|z|."""
    lam = gen.decay_page_schedule(16)
    c, g, aug, nw = fused_case(1, 260, 16, 630, lam=lam)
    d = case_to_dev(c)
    gd = to_dev(g, "bf16")
    z, _ = gla.gla_chunk_fwd_mixer(d["q"], d["k"], d["v"], gd, d["ll"], None, c.scale, 128, f32_dev(aug),
                                   f32_dev(nw), 1e-5)
    o, _ = gla.gla_chunk_fwd(d["q"], d["k"], d["v"], d["ll"], None, c.scale, 128)
    z2 = gla.gla_mixer_epilogue(o, d["q"], d["k"], d["v"], gd, f32_dev(aug), f32_dev(nw), 1e-5)
    gla.gla_check()
    ref, _, kappa = fused_reference(c, g, aug, nw, 1e-5)
    check_fused(to_host(z), ref, kappa)
    check_fused(to_host(z2), ref, kappa)


def test_forward_epilogue_segmented_long_sequence(gla):
    """Few (b, h) pairs and a long sequence: the forward splits each sequence
    into segments run in parallel (workspace given); the epilogue is per token
    and gives the oracle's z."""
    c, g, aug, nw = fused_case(1, 8192, 2, 640, lam_random=True, h0_std=0.1)
    d = case_to_dev(c)
    assert gla.gla_chunk_fwd_workspace_size(1, 8192, 2, 96, 192, 128) > 0
    z, hT = gla.gla_chunk_fwd_mixer(d["q"], d["k"], d["v"], to_dev(g, "bf16"), d["ll"], d["h0"], c.scale, 128,
                                    f32_dev(aug), f32_dev(nw), 1e-6)
    gla.gla_check()
    ref, hT_ref, kappa = fused_reference(c, g, aug, nw, 1e-6)
    check_fused(to_host(z), ref, kappa)
    assert relerr(to_host(hT), hT_ref) <= TOL["bf16"]


def test_forward_epilogue_full_size_sampled_heads(gla):
    """The layer-forward workload (8 x 2048 x 16, one launch as the benchmark
    times it): every token of a sample of (b, h) pairs against the oracle."""
    c, g, aug, nw = fused_case(8, 2048, 16, 650, lam=gen.decay_layer_schedule(16), normalise_k=True)
    d = case_to_dev(c)
    z, _ = gla.gla_chunk_fwd_mixer(d["q"], d["k"], d["v"], to_dev(g, "bf16"), d["ll"], None, c.scale, 128,
                                   f32_dev(aug), f32_dev(nw), 1e-6)
    gla.gla_check()
    zh = to_host(z)
    for b, h in ((0, 0), (3, 7), (7, 15), (5, 1)):
        sl = lambda x: x[b:b + 1, :, h:h + 1]
        one = gen.Case(**{**c.__dict__, "q": sl(c.q), "k": sl(c.k), "v": sl(c.v), "h0": None,
                          "log_lambda": c.log_lambda[h:h + 1]})
        ref, _, kappa = fused_reference(one, sl(g), aug[h:h + 1], nw[h:h + 1], 1e-6)
        check_fused(zh[b:b + 1, :, h:h + 1], ref, kappa)


def test_standalone_epilogue_on_the_oracle_output_kappa106(gla):
    """Where the widened bar of the fused forward comes from. On the page-
    schedule case with the kappa = 106 row, the standalone epilogue is fed the
    oracle's own forward output o (double), so the forward kernel's error is
    out of the picture:
      - bf16 mode, o rounded to bf16: the GPU result equals the oracle's
        epilogue of the same bf16 o within the plain bar (the kernel's own
        error), yet is off from the exact z by about 2.8 % of max|z| on the
        kappa = 106 row: rounding o to bf16 alone costs that much there;
      - fp32 mode, o in fp32: the plain fp32 bar (1e-4) against the exact z,
        on every row including kappa = 106."""
    lam = gen.decay_page_schedule(16)
    c, g, aug, nw = fused_case(1, 260, 16, 630, lam=lam)
    ref, _, kappa = fused_reference(c, g, aug, nw, 1e-5)
    assert kappa.max() > 100
    o, _ = oracle.fwd_recurrent(c.q, c.k, c.v, c.log_lambda, None, c.scale)
    ob = gen.bf16_round(o)
    z = gla.gla_mixer_epilogue(to_dev(ob, "bf16"), to_dev(c.q, "bf16"), to_dev(c.k, "bf16"), to_dev(c.v, "bf16"),
                               to_dev(g, "bf16"), f32_dev(aug), f32_dev(nw), 1e-5)
    gla.gla_check()
    zh = to_host(z)
    assert relerr(zh, oracle.mixer_epilogue(ob, c.q, c.k, c.v, g, aug, nw, 1e-5)) <= TOL["bf16"]
    row_err = np.abs(zh - ref).max(-1) / np.abs(ref).max()
    assert row_err[kappa > 100].max() > TOL["bf16"]          # bf16 storage of o, amplified by kappa
    assert row_err[kappa <= 4].max() <= TOL["bf16"]
    check_fused(zh, ref, kappa)
    z32 = gla.gla_mixer_epilogue(f32_dev(o), f32_dev(c.q), f32_dev(c.k), f32_dev(c.v), f32_dev(g), f32_dev(aug),
                                 f32_dev(nw), 1e-5)
    gla.gla_check()
    assert relerr(to_host(z32), ref) <= TOL["fp32"]
