"""GPU parity of the mixer epilogue (self-augmentation, Head RMSNorm, SiLU(g)
gate) against the oracle: the standalone kernel over forward outputs, and the
decode step with the epilogue fused, in bf16 and in the fp32 validation mode."""
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
