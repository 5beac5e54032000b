"""Pins of the oracle's mixer epilogue (O7): properties that the self-
augmentation gate, the Head RMSNorm and the SiLU(g) output gate must have,
checked without retyping the oracle's formula.

Reading of the "GLA mixer" paragraph of "Beyond the KV cache: Training and
serving i14's Laplace 3B linear attention model on AWS Trainium2 with native
PyTorch" (its equations did not survive extraction): u = o + sigmoid(q.(a*k)) v,
y = w * u / sqrt(mean(u^2) + eps) over the head's dv channels, z = y * SiLU(g)."""
import numpy as np
import pytest

import oracle

pytestmark = pytest.mark.filterwarnings("ignore")


def case(seed, NT=5, H=3, dk=6, dv=8):
    rng = np.random.default_rng(seed)
    return dict(o=rng.normal(size=(NT, H, dv)), q=rng.normal(size=(NT, H, dk)), k=rng.normal(size=(NT, H, dk)),
                v=rng.normal(size=(NT, H, dv)), g=rng.normal(size=(NT, H, dv)), aug=rng.normal(size=(H, dk)),
                norm_w=rng.normal(size=(H, dv)))


def epi(c, **kw):
    a = dict(c)
    a.update(kw)
    return oracle.mixer_epilogue(a["o"], a["q"], a["k"], a["v"], a["g"], a.get("aug"), a.get("norm_w"),
                                 a.get("eps", 0.0))


def test_zero_output_makes_the_gate_cancel():
    """o = 0: u = gate * v with gate > 0, which the norm removes, so z does not
    depend on the augmentation weights (a gate applied to o would give 0/0)."""
    c = case(1)
    z1 = epi(c, o=np.zeros_like(c["o"]))
    z2 = epi(c, o=np.zeros_like(c["o"]), aug=-3.0 * c["aug"])
    z3 = epi(c, o=np.zeros_like(c["o"]), aug=None)
    assert np.allclose(z1, z2, rtol=1e-12, atol=1e-14)
    assert np.allclose(z1, z3, rtol=1e-12, atol=1e-14)


def test_norm_is_scale_invariant():
    c = case(2)
    z = epi(c)
    for s in (1e-3, 0.5, 7.0, 1e4):
        assert np.allclose(epi(c, o=s * c["o"], v=s * c["v"]), z, rtol=1e-11, atol=1e-14)


def test_unit_rms_before_the_gate():
    """w = 1, eps = 0 and g = 40 (SiLU(40) = 40 to 1e-17): mean(z^2) = 1600 per (token, head)."""
    c = case(3)
    z = epi(c, norm_w=None, g=np.full_like(c["g"], 40.0))
    assert np.allclose((z ** 2).mean(axis=-1), 1600.0, rtol=1e-12)


def test_half_strength_skip_at_zero_augmentation():
    """a = 0 gives the gate 1/2: with o = -v/2 the head's u is exactly zero."""
    c = case(4)
    z = epi(c, aug=np.zeros_like(c["aug"]), o=-0.5 * c["v"], eps=1e-6)
    assert np.array_equal(z, np.zeros_like(z))
    z_other = epi(c, aug=np.zeros_like(c["aug"]), o=+0.5 * c["v"], eps=1e-6)
    assert np.abs(z_other).max() > 0.1


def test_gate_limits():
    """q.(a*k) -> +inf adds the whole value, -inf none of it."""
    c = case(5, dk=1)
    qk = c["q"][..., 0] * c["k"][..., 0]
    big = 60.0 / qk                                   # per (token, head): q a k = +60
    for sign in (1.0, -1.0):
        zs = []
        for t in range(c["o"].shape[0]):
            for h in range(c["o"].shape[1]):
                one = {key: c[key][t:t + 1, h:h + 1] for key in ("o", "q", "k", "v", "g")}
                one["aug"] = np.array([[sign * big[t, h]]])
                one["norm_w"] = c["norm_w"][h:h + 1]
                zs.append(epi(one)[0, 0])
        z = np.array(zs).reshape(c["o"].shape)
        ref = epi(c, o=c["o"] + (c["v"] if sign > 0 else 0.0), v=np.zeros_like(c["v"]))
        assert np.allclose(z, ref, rtol=1e-12, atol=1e-14)


def test_output_gate_is_silu():
    """SiLU(g) - SiLU(-g) = g: z(g) - z(-g) = y * g, with y read from g = 40."""
    c = case(6)
    y = epi(c, g=np.full_like(c["g"], 40.0)) / 40.0
    d = epi(c) - epi(c, g=-c["g"])
    assert np.allclose(d, y * c["g"], rtol=1e-11, atol=1e-13)
    assert np.array_equal(epi(c, g=np.zeros_like(c["g"])), np.zeros_like(c["o"]))


def test_rows_are_independent_and_weights_per_head():
    """z of (token, head) depends only on that row's inputs and that head's
    weights; q and k enter the gate symmetrically."""
    c = case(7)
    z = epi(c, eps=1e-6)
    c2 = {key: val.copy() for key, val in c.items()}
    c2["o"][2, 1] += 5.0
    c2["v"][3, 0] *= -2.0
    c2["aug"][2] *= 3.0
    z2 = epi(c2, eps=1e-6)
    changed = np.zeros(z.shape[:2], dtype=bool)
    changed[2, 1] = changed[3, 0] = True
    changed[:, 2] = True
    assert np.array_equal(z[~changed], z2[~changed])
    assert not np.allclose(z[2, 1], z2[2, 1])
    for t in range(z.shape[0]):       # head 2's own augmentation weights reach every one of its rows
        assert not np.allclose(z[t, 2], z2[t, 2])
    assert np.allclose(epi(c, q=c["k"], k=c["q"]), epi(c), rtol=1e-13, atol=1e-15)


def test_norm_weight_is_per_channel_and_linear():
    c = case(8)
    z = epi(c)
    w2 = c["norm_w"].copy()
    w2[:, 3] *= 2.5
    z2 = epi(c, norm_w=w2)
    assert np.allclose(z2[..., 3], 2.5 * z[..., 3], rtol=1e-13)
    assert np.array_equal(np.delete(z2, 3, axis=-1), np.delete(z, 3, axis=-1))
