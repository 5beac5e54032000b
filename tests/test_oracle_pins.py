"""Pins of the double-precision oracle to facts outside itself.

Each test checks the oracle against something the pages or the mathematics
fix, chosen so that a plausible slip in the oracle (a dropped decay term, a
wrong exponent, a transposed state, the scale on the state instead of the
readout, the readout before the update) fails at least one of them:

  - hand-worked fixtures (tests/golden/hand_worked.json);
  - the brute-force unrolled sum against the recurrence;
  - lambda = 1: causal linear attention, a masked matrix product;
  - lambda = 0: o_t = scale (q_t . k_t) v_t;
  - the closed-form final state as an einsum of decayed outer products;
  - chunk-size invariance of the chunked form, ragged tails included;
  - split-call invariance (hT of the first half is h0 of the second);
  - linearity in v and in h0; T = 1 forward equals one decode step;
  - central finite differences of L = sum<do, o> + <dhT, hT> for the backward,
    and the brute-force transposed sums for every gradient;
  - the printed decay-schedule endpoints for the generator's page schedule.
"""
import json
import math
import os

import numpy as np
import pytest

import gla_gen as gen
import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def rel(a, b):
    a, b = np.asarray(a, np.float64), np.asarray(b, np.float64)
    den = max(np.max(np.abs(b)), 1e-300)
    return float(np.max(np.abs(a - b)) / den)


def rand_case(seed, B=2, T=37, H=3, dk=5, dv=7, h0=True, lam=None, grad=False):
    rng = np.random.default_rng(1000 + seed)
    q = rng.standard_normal((B, T, H, dk))
    k = rng.standard_normal((B, T, H, dk))
    v = rng.standard_normal((B, T, H, dv))
    H0 = rng.standard_normal((B, H, dk, dv)) * 0.5 if h0 else None
    if lam is None:
        lam = rng.uniform(0.3, 0.999, size=H)
    lam = np.broadcast_to(np.asarray(lam, np.float64), (H,)).copy()
    with np.errstate(divide="ignore"):
        ll = np.log(lam)
    out = dict(q=q, k=k, v=v, h0=H0, ll=ll, lam=lam, scale=0.37)
    if grad:
        out["do"] = rng.standard_normal((B, T, H, dv))
        out["dhT"] = rng.standard_normal((B, H, dk, dv)) * 0.3
    return out


# ------------------------------------------------------------------ fixtures
def test_hand_worked_forward():
    g = json.load(open(os.path.join(GOLDEN, "hand_worked.json")))["forward"]
    q = np.array(g["q"], float)[None, :, None, :]
    k = np.array(g["k"], float)[None, :, None, :]
    v = np.array(g["v"], float)[None, :, None, :]
    ll = np.array([math.log(g["lambda"])])
    for fn in (oracle.fwd_recurrent, oracle.fwd_quadratic):
        o, hT = fn(q, k, v, ll, None, g["scale"])
        assert np.array_equal(o[0, :, 0, :], np.array(g["o"], float))
        assert np.array_equal(hT[0, 0], np.array(g["hT"], float))
    o, hT = oracle.fwd_chunked(q, k, v, ll, None, g["scale"], chunk=1)
    assert np.array_equal(o[0, :, 0, :], np.array(g["o"], float))
    assert np.array_equal(hT[0, 0], np.array(g["hT"], float))


def test_hand_worked_decode():
    g = json.load(open(os.path.join(GOLDEN, "hand_worked.json")))["decode"]
    S = np.array(g["S"], float)[None, None]
    q = np.array(g["q"], float)[None, None]
    k = np.array(g["k"], float)[None, None]
    v = np.array(g["v"], float)[None, None]
    o, S_new = oracle.decode(q, k, v, np.array([math.log(g["lambda"])]), S, g["scale"])
    assert np.array_equal(S_new[0, 0], np.array(g["S_new"], float))
    assert np.array_equal(o[0, 0], np.array(g["o"], float))


def test_hand_worked_backward():
    g = json.load(open(os.path.join(GOLDEN, "hand_worked.json")))["backward"]
    sh = lambda x: np.array(x, float).reshape(1, 2, 1, 1)
    q, k, v, do = sh(g["q"]), sh(g["k"]), sh(g["v"]), sh(g["do"])
    h0 = np.full((1, 1, 1, 1), float(g["h0"]))
    dhT = np.full((1, 1, 1, 1), float(g["dhT"]))
    ll = np.array([math.log(g["lambda"])])
    o, hT = oracle.fwd_recurrent(q, k, v, ll, h0, g["scale"])
    assert np.allclose(o.ravel(), g["o"], rtol=0, atol=1e-15) and abs(hT.item() - g["hT"]) < 1e-15
    for fn in (oracle.bwd, lambda *a: oracle.bwd_chunked(*a, chunk=1)):
        dq, dk, dv, dh0 = fn(q, k, v, ll, h0, g["scale"], do, dhT)
        assert np.allclose(dq.ravel(), g["dq"], rtol=0, atol=1e-15)
        assert np.allclose(dk.ravel(), g["dk"], rtol=0, atol=1e-15)
        assert np.allclose(dv.ravel(), g["dv"], rtol=0, atol=1e-15)
        assert abs(dh0.item() - g["dh0"]) < 1e-15


def test_page_decay_schedule_endpoints():
    g = json.load(open(os.path.join(GOLDEN, "decay_schedule_endpoints.json")))
    lam = gen.decay_page_schedule(g["H"], g["T_min"], g["T_max"])
    assert lam[0] == g["lambda_0"]
    assert round(float(lam[-1]), g["lambda_15_printed_digits"]) == g["lambda_15_printed"]
    # half-lives: lambda^T_h = 1/2 at the printed ends
    assert abs(lam[0] ** g["half_life_0_tokens"] - 0.5) < 1e-15
    assert abs(lam[-1] ** g["half_life_15_tokens"] - 0.5) < 1e-12
    assert np.all(np.diff(lam) > 0)


# ---------------------------------------------------- forward special cases
@pytest.mark.parametrize("seed", [0, 1, 2])
def test_bruteforce_equals_recurrence(seed):
    c = rand_case(seed, T=41 + seed)
    o1, h1 = oracle.fwd_quadratic(c["q"], c["k"], c["v"], c["ll"], c["h0"], c["scale"])
    o2, h2 = oracle.fwd_recurrent(c["q"], c["k"], c["v"], c["ll"], c["h0"], c["scale"])
    assert rel(o2, o1) < 1e-12 and rel(h2, h1) < 1e-12


def test_lambda_one_is_causal_linear_attention():
    c = rand_case(3, T=50, lam=1.0)
    o, hT = oracle.fwd_recurrent(c["q"], c["k"], c["v"], c["ll"], c["h0"], c["scale"])
    T = c["q"].shape[1]
    mask = np.tril(np.ones((T, T)))
    for b in range(c["q"].shape[0]):
        for h in range(c["q"].shape[2]):
            Q, K, V = c["q"][b, :, h], c["k"][b, :, h], c["v"][b, :, h]
            ref = c["scale"] * ((Q @ K.T) * mask) @ V + c["scale"] * Q @ c["h0"][b, h]
            assert rel(o[b, :, h], ref) < 1e-12
            assert rel(hT[b, h], c["h0"][b, h] + K.T @ V) < 1e-12


def test_lambda_zero_is_diagonal():
    c = rand_case(4, T=23, lam=0.0)
    assert np.all(np.isneginf(c["ll"]))
    o, hT = oracle.fwd_recurrent(c["q"], c["k"], c["v"], c["ll"], c["h0"], c["scale"])
    qk = np.sum(c["q"] * c["k"], axis=-1, keepdims=True)
    assert rel(o, c["scale"] * qk * c["v"]) < 1e-14
    ref_h = np.einsum("bhi,bhj->bhij", c["k"][:, -1], c["v"][:, -1])
    assert rel(hT, ref_h) < 1e-14
    for C in (1, 4, 16):
        oc, hc = oracle.fwd_chunked(c["q"], c["k"], c["v"], c["ll"], c["h0"], c["scale"], chunk=C)
        assert rel(oc, o) < 1e-14 and rel(hc, hT) < 1e-14


def test_closed_form_final_state():
    c = rand_case(5, T=33)
    _, hT = oracle.fwd_recurrent(c["q"], c["k"], c["v"], c["ll"], c["h0"], c["scale"], want_o=False)
    T = c["q"].shape[1]
    w = c["lam"][None, :] ** (T - 1 - np.arange(T))[:, None]          # [T, H]
    ref = np.einsum("th,bthi,bthj->bhij", w, c["k"], c["v"]) + \
        (c["lam"] ** T)[None, :, None, None] * c["h0"]
    assert rel(hT, ref) < 1e-12


@pytest.mark.parametrize("C", [1, 3, 16, 64, 128, 256])
def test_chunk_size_invariance(C):
    c = rand_case(6, T=200, dk=6, dv=9)
    o, hT = oracle.fwd_recurrent(c["q"], c["k"], c["v"], c["ll"], c["h0"], c["scale"])
    oc, hc = oracle.fwd_chunked(c["q"], c["k"], c["v"], c["ll"], c["h0"], c["scale"], chunk=C)
    assert rel(oc, o) < 1e-12 and rel(hc, hT) < 1e-12


def test_split_call_invariance():
    c = rand_case(7, T=90)
    o, hT = oracle.fwd_recurrent(c["q"], c["k"], c["v"], c["ll"], c["h0"], c["scale"])
    t1 = 37
    oa, ha = oracle.fwd_recurrent(c["q"][:, :t1], c["k"][:, :t1], c["v"][:, :t1], c["ll"], c["h0"], c["scale"])
    ob, hb = oracle.fwd_recurrent(c["q"][:, t1:], c["k"][:, t1:], c["v"][:, t1:], c["ll"], ha, c["scale"])
    assert rel(np.concatenate([oa, ob], axis=1), o) < 1e-13 and rel(hb, hT) < 1e-13


def test_prefill_then_decode_equals_longer_prefill():
    c = rand_case(8, B=2, T=30, H=2)
    o, hT = oracle.fwd_recurrent(c["q"], c["k"], c["v"], c["ll"], c["h0"], c["scale"])
    t1 = 25
    _, S = oracle.fwd_recurrent(c["q"][:, :t1], c["k"][:, :t1], c["v"][:, :t1], c["ll"], c["h0"], c["scale"])
    for t in range(t1, 30):
        od, S = oracle.decode(c["q"][:, t], c["k"][:, t], c["v"][:, t], c["ll"], S, c["scale"])
        assert rel(od, o[:, t]) < 1e-13
    assert rel(S, hT) < 1e-13


def test_T1_forward_equals_decode():
    c = rand_case(9, B=3, T=1, H=4)
    o, hT = oracle.fwd_recurrent(c["q"], c["k"], c["v"], c["ll"], c["h0"], c["scale"])
    od, S = oracle.decode(c["q"][:, 0], c["k"][:, 0], c["v"][:, 0], c["ll"], c["h0"], c["scale"])
    assert rel(od, o[:, 0]) < 1e-15 and rel(S, hT) < 1e-15


def test_linearity_in_v_and_h0():
    c = rand_case(10, T=40)
    rng = np.random.default_rng(77)
    v2 = rng.standard_normal(c["v"].shape)
    f = lambda v, h0: oracle.fwd_recurrent(c["q"], c["k"], v, c["ll"], h0, c["scale"])
    oa, ha = f(c["v"], None)
    ob, hb = f(v2, None)
    oc, hc = f(2.0 * c["v"] - 3.0 * v2, None)
    assert rel(oc, 2 * oa - 3 * ob) < 1e-12 and rel(hc, 2 * ha - 3 * hb) < 1e-12
    z = np.zeros_like(c["v"])
    oh, hh = f(z, c["h0"])
    of, hf = f(c["v"], c["h0"])
    assert rel(of, oa + oh) < 1e-12 and rel(hf, ha + hh) < 1e-12
    # the h0-only response decays as lambda^(t+1) along the sequence
    T = c["q"].shape[1]
    ref = np.einsum("bthi,bhij->bthj", c["q"], c["h0"]) * c["scale"] * \
        (c["lam"][None, :] ** (np.arange(T)[:, None] + 1.0))[None, :, :, None]
    assert rel(oh, ref) < 1e-12


def test_zero_length_and_no_state():
    c = rand_case(11, T=0)
    o, hT = oracle.fwd_recurrent(c["q"], c["k"], c["v"], c["ll"], c["h0"], c["scale"])
    assert o.shape[1] == 0 and np.array_equal(hT, c["h0"])


# --------------------------------------------------------------- backward
def _loss(c, q, k, v, h0):
    o, hT = oracle.fwd_recurrent(q, k, v, c["ll"], h0, c["scale"])
    return float(np.sum(o * c["do"]) + np.sum(hT * c["dhT"]))


@pytest.mark.parametrize("seed", [0, 1])
def test_backward_matches_central_differences(seed):
    c = rand_case(20 + seed, B=1, T=9, H=2, dk=3, dv=4, grad=True)
    dq, dk, dv, dh0 = oracle.bwd(c["q"], c["k"], c["v"], c["ll"], c["h0"], c["scale"], c["do"], c["dhT"])
    eps = 1e-6
    for name, grad in (("q", dq), ("k", dk), ("v", dv), ("h0", dh0)):
        x = c[name]
        num = np.zeros_like(x)
        it = np.nditer(x, flags=["multi_index"])
        for _ in it:
            idx = it.multi_index
            args = {n: c[n].copy() for n in ("q", "k", "v", "h0")}
            args[name][idx] += eps
            lp = _loss(c, args["q"], args["k"], args["v"], args["h0"])
            args[name][idx] -= 2 * eps
            lm = _loss(c, args["q"], args["k"], args["v"], args["h0"])
            num[idx] = (lp - lm) / (2 * eps)
        assert rel(grad, num) < 1e-7, name


def test_backward_matches_bruteforce_sums():
    c = rand_case(30, B=2, T=19, H=2, dk=4, dv=5, grad=True)
    dq, dk, dv, dh0 = oracle.bwd(c["q"], c["k"], c["v"], c["ll"], c["h0"], c["scale"], c["do"], c["dhT"])
    s, T = c["scale"], c["q"].shape[1]
    for b in range(2):
        for h in range(2):
            lam = c["lam"][h]
            Q, K, V, dO = c["q"][b, :, h], c["k"][b, :, h], c["v"][b, :, h], c["do"][b, :, h]
            H0, G = c["h0"][b, h], c["dhT"][b, h]
            D = np.array([[lam ** (t - u) if u <= t else 0.0 for u in range(T)] for t in range(T)])
            Aqk = (Q @ K.T) * D          # [t, u]
            Adv = (dO @ V.T) * D         # [t, u]
            wq = lam ** (np.arange(T) + 1.0)
            wT = lam ** (T - 1.0 - np.arange(T))
            ref_dq = s * Adv @ K + s * wq[:, None] * (dO @ H0.T)
            ref_dk = s * Adv.T @ Q + wT[:, None] * (V @ G.T)
            ref_dv = s * Aqk.T @ dO + wT[:, None] * (K @ G)
            ref_dh0 = s * (Q * wq[:, None]).T @ dO + lam ** T * G
            assert rel(dq[b, :, h], ref_dq) < 1e-12
            assert rel(dk[b, :, h], ref_dk) < 1e-12
            assert rel(dv[b, :, h], ref_dv) < 1e-12
            assert rel(dh0[b, h], ref_dh0) < 1e-12


@pytest.mark.parametrize("C", [1, 5, 16, 64])
def test_chunked_backward_equals_backward(C):
    c = rand_case(31, B=2, T=70, H=2, dk=4, dv=6, grad=True)
    ref = oracle.bwd(c["q"], c["k"], c["v"], c["ll"], c["h0"], c["scale"], c["do"], c["dhT"])
    got = oracle.bwd_chunked(c["q"], c["k"], c["v"], c["ll"], c["h0"], c["scale"], c["do"], c["dhT"], chunk=C)
    for g, r in zip(got, ref):
        assert rel(g, r) < 1e-12


def test_backward_lambda_zero_and_no_optional_inputs():
    c = rand_case(32, B=1, T=12, H=2, dk=3, dv=4, lam=0.0, grad=True)
    dq, dk, dv, dh0 = oracle.bwd(c["q"], c["k"], c["v"], c["ll"], None, c["scale"], c["do"], None)
    s = c["scale"]
    dov = np.sum(c["do"] * c["v"], -1, keepdims=True)
    qk = np.sum(c["q"] * c["k"], -1, keepdims=True)
    assert rel(dq, s * dov * c["k"]) < 1e-14
    assert rel(dk, s * dov * c["q"]) < 1e-14
    assert rel(dv, s * qk * c["do"]) < 1e-14
    assert np.all(dh0 == 0)


# --------------------------------------------------------------- generator
def test_generator_is_seeded_and_rounded():
    a = gen.make_case(1, 20, 2, 8, 16, seed=5, normalise_k=True)
    b = gen.make_case(1, 20, 2, 8, 16, seed=5, normalise_k=True)
    assert np.array_equal(a.q, b.q) and np.array_equal(a.k, b.k)
    assert np.array_equal(gen.bf16_round(a.q), a.q)
    n = np.sqrt(np.sum(a.k.astype(np.float64) ** 2, -1))
    assert np.all(np.abs(n - 1) < 1e-2)
    lam = gen.decay_layer_schedule(16)
    assert lam[0] == 0.96875 and abs(lam[-1] - (1 - 2 ** -12)) < 1e-15


def test_bf16_rounding_ties_to_even():
    x = np.array([1.0, 1.0 + 2 ** -8, 1.0 + 3 * 2 ** -8, -2.5, 3.0e38], np.float32)
    r = gen.bf16_round(x)
    assert r[0] == 1.0 and r[1] == 1.0 and r[2] == 1.0 + 2 ** -6 and r[3] == -2.5
    assert np.isinf(gen.bf16_round(np.array([3.4e38], np.float32)))[0]
