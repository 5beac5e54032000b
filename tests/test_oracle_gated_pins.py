"""Pins of the oracle's per-token (data-dependent) decay, O9, O10 and its
backward O11.

The gated recurrence S_t = exp(g_t) S_{t-1} + k_t v_t^T, o_t = scale S_t^T q_t
is checked against facts outside its own code, chosen so that a plausible
slip (the decay applied after adding k v^T, the gate of token t used at
t+1, a cumulative decay that includes the token's own gate, a missing h0
decay, a transposed state) fails at least one of them:

  - a hand-worked fixture with a cleared state (tests/golden/gated_hand_worked.json);
  - a constant gate g_t = log lambda_h reproduces the fixed-decay oracle,
    itself pinned in test_oracle_pins.py;
  - the unrolled sums against the recurrence, -inf gates included;
  - the chunk equations at several chunk lengths against the recurrence;
  - g = 0: causal linear attention as a masked matrix product;
  - a -inf gate clears the state: the outputs from there on are those of a
    fresh call over the rest of the sequence;
  - split-call invariance;
  - the final state in closed form from cumulative sums of g;
  - one decode step equals the forward at T = 1, and a prefill followed by
    decode steps equals one longer prefill;
  - linearity in (v, h0) jointly;
  - O11: central differences of L = sum <do, o> + <dhT, hT> for every
    gradient including the gate's (a sign slip in dg, the gate of t used at
    t+1, a dh0 without its decay fail these); a constant gate reproduces the
    fixed-decay backward, and its dg summed over tokens the gradient of
    log lambda; a -inf gate has dg = 0 and cuts the gradient paths across it.
"""
import json
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


def case(seed, B=2, T=29, H=3, dk=4, dv=5, h0=True, kind="wide"):
    rng = np.random.default_rng(4000 + seed)
    q = rng.standard_normal((B, T, H, dk))
    k = rng.standard_normal((B, T, H, dk))
    v = rng.standard_normal((B, T, H, dv))
    H0 = rng.standard_normal((B, H, dk, dv)) * 0.5 if h0 else None
    g = gen.log_gates(rng, (B, T, H), kind).astype(np.float64)
    return q, k, v, g, H0


def test_hand_worked_forward():
    f = json.load(open(os.path.join(GOLDEN, "gated_hand_worked.json")))["forward"]
    q = np.array(f["q"], float)[None, :, None, :]
    k = np.array(f["k"], float)[None, :, None, :]
    v = np.array(f["v"], float)[None, :, None, :]
    with np.errstate(divide="ignore"):
        g = np.log(np.array(f["alpha"], float))[None, :, None]
    h0 = np.array(f["h0"], float)[None, None]
    for form in ("recurrent", "quadratic", "chunked"):
        o, hT = oracle.fwd_gated(q, k, v, g, h0, f["scale"], form=form, chunk=2)
        assert np.array_equal(o[0, :, 0], np.array(f["o"], float)), form
        assert np.array_equal(hT[0, 0], np.array(f["hT"], float)), form


def test_hand_worked_decode():
    f = json.load(open(os.path.join(GOLDEN, "gated_hand_worked.json")))["decode"]
    q = np.array(f["q"], float)[None, None]
    k = np.array(f["k"], float)[None, None]
    v = np.array(f["v"], float)[None, None]
    S = np.array(f["S"], float)[None, None]
    g = np.log(np.array([[f["alpha"]]], float))
    o, S_new = oracle.decode_gated(q, k, v, g, S, f["scale"])
    assert np.array_equal(o[0, 0], np.array(f["o"], float))
    assert np.array_equal(S_new[0, 0], np.array(f["S_new"], float))


@pytest.mark.parametrize("form", ["recurrent", "quadratic"])
def test_constant_gate_is_the_fixed_decay(form):
    q, k, v, _, h0 = case(1)
    lam = np.array([0.3, 0.9, 0.999])
    ll = np.log(lam)
    g = np.broadcast_to(ll, q.shape[:3]).copy()
    o_ref, hT_ref = oracle.fwd_recurrent(q, k, v, ll, h0, 0.37)
    o, hT = oracle.fwd_gated(q, k, v, g, h0, 0.37, form=form)
    assert rel(o, o_ref) < 1e-12 and rel(hT, hT_ref) < 1e-12


@pytest.mark.parametrize("kind", ["wide", "gla"])
def test_unrolled_sums_match_recurrence(kind):
    q, k, v, g, h0 = case(2, kind=kind)
    g[0, 5, 1] = -np.inf
    g[1, 0, 2] = -np.inf
    o1, h1 = oracle.fwd_gated(q, k, v, g, h0, 0.5)
    o2, h2 = oracle.fwd_gated(q, k, v, g, h0, 0.5, form="quadratic")
    assert rel(o2, o1) < 1e-12 and rel(h2, h1) < 1e-12


@pytest.mark.parametrize("C", [1, 3, 16, 64])
def test_chunk_equations_match_recurrence(C):
    q, k, v, g, h0 = case(3, T=70, kind="gla")
    g[0, 40, 0] = -np.inf
    o1, h1 = oracle.fwd_gated(q, k, v, g, h0, 0.3)
    o2, h2 = oracle.fwd_gated(q, k, v, g, h0, 0.3, form="chunked", chunk=C)
    assert rel(o2, o1) < 1e-12 and rel(h2, h1) < 1e-12


def test_zero_gate_is_causal_linear_attention():
    q, k, v, _, h0 = case(4)
    g = np.zeros(q.shape[:3])
    o, hT = oracle.fwd_gated(q, k, v, g, h0, 0.7)
    T = q.shape[1]
    mask = np.tril(np.ones((T, T)))
    ref = 0.7 * (np.einsum("btha,bsha,ts,bshc->bthc", q, k, mask, v) + np.einsum("btha,bhac->bthc", q, h0))
    assert rel(o, ref) < 1e-12
    assert rel(hT, h0 + np.einsum("btha,bthc->bhac", k, v)) < 1e-12


def test_minus_inf_gate_clears_the_state():
    q, k, v, g, h0 = case(5, T=24)
    r = 11
    g[:, r, :] = -np.inf
    o, hT = oracle.fwd_gated(q, k, v, g, h0, 0.4)
    g_rest = g[:, r:].copy()
    g_rest[:, 0, :] = 0.0            # no state enters, so its decay does not matter
    o2, hT2 = oracle.fwd_gated(q[:, r:], k[:, r:], v[:, r:], g_rest, None, 0.4)
    assert rel(o[:, r:], o2) < 1e-12 and rel(hT, hT2) < 1e-12


def test_split_call_invariance():
    q, k, v, g, h0 = case(6, T=40, kind="gla")
    t1 = 17
    o, hT = oracle.fwd_gated(q, k, v, g, h0, 0.25)
    oa, ha = oracle.fwd_gated(q[:, :t1], k[:, :t1], v[:, :t1], g[:, :t1], h0, 0.25)
    ob, hb = oracle.fwd_gated(q[:, t1:], k[:, t1:], v[:, t1:], g[:, t1:], ha, 0.25)
    assert rel(np.concatenate([oa, ob], axis=1), o) < 1e-12 and rel(hb, hT) < 1e-12


def test_final_state_closed_form():
    q, k, v, g, h0 = case(7, T=33, kind="gla")
    _, hT = oracle.fwd_gated(q, k, v, g, h0, 1.0)
    G = np.cumsum(g, axis=1)                       # G[t] = g_0 + ... + g_t
    GT = G[:, -1]                                  # [B, H]
    w = np.exp(GT[:, None, :] - G)                 # decay of tokens u+1..T-1
    ref = np.exp(GT)[:, :, None, None] * h0 + np.einsum("bth,btha,bthc->bhac", w, k, v)
    assert rel(hT, ref) < 1e-12


def test_decode_step_is_forward_at_T1():
    q, k, v, g, h0 = case(8, T=1)
    o, hT = oracle.fwd_gated(q, k, v, g, h0, 0.6)
    B, _, H, dk = q.shape
    od, S = oracle.decode_gated(q[:, 0], k[:, 0], v[:, 0], g[:, 0], h0, 0.6)
    assert rel(od, o[:, 0]) < 1e-14 and rel(S, hT) < 1e-14


def test_linear_in_v_and_h0():
    """For fixed q, k and g the outputs and the final state are linear in
    (v, h0) jointly: a term that does not scale with them (a bias, a gate
    applied to k v^T twice, a squared state) breaks this."""
    q, k, v, g, h0 = case(9, T=37, kind="gla")
    rng = np.random.default_rng(4109)
    v2 = rng.standard_normal(v.shape)
    h2 = rng.standard_normal(h0.shape)
    a, b = 0.7, -1.3
    o1, s1 = oracle.fwd_gated(q, k, v, g, h0, 0.5)
    o2, s2 = oracle.fwd_gated(q, k, v2, g, h2, 0.5)
    o3, s3 = oracle.fwd_gated(q, k, a * v + b * v2, g, a * h0 + b * h2, 0.5)
    assert rel(o3, a * o1 + b * o2) < 1e-12 and rel(s3, a * s1 + b * s2) < 1e-12


def test_prefill_then_decode_equals_longer_prefill():
    """A prefill over T tokens followed by decode steps over the next ones
    gives the outputs and state of one prefill over all of them, clearing
    gates in both parts included."""
    q, k, v, g, h0 = case(10, T=24, kind="gla")
    g = g.copy()
    g[0, 5, 1] = -np.inf
    g[1, 21, 2] = -np.inf                            # inside the decoded tail
    t1 = 18
    o, hT = oracle.fwd_gated(q, k, v, g, h0, 0.3)
    op, S = oracle.fwd_gated(q[:, :t1], k[:, :t1], v[:, :t1], g[:, :t1], h0, 0.3)
    outs = [op]
    for t in range(t1, q.shape[1]):
        ot, S = oracle.decode_gated(q[:, t], k[:, t], v[:, t], g[:, t], S, 0.3)
        outs.append(ot[:, None])
    assert rel(np.concatenate(outs, axis=1), o) < 1e-12 and rel(S, hT) < 1e-12


# ------------------------------------------------------------- O11: backward
def gated_loss(q, k, v, g, h0, scale, do, dhT):
    o, hT = oracle.fwd_gated(q, k, v, g, h0, scale)
    return float(np.sum(do * o) + np.sum(dhT * hT))


@pytest.mark.parametrize("T", [7, 70])
def test_gated_backward_finite_differences(T):
    """Every gradient, the gate's included, against central differences of
    L = sum <do, o> + <dhT, hT> (T = 70 crosses the oracle's checkpoints)."""
    q, k, v, g, h0 = case(20 + T, B=1, T=T, H=2, dk=3, dv=4, kind="wide")
    rng = np.random.default_rng(21 + T)
    do = rng.standard_normal(v.shape)
    dhT = rng.standard_normal(h0.shape) * 0.5
    grads = oracle.bwd_gated(q, k, v, g, h0, 0.6, do, dhT)
    args = dict(q=q, k=k, v=v, g=g, h0=h0)
    eps = 1e-6
    for name, grad in zip(("q", "k", "v", "h0", "g"), grads):
        x = args[name]
        idx = [tuple(rng.integers(0, n) for n in x.shape) for _ in range(6)]
        for ix in idx:
            xp, xm = x.copy(), x.copy()
            xp[ix] += eps
            xm[ix] -= eps
            ap, am = dict(args, **{name: xp}), dict(args, **{name: xm})
            fd = (gated_loss(ap["q"], ap["k"], ap["v"], ap["g"], ap["h0"], 0.6, do, dhT) -
                  gated_loss(am["q"], am["k"], am["v"], am["g"], am["h0"], 0.6, do, dhT)) / (2 * eps)
            assert abs(fd - grad[ix]) <= 1e-6 * max(1.0, abs(fd)), (name, ix, fd, grad[ix])


def test_gated_backward_constant_gate_is_the_fixed_backward():
    """A constant gate reproduces the fixed-decay gradients; the gate's
    gradient summed over tokens is the gradient of log lambda (checked by
    central differences of the fixed-decay loss)."""
    q, k, v, _, h0 = case(22, B=1, T=40, H=3, dk=4, dv=5)
    rng = np.random.default_rng(23)
    do = rng.standard_normal(v.shape)
    dhT = rng.standard_normal(h0.shape) * 0.3
    ll = np.log(np.array([0.4, 0.8, 0.97]))
    g = np.broadcast_to(ll, q.shape[:3]).copy()
    dq, dk, dv, dh0, dg = oracle.bwd_gated(q, k, v, g, h0, 0.5, do, dhT)
    rq, rk, rv, rh0 = oracle.bwd(q, k, v, ll, h0, 0.5, do, dhT)
    for a, b in ((dq, rq), (dk, rk), (dv, rv), (dh0, rh0)):
        assert rel(a, b) < 1e-12
    eps = 1e-6

    def loss(ll_):
        o, hT = oracle.fwd_recurrent(q, k, v, ll_, h0, 0.5)
        return float(np.sum(do * o) + np.sum(dhT * hT))
    for h in range(3):
        e = np.zeros(3)
        e[h] = eps
        fd = (loss(ll + e) - loss(ll - e)) / (2 * eps)
        assert abs(dg[0, :, h].sum() - fd) <= 1e-6 * max(1.0, abs(fd))


def test_gated_backward_clearing_gate():
    """A -inf gate at r: its own gradient is 0, and nothing after r reaches
    the tokens before it except through k_r v_r^T (so dq of tokens < r and
    dh0 equal those of the loss restricted to outputs < r)."""
    q, k, v, g, h0 = case(24, B=1, T=30, H=2, dk=3, dv=4, kind="gla")
    r = 13
    g[:, r, :] = -np.inf
    rng = np.random.default_rng(25)
    do = rng.standard_normal(v.shape)
    dq, dk, dv, dh0, dg = oracle.bwd_gated(q, k, v, g, h0, 0.5, do, None)
    assert np.all(dg[:, r, :] == 0.0)
    dq2, dk2, dv2, dh02, dg2 = oracle.bwd_gated(q[:, :r], k[:, :r], v[:, :r], g[:, :r], h0, 0.5, do[:, :r], None)
    assert rel(dq[:, :r], dq2) < 1e-12 and rel(dh0, dh02) < 1e-12
    assert rel(dk[:, :r], dk2) < 1e-12 and rel(dv[:, :r], dv2) < 1e-12 and rel(dg[:, :r], dg2) < 1e-12
