"""GPU parity of the variable-length forward (gla_chunk_fwd_varlen): sequences
of different lengths packed token-major, each entering from and leaving its
state in a pool slot, checked per sequence against the double-precision
oracle; the hand-off to the decode step on the same pool; and equality with
the batched forward when every sequence has the same length."""
import numpy as np
import pytest

import gla_gen as gen
import oracle
from gpu_util import TOL, f32_dev, relerr, to_dev, to_host

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def gla():
    import linear_attention_chunk_gb300 as m
    from linear_attention_chunk_gb300.build import build
    build()
    return m


def dev_case(c):
    import torch
    return dict(q=to_dev(c.q, "bf16"), k=to_dev(c.k, "bf16"), v=to_dev(c.v, "bf16"), ll=f32_dev(c.log_lambda),
                cu=torch.from_numpy(c.cu_seqlens).cuda(), slots=torch.from_numpy(c.slots).cuda(),
                pool=f32_dev(c.pool))


def oracle_seq(c, n, pool_before):
    """Oracle output and final state of sequence n of the case."""
    a, b = int(c.cu_seqlens[n]), int(c.cu_seqlens[n + 1])
    h0 = pool_before[c.slots[n]][None].astype(np.float32)   # the fp32 values the GPU holds
    o, hT = oracle.fwd_recurrent(c.q[None, a:b], c.k[None, a:b], c.v[None, a:b], c.log_lambda, h0, c.scale)
    return o[0], hT[0]


@pytest.mark.parametrize("C", [128, 64])
@pytest.mark.parametrize("H", [4, 8])
def test_varlen_matches_oracle_per_sequence(gla, C, H):
    """40 (sequence, head) chains run two CTAs each (half the state each), 80
    chains one CTA each (the whole state)."""
    lengths = [0, 1, 63, 64, 65, 128, 129, 200, 333, 1000]
    c = gen.make_varlen_case(lengths, H, seed=500 + C + H, n_slots=14)
    d = dev_case(c)
    o = gla.gla_chunk_fwd_varlen(d["q"], d["k"], d["v"], d["ll"], d["cu"], d["pool"], d["slots"], c.scale, C)
    gla.gla_check()
    oh, pool = to_host(o), to_host(d["pool"])
    for n in range(len(lengths)):
        a, b = int(c.cu_seqlens[n]), int(c.cu_seqlens[n + 1])
        if b == a:
            continue
        ro, rh = oracle_seq(c, n, c.pool)
        assert relerr(oh[a:b], ro) <= TOL["bf16"], f"o of sequence {n} (length {b - a})"
        assert relerr(pool[c.slots[n]], rh) <= TOL["bf16"], f"state of sequence {n}"
    # a length-0 sequence and the slots no sequence uses keep their bytes
    untouched = [s for s in range(14) if s not in set(c.slots[1:].tolist())]
    assert c.slots[0] in untouched
    for s in untouched:
        assert np.array_equal(pool[s], c.pool[s].astype(np.float32).astype(np.float64)), f"slot {s} changed"


@pytest.mark.parametrize("H", [8, 32])
def test_varlen_equals_batched_forward(gla, H):
    """Equal lengths, slot n = sequence n: the packed call and the batched call
    compute the same chunks from the same states, so they agree bit for bit,
    including the masked last partial chunk (24 chains: two CTAs per chain in
    both calls; 96: one CTA per chain in both)."""
    import torch
    nseq, T = 3, 300
    c = gen.make_varlen_case([T] * nseq, H, seed=510, n_slots=nseq)
    c.slots[:] = np.arange(nseq, dtype=np.int32)
    d = dev_case(c)
    h0 = d["pool"].clone()
    o = gla.gla_chunk_fwd_varlen(d["q"], d["k"], d["v"], d["ll"], d["cu"], d["pool"], None, c.scale, 128)
    ob, hTb = gla.gla_chunk_fwd(d["q"].view(nseq, T, H, 96), d["k"].view(nseq, T, H, 96),
                                d["v"].view(nseq, T, H, 192), d["ll"], h0, c.scale, 128,
                                workspace=torch.empty(0, dtype=torch.uint8, device="cuda"))
    gla.gla_check()
    assert torch.equal(o.view(nseq, T, H, 192), ob)
    assert torch.equal(d["pool"], hTb)


def test_prefill_then_decode_continues_each_sequence(gla):
    """Prefill sequences of different lengths into the pool, then one decode
    step for every sequence on the same pool: the decode output and the new
    states match the oracle run over the prompt plus the new token."""
    lengths = [5, 130, 257, 64, 1]
    H = 4
    c = gen.make_varlen_case(lengths, H, seed=520, n_slots=len(lengths))
    c.slots[:] = np.arange(len(lengths), dtype=np.int32)
    d = dev_case(c)
    gla.gla_chunk_fwd_varlen(d["q"], d["k"], d["v"], d["ll"], d["cu"], d["pool"], None, c.scale, 128)
    tok = gen.decode_tokens(len(lengths), H, 96, 192, seed=521)
    o = gla.gla_decode_step(to_dev(tok["q"], "bf16"), to_dev(tok["k"], "bf16"), to_dev(tok["v"], "bf16"),
                            d["ll"], d["pool"], c.scale)
    gla.gla_check()
    oh, pool = to_host(o), to_host(d["pool"])
    for n in range(len(lengths)):
        a, b = int(c.cu_seqlens[n]), int(c.cu_seqlens[n + 1])
        q = np.concatenate([c.q[a:b], tok["q"][n][None]])[None]
        k = np.concatenate([c.k[a:b], tok["k"][n][None]])[None]
        v = np.concatenate([c.v[a:b], tok["v"][n][None]])[None]
        ro, rh = oracle.fwd_recurrent(q, k, v, c.log_lambda, c.pool[n][None].astype(np.float32), c.scale)
        assert relerr(oh[n], ro[0, -1]) <= TOL["bf16"], f"decode output of sequence {n}"
        assert relerr(pool[n], rh[0]) <= TOL["bf16"], f"state of sequence {n}"


def test_varlen_bad_device_offsets_are_reported(gla):
    """A decreasing cu_seqlens entry is device data the host cannot check: the
    kernel skips that sequence, leaves its slot alone, computes the others,
    and gla_check reports GLA_ERR_INVALID_ARG."""
    import torch
    lengths = [100, 50, 80]
    c = gen.make_varlen_case(lengths, 2, seed=530, n_slots=3)
    c.slots[:] = np.arange(3, dtype=np.int32)
    d = dev_case(c)
    bad = c.cu_seqlens.copy()
    bad[2] = bad[1] - 1   # sequence 1 ends before it starts; sequence 2 then starts there
    d["cu"] = torch.from_numpy(bad).cuda()
    gla.gla_chunk_fwd_varlen(d["q"], d["k"], d["v"], d["ll"], d["cu"], d["pool"], None, c.scale, 128)
    with pytest.raises(gla.GlaError) as ei:
        gla.gla_check()
    assert ei.value.status == gla.GLA_ERR_INVALID_ARG
    pool = to_host(d["pool"])
    assert np.array_equal(pool[1], c.pool[1].astype(np.float32).astype(np.float64))
    a = int(bad[0]); b = int(bad[1])
    _, rh = oracle.fwd_recurrent(c.q[None, a:b], c.k[None, a:b], c.v[None, a:b], c.log_lambda,
                                 c.pool[0][None].astype(np.float32), c.scale)
    assert relerr(pool[0], rh[0]) <= TOL["bf16"]
    gla.gla_check()   # the status word was cleared by the report
