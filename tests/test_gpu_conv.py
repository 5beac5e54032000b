"""GPU parity of the causal depthwise Conv1d with SiLU (gla_conv1d_fwd,
gla_conv1d_varlen, gla_conv1d_step) against the double-precision oracle,
plus the properties that tie the three together: a call split at any point
(or run token by token through the serving step) gives the same bits as one
call, because every token sees the same four inputs in the same order."""
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


def dev(c):
    return to_dev(c.x, c.dtype), f32_dev(c.w), f32_dev(c.b), f32_dev(c.window)


@pytest.mark.parametrize("dtype,B,T,D", [("bf16", 3, 37, 3072), ("bf16", 2, 300, 24), ("bf16", 1, 1, 3072),
                                         ("bf16", 4, 2, 1032), ("fp32", 2, 53, 516), ("fp32", 1, 3, 4),
                                         ("bf16", 2, 40, 4096), ("fp32", 2, 21, 3072), ("bf16", 2, 33, 3840),
                                         ("fp32", 2, 19, 1920)])
def test_fwd_matches_oracle(gla, dtype, B, T, D):
    c = gen.make_conv_case(B, T, D, seed=600 + T, dtype=dtype)
    x, w, b, win = dev(c)
    y, wo = gla.gla_conv1d_fwd(x, w, b, win)
    gla.gla_check()
    ry, rw = oracle.conv1d(c.x, c.w, c.b, c.window)
    assert relerr(to_host(y), ry) <= TOL[dtype]
    assert np.array_equal(to_host(wo), rw)          # windows hold inputs: exact
    # no window in (zeros) and no bias
    y0, _ = gla.gla_conv1d_fwd(x, w, None, None, want_window=False)
    gla.gla_check()
    assert relerr(to_host(y0), oracle.conv1d(c.x, c.w, None, None)[0]) <= TOL[dtype]


def test_fwd_in_place_window_and_empty_call(gla):
    import torch
    c = gen.make_conv_case(2, 7, 3072, seed=610)
    x, w, b, win = dev(c)
    ref = win.clone()
    y, wo = gla.gla_conv1d_fwd(x, w, b, win, win_out=win)
    gla.gla_check()
    assert wo is win
    assert np.array_equal(to_host(win), oracle.conv1d(c.x, c.w, c.b, c.window)[1])
    y2, _ = gla.gla_conv1d_fwd(x, w, b, ref, want_window=False)
    gla.gla_check()
    assert torch.equal(y, y2)
    # T = 0 copies the window through
    e = x[:, :0].contiguous()
    _, wo0 = gla.gla_conv1d_fwd(e, w, b, ref)
    gla.gla_check()
    assert torch.equal(wo0, ref)


def test_split_calls_equal_one_call_bitwise(gla):
    import torch
    c = gen.make_conv_case(2, 45, 3072, seed=620)
    x, w, b, win = dev(c)
    y, wo = gla.gla_conv1d_fwd(x, w, b, win)
    for cuts in ([1, 2, 3, 20], [16, 32], [44]):
        edges = [0] + cuts + [45]
        cur = win.clone()
        ys = []
        for a, e in zip(edges[:-1], edges[1:]):
            yy, _ = gla.gla_conv1d_fwd(x[:, a:e].contiguous(), w, b, cur, win_out=cur)
            ys.append(yy)
        gla.gla_check()
        assert torch.equal(torch.cat(ys, dim=1), y)
        assert torch.equal(cur, wo)


def test_step_matches_oracle_and_chains_to_the_fwd(gla):
    """One serving step equals the oracle on one token; T steps equal one
    forward call over the T tokens, output and window, bit for bit."""
    import torch
    N, T, D = 5, 6, 3072
    c = gen.make_conv_case(N, T, D, seed=630)
    x, w, b, win = dev(c)
    cur = win.clone()
    y1 = gla.gla_conv1d_step(x[:, 0].contiguous(), w, b, cur)
    gla.gla_check()
    ry, rw = oracle.conv1d(c.x[:, :1], c.w, c.b, c.window)
    assert relerr(to_host(y1), ry[:, 0]) <= TOL["bf16"]
    assert np.array_equal(to_host(cur), rw)
    ys = [y1]
    for t in range(1, T):
        ys.append(gla.gla_conv1d_step(x[:, t].contiguous(), w, b, cur))
    yf, wf = gla.gla_conv1d_fwd(x, w, b, win)
    gla.gla_check()
    assert torch.equal(torch.stack(ys, dim=1), yf)
    assert torch.equal(cur, wf)
    # fp32 validation mode
    c32 = gen.make_conv_case(3, 1, 516, seed=631, dtype="fp32")
    x32, w32, b32, win32 = dev(c32)
    y32 = gla.gla_conv1d_step(x32[:, 0].contiguous(), w32, b32, win32)
    gla.gla_check()
    ry, rw = oracle.conv1d(c32.x, c32.w, c32.b, c32.window)
    assert relerr(to_host(y32), ry[:, 0]) <= TOL["fp32"]
    assert np.array_equal(to_host(win32), rw)


def varlen_case(lengths, n_slots, seed, D=3072):
    rng = np.random.default_rng(seed)
    lengths = np.asarray(lengths)
    cu = np.zeros(len(lengths) + 1, dtype=np.int32)
    cu[1:] = np.cumsum(lengths)
    c = gen.make_conv_case(1, int(cu[-1]), D, seed=seed)
    pool = gen.make_conv_case(n_slots, 0, D, seed=seed + 1).window
    slots = rng.permutation(n_slots)[:len(lengths)].astype(np.int32)
    return c, cu, slots, pool


def test_varlen_matches_oracle_per_sequence(gla):
    import torch
    lengths = [0, 1, 2, 3, 4, 5, 15, 16, 17, 31, 100, 200]
    n_slots = 16
    c, cu, slots, pool = varlen_case(lengths, n_slots, 640)
    x = to_dev(c.x[0], "bf16")
    total = int(cu[-1])
    pad = torch.zeros((total + 9, 3072), dtype=torch.bfloat16, device="cuda")   # 9 tokens past the last sequence
    pad[:total] = x
    y = torch.full_like(pad, 7.0)
    pool_d = f32_dev(pool)
    gla.gla_conv1d_varlen(pad, f32_dev(c.w), f32_dev(c.b), torch.from_numpy(cu).cuda(), pool_d,
                          torch.from_numpy(slots).cuda(), y=y)
    gla.gla_check()
    yh, ph = to_host(y), to_host(pool_d)
    for n, L in enumerate(lengths):
        a, e = int(cu[n]), int(cu[n + 1])
        if L == 0:
            continue
        ry, rw = oracle.conv1d(c.x[:, a:e], c.w, c.b, pool[slots[n]][None])
        assert relerr(yh[a:e], ry[0]) <= TOL["bf16"], f"y of sequence {n} (length {L})"
        assert np.array_equal(ph[slots[n]], rw[0]), f"window of sequence {n}"
    used = set(int(slots[n]) for n, L in enumerate(lengths) if L > 0)
    for s in range(n_slots):
        if s not in used:
            assert np.array_equal(ph[s], pool[s].astype(np.float64)), f"slot {s} changed"
    assert np.all(yh[total:] == 7.0)                 # tokens past cu_seqlens[nseq]: no output


def test_varlen_equals_batched(gla):
    import torch
    B, T = 3, 50
    c = gen.make_conv_case(B, T, 3072, seed=650)
    x, w, b, win = dev(c)
    y, wo = gla.gla_conv1d_fwd(x, w, b, win)
    cu = torch.arange(0, B * T + 1, T, dtype=torch.int32, device="cuda")
    pool = win.clone()
    yv = gla.gla_conv1d_varlen(x.view(B * T, 3072), w, b, cu, pool)
    gla.gla_check()
    assert torch.equal(yv.view(B, T, 3072), y)
    assert torch.equal(pool, wo)


def test_varlen_prefill_then_steps(gla):
    """Prefill prompts of different lengths into the window pool, then two
    serving steps per sequence: the outputs and windows continue each
    sequence exactly as the oracle over prompt + new tokens."""
    import torch
    lengths = [3, 1, 40, 2]
    c, cu, _, _ = varlen_case(lengths, 4, 660)
    pool = torch.zeros((4, 4, 3072), dtype=torch.float32, device="cuda")
    w, b = f32_dev(c.w), f32_dev(c.b)
    gla.gla_conv1d_varlen(to_dev(c.x[0], "bf16"), w, b, torch.from_numpy(cu).cuda(), pool)
    new = gen.make_conv_case(4, 2, 3072, seed=661)
    ys = [gla.gla_conv1d_step(to_dev(np.ascontiguousarray(new.x[:, t]), "bf16"), w, b, pool) for t in range(2)]
    gla.gla_check()
    for n in range(4):
        a, e = int(cu[n]), int(cu[n + 1])
        xs = np.concatenate([c.x[0, a:e], new.x[n]])[None]
        ry, rw = oracle.conv1d(xs, c.w, c.b, None)
        for t in range(2):
            assert relerr(to_host(ys[t])[n], ry[0, e - a + t]) <= TOL["bf16"]
        assert np.array_equal(to_host(pool)[n], rw[0])


def test_varlen_bad_offsets_are_reported(gla):
    import torch
    lengths = [30, 20, 25]
    c, cu, _, pool = varlen_case(lengths, 3, 670)
    bad = cu.copy()
    bad[2] = bad[1] - 1          # sequence 1 ends before it starts
    pool_d = f32_dev(pool)
    y = torch.zeros((int(cu[-1]), 3072), dtype=torch.bfloat16, device="cuda")
    gla.gla_conv1d_varlen(to_dev(c.x[0], "bf16"), f32_dev(c.w), f32_dev(c.b), torch.from_numpy(bad).cuda(), pool_d,
                          y=y)
    with pytest.raises(gla.GlaError) as ei:
        gla.gla_check()
    assert ei.value.status == gla.GLA_ERR_INVALID_ARG
    ph = to_host(pool_d)
    assert np.array_equal(ph[1], pool[1].astype(np.float64))      # the bad sequence's slot is untouched
    ry, rw = oracle.conv1d(c.x[:, :int(bad[1])], c.w, c.b, pool[0][None])
    assert relerr(to_host(y)[:int(bad[1])], ry[0]) <= TOL["bf16"]
    assert np.array_equal(ph[0], rw[0])
    gla.gla_check()


def test_full_size_sampled_channels(gla):
    """The layer-forward workload ([8, 2048, 3072] bf16, one launch as the
    benchmark times it): every token of a sample of channels against the
    oracle (the conv is depthwise, so a channel subset is exact)."""
    import torch
    B, T, D = 8, 2048, 3072
    c = gen.make_conv_case(B, T, D, seed=680)
    x, w, b, win = dev(c)
    y, wo = gla.gla_conv1d_fwd(x, w, b, win)
    gla.gla_check()
    ch = np.array([0, 1, 7, 8, 1023, 1024, 2047, 3064, 3071])
    ry, rw = oracle.conv1d(c.x[:, :, ch], c.w[ch], c.b[ch], c.window[:, :, ch])
    idx = torch.from_numpy(ch).cuda()
    assert relerr(to_host(y[:, :, idx]), ry) <= TOL["bf16"]
    assert np.array_equal(to_host(wo[:, :, idx]), rw)


def test_varlen_serving_prefill_sampled_channels(gla):
    """The serving prefill mix (64 prompts, log-uniform 64..4096 tokens) at
    D = 3072: every CTA streams many tiles across sequence boundaries. Every
    token of a sample of channels, and their windows, against the oracle."""
    import torch
    lengths = gen.serving_prefill_lengths()
    n_slots = 80
    c, cu, slots, pool = varlen_case(lengths, n_slots, 690)
    pool_d = f32_dev(pool)
    y = gla.gla_conv1d_varlen(to_dev(c.x[0], "bf16"), f32_dev(c.w), f32_dev(c.b), torch.from_numpy(cu).cuda(),
                              pool_d, torch.from_numpy(slots).cuda())
    gla.gla_check()
    ch = np.array([0, 5, 8, 1000, 2047, 2048, 3071])
    yh = to_host(y[:, torch.from_numpy(ch).cuda()])
    ph = to_host(pool_d)[:, :, ch]
    for n in range(len(lengths)):
        a, e = int(cu[n]), int(cu[n + 1])
        ry, rw = oracle.conv1d(c.x[:, a:e][:, :, ch], c.w[ch], c.b[ch], pool[slots[n]][None][:, :, ch])
        assert relerr(yh[a:e], ry[0]) <= TOL["bf16"], f"sequence {n}"
        assert np.array_equal(ph[slots[n]], rw[0]), f"window of sequence {n}"
