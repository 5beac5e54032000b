"""Pins of the oracle's causal depthwise Conv1d (O8), checked without
retyping its formula: the linear part against numpy's convolution, SiLU by
its odd-part identity, causality, channel independence, and the window that
carries a sequence across calls.

Reading of "Beyond the KV cache: Training and serving i14's Laplace 3B linear
attention model on AWS Trainium2 with native PyTorch", section "i14 and the
Laplace 3B architecture", paragraph "Normalisation and convolution" (no
equation printed): y_t = SiLU(sum_i w[:, i] x_{t-3+i} + b) per channel, with
the inputs before a call taken from a window of the last four inputs."""
import numpy as np
import pytest

import oracle

pytestmark = pytest.mark.filterwarnings("ignore")


def case(seed, B=2, T=11, D=5):
    rng = np.random.default_rng(seed)
    return rng.normal(size=(B, T, D)), rng.normal(size=(D, 4)), rng.normal(size=D), rng.normal(size=(B, 4, D))


def odd(x, w, window=None):
    """y(x) - y(-x) with no bias: SiLU(a) - SiLU(-a) = a, so this is the
    pre-activation, the plain linear convolution."""
    wn = None if window is None else -window
    return oracle.conv1d(x, w, None, window)[0] - oracle.conv1d(-x, w, None, wn)[0]


def test_linear_part_is_numpy_causal_convolution():
    """The pre-activation of channel c is np.convolve of [window, x] with the
    taps reversed (a correlation), taking the outputs that end at each token:
    a swapped tap order or an off-by-one shift fails."""
    x, w, _, win = case(1)
    B, T, D = x.shape
    lin = odd(x, w, win)
    for bi in range(B):
        for c in range(D):
            seq = np.concatenate([win[bi, :, c], x[bi, :, c]])
            full = np.convolve(seq, w[c, ::-1], mode="valid")   # full[j] = sum_i w[i] seq[j + i]
            assert np.allclose(lin[bi, :, c], full[1:], rtol=1e-12, atol=1e-12)


def test_impulse_response_reads_the_taps_newest_last():
    """A unit input at token 2 reaches tokens 2, 3, 4, 5 through taps 3, 2, 1, 0."""
    x = np.zeros((1, 9, 3))
    x[0, 2] = 1.0
    w = np.arange(12, dtype=float).reshape(3, 4) + 1.0
    lin = odd(x, w)
    expect = np.zeros_like(x)
    for j, tap in enumerate((3, 2, 1, 0)):
        expect[0, 2 + j] = w[:, tap]
    assert np.allclose(lin, expect, rtol=1e-13, atol=1e-15)


def test_activation_is_silu():
    """w = 0 leaves SiLU(b) at every token: zero at b = 0, b at large b, 0 at
    very negative b, and SiLU(b) - SiLU(-b) = b."""
    x, _, _, _ = case(2)
    w = np.zeros((x.shape[2], 4))
    b = np.array([0.0, 40.0, -40.0, 1.5, -0.25])
    y = oracle.conv1d(x, w, b)[0]
    assert np.array_equal(y[..., 0], np.zeros_like(y[..., 0]))
    assert np.allclose(y[..., 1], 40.0, rtol=1e-15)
    assert np.all(np.abs(y[..., 2]) < 1e-15)
    yn = oracle.conv1d(x, w, -b)[0]
    assert np.allclose(y - yn, np.broadcast_to(b, y.shape), rtol=1e-13, atol=1e-15)
    # SiLU(1) = 1 / (1 + e^-1) to 1e-15 (the logistic function's textbook value)
    y1 = oracle.conv1d(np.zeros((1, 1, 1)), np.zeros((1, 4)), np.ones(1))[0]
    assert abs(y1[0, 0, 0] - 0.7310585786300049) < 1e-15


def test_causal():
    """Changing token t leaves the outputs of tokens before t unchanged and
    the ones after t + 3 too."""
    x, w, b, win = case(3)
    y = oracle.conv1d(x, w, b, win)[0]
    x2 = x.copy()
    x2[:, 5] += 3.0
    y2 = oracle.conv1d(x2, w, b, win)[0]
    assert np.array_equal(y[:, :5], y2[:, :5])
    assert np.array_equal(y[:, 9:], y2[:, 9:])
    assert not np.allclose(y[:, 5:9], y2[:, 5:9])


def test_depthwise():
    x, w, b, win = case(4)
    y = oracle.conv1d(x, w, b, win)[0]
    x2, w2 = x.copy(), w.copy()
    x2[..., 2] *= -2.0
    w2[3] += 1.0
    y2 = oracle.conv1d(x2, w2, b, win)[0]
    assert np.array_equal(np.delete(y, [2, 3], axis=-1), np.delete(y2, [2, 3], axis=-1))


def test_split_calls_carry_the_window():
    """One call over T tokens equals calls over the pieces of any split, each
    starting from the window the previous piece left (pieces of 1, 2 and 3
    tokens exercise the window carry-through)."""
    x, w, b, win = case(5, T=13)
    y, wout = oracle.conv1d(x, w, b, win)
    for cuts in ([1, 2, 3, 7], [4], [6, 7, 8], [12]):
        edges = [0] + cuts + [x.shape[1]]
        cur = win
        ys = []
        for a, e in zip(edges[:-1], edges[1:]):
            yy, cur = oracle.conv1d(x[:, a:e], w, b, cur)
            ys.append(yy)
        assert np.array_equal(np.concatenate(ys, axis=1), y)
        assert np.array_equal(cur, wout)


def test_window_contents():
    """The window out is the last four inputs; with fewer than four tokens the
    newest rows of the window in move up; a zero-length call returns it as is;
    no window equals a zero window."""
    x, w, b, win = case(6, T=6)
    assert np.array_equal(oracle.conv1d(x, w, b, win)[1], x[:, 2:6])
    for T in (1, 2, 3):
        _, wo = oracle.conv1d(x[:, :T], w, b, win)
        assert np.array_equal(wo, np.concatenate([win[:, T:], x[:, :T]], axis=1))
    y0, wo = oracle.conv1d(x[:, :0], w, b, win)
    assert y0.shape == (2, 0, 5) and np.array_equal(wo, win)
    assert np.array_equal(oracle.conv1d(x, w, b)[0], oracle.conv1d(x, w, b, np.zeros_like(win))[0])
    # the oldest window row is carried, never multiplied
    win2 = win.copy()
    win2[:, 0] = 1e6
    assert np.array_equal(oracle.conv1d(x, w, b, win2)[0], oracle.conv1d(x, w, b, win)[0])
