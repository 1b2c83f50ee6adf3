"""Pins of the FP64 conv1d + SiLU oracle (oracle/conv1d.py) to facts outside the oracle itself.

* a hand-worked three-token example (pre-activations worked out by hand);
* the identity tap reduces to SiLU, written here with scipy's logistic function;
* the oldest tap alone is a pure three-token shift inside each document (causal direction and
  the reset at document starts);
* every channel of every document equals numpy.convolve of the channel with the reversed taps;
* a document cut in two, with the first piece's last three tokens as the second piece's halo,
  gives the same outputs and gradients as the whole document;
* central finite differences of L = sum(y * dy) for dx, dw, db and dhalo.
"""
import numpy as np
import pytest
from scipy.special import expit

from oracle import conv1d


def _case(rng, lens, C, halo=False):
    T = int(sum(lens))
    cu = np.concatenate([[0], np.cumsum(lens)]).astype(np.int64)
    x = rng.standard_normal((T, C))
    w = rng.standard_normal((C, 4)) * 0.5
    b = rng.standard_normal(C) * 0.1
    h = rng.standard_normal((len(lens), 3, C)) if halo else None
    return x, w, b, cu, h


def test_hand_worked_example():
    # one channel, taps w = (0.5, -1, 2, 1) on x[t-3], x[t-2], x[t-1], x[t], bias 0.25
    x = np.array([[1.0], [2.0], [-1.0]])
    w = np.array([[0.5, -1.0, 2.0, 1.0]])
    y, z = conv1d.conv_fwd(x, w, [0, 3], bias=np.array([0.25]))
    # z0 = 0.25 + 1*1;  z1 = 0.25 + 2*1 + 1*2;  z2 = 0.25 - 1*1 + 2*2 + 1*(-1)
    assert np.allclose(z[:, 0], [1.25, 4.25, 2.25], rtol=0, atol=1e-15)
    assert np.allclose(y[:, 0], [1.25 / (1 + np.exp(-1.25)), 4.25 / (1 + np.exp(-4.25)),
                                 2.25 / (1 + np.exp(-2.25))], rtol=1e-15)


def test_identity_tap_is_silu():
    rng = np.random.default_rng(0)
    x, _, _, cu, _ = _case(rng, [9, 4], 5)
    w = np.zeros((5, 4))
    w[:, 3] = 1.0
    y, _ = conv1d.conv_fwd(x, w, cu)
    assert np.allclose(y, x * expit(x), rtol=1e-14, atol=1e-15)


def test_oldest_tap_is_a_causal_shift_reset_per_document():
    rng = np.random.default_rng(1)
    lens = [7, 2, 5]
    x, _, _, cu, _ = _case(rng, lens, 3)
    w = np.zeros((3, 4))
    w[:, 0] = 1.0
    _, z = conv1d.conv_fwd(x, w, cu, activation=False)
    want = np.zeros_like(x)
    for a, e in zip(cu[:-1], cu[1:]):
        for t in range(a, e):
            if t - 3 >= a:
                want[t] = x[t - 3]
    assert np.array_equal(z, want)


def test_every_channel_equals_numpy_convolve():
    rng = np.random.default_rng(2)
    lens = [11, 1, 6]
    x, w, b, cu, _ = _case(rng, lens, 4)
    _, z = conv1d.conv_fwd(x, w, cu, bias=b)
    for a, e in zip(cu[:-1], cu[1:]):
        for c in range(4):
            ref = np.convolve(x[a:e, c], w[c, ::-1], mode="full")[: e - a] + b[c]
            assert np.allclose(z[a:e, c], ref, rtol=1e-13, atol=1e-14)


@pytest.mark.parametrize("cut", [1, 2, 3, 6])
def test_halo_split_equals_whole_document(cut):
    rng = np.random.default_rng(3)
    x, w, b, _, _ = _case(rng, [10], 3)
    dy = rng.standard_normal(x.shape)
    whole_y, _ = conv1d.conv_fwd(x, w, [0, 10], bias=b)
    whole_g = conv1d.conv_bwd(x, w, [0, 10], dy, bias=b)
    # two pieces: the second piece's halo = the three tokens before it (zeros before the start)
    halo = np.zeros((2, 3, 3))
    for i in range(3):
        t = cut - 3 + i
        if t >= 0:
            halo[1, i] = x[t]
    y, _ = conv1d.conv_fwd(x, w, [0, cut, 10], bias=b, halo=halo)
    g = conv1d.conv_bwd(x, w, [0, cut, 10], dy, bias=b, halo=halo)
    assert np.allclose(y, whole_y, rtol=1e-14, atol=1e-15)
    assert np.allclose(g["dw"], whole_g["dw"], rtol=1e-13, atol=1e-14)
    assert np.allclose(g["db"], whole_g["db"], rtol=1e-13, atol=1e-14)
    # the second piece's halo gradient is what flows back into the first piece's last tokens
    dx = g["dx"].copy()
    for i in range(3):
        t = cut - 3 + i
        if t >= 0:
            dx[t] += g["dhalo"][1, i]
    assert np.allclose(dx, whole_g["dx"], rtol=1e-13, atol=1e-14)


def test_gradients_by_central_differences():
    rng = np.random.default_rng(4)
    x, w, b, cu, h = _case(rng, [6, 3], 3, halo=True)
    dy = rng.standard_normal(x.shape)

    def loss(x_, w_, b_, h_):
        y, _ = conv1d.conv_fwd(x_, w_, cu, bias=b_, halo=h_)
        return float(np.sum(y * dy))

    g = conv1d.conv_bwd(x, w, cu, dy, bias=b, halo=h)
    eps = 1e-6
    for name, arr, grad in (("x", x, g["dx"]), ("w", w, g["dw"]), ("b", b, g["db"]),
                            ("halo", h, g["dhalo"])):
        fd = np.zeros_like(arr)
        for idx in np.ndindex(arr.shape):
            p, m = arr.copy(), arr.copy()
            p[idx] += eps
            m[idx] -= eps
            args_p = {"x": x, "w": w, "b": b, "halo": h}
            args_m = dict(args_p)
            args_p[name], args_m[name] = p, m
            fd[idx] = (loss(args_p["x"], args_p["w"], args_p["b"], args_p["halo"])
                       - loss(args_m["x"], args_m["w"], args_m["b"], args_m["halo"])) / (2 * eps)
        err = np.max(np.abs(fd - grad)) / max(np.max(np.abs(grad)), 1e-30)
        assert err < 1e-6, (name, err)
