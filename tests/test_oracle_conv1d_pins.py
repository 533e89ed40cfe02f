"""Pins of the conv1d oracle (``oracle.conv1d``) to facts fixed by the page
("GDN Conv1D Kernel API Reference") and by the mathematics: a hand-worked
example, a library routine (numpy.convolve) on each channel, the impulse
response, closed-form values of SiLU, the K = 1 special case, the conv_state
as the raw tail, and the decode step chained token by token reproducing the
prefill (the two entry points' definitions written independently)."""
import json
import math
import os

import numpy as np
import pytest

from oracle import conv1d as oc

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def test_hand_worked_example():
    with open(os.path.join(GOLDEN, "conv1d_hand_worked.json")) as f:
        d = json.load(f)
    x = np.array(d["x"])[None, None, :]
    w = np.array(d["w"])[None, :]
    np.testing.assert_allclose(oc.causal_conv1d(x, w)[0, 0], d["z"], rtol=0, atol=1e-14)
    out, st = oc.conv1d_prefill(x, w)
    np.testing.assert_allclose(st[0, 0], d["state"], rtol=0, atol=0)
    yd, hs = oc.conv1d_decode(np.array([[[d["decode_x"]]]]), st, w)
    np.testing.assert_allclose(hs[0, 0], d["decode_state"], rtol=0, atol=0)
    # silu(9) through the closed form of the logistic function
    np.testing.assert_allclose(yd[0, 0, 0], 9.0 / (1.0 + math.exp(-9.0)), rtol=1e-15)


def test_matches_numpy_convolve_per_channel():
    """Causal depthwise conv == full convolution with the reversed taps, truncated."""
    rng = np.random.default_rng(11)
    B, C, T, K = 2, 5, 23, 4
    x = rng.standard_normal((B, C, T))
    w = rng.standard_normal((C, K))
    z = oc.causal_conv1d(x, w)
    for b in range(B):
        for c in range(C):
            ref = np.convolve(x[b, c], w[c, ::-1], mode="full")[:T]
            np.testing.assert_allclose(z[b, c], ref, rtol=1e-13, atol=1e-13)


def test_impulse_response_is_the_reversed_taps():
    K, T, t0 = 5, 16, 6
    w = np.arange(1, K + 1, dtype=np.float64)[None, :]
    x = np.zeros((1, 1, T))
    x[0, 0, t0] = 1.0
    z = oc.causal_conv1d(x, w)[0, 0]
    assert np.all(z[:t0] == 0)  # causal: nothing before the impulse
    np.testing.assert_array_equal(z[t0:t0 + K], w[0, ::-1])
    assert np.all(z[t0 + K:] == 0)


def test_silu_closed_forms():
    # sigmoid(ln 3) = 3/4, sigmoid(0) = 1/2, silu(-z) = silu(z) - z
    np.testing.assert_allclose(oc.silu(math.log(3.0)), 0.75 * math.log(3.0), rtol=1e-15)
    assert oc.silu(0.0) == 0.0
    z = np.linspace(-20, 20, 81)
    np.testing.assert_allclose(oc.silu(-z), oc.silu(z) - z, rtol=1e-12, atol=1e-12)
    assert abs(oc.silu(-40.0)) < 1e-15 and abs(oc.silu(40.0) - 40.0) < 1e-12


def test_single_tap_is_elementwise():
    rng = np.random.default_rng(3)
    x = rng.standard_normal((2, 3, 9))
    w = rng.standard_normal((3, 1))
    np.testing.assert_allclose(oc.causal_conv1d(x, w), w[None, :, :] * x, rtol=1e-15)


@pytest.mark.parametrize("T", [0, 1, 2, 3, 4, 7])
def test_state_is_the_raw_tail(T):
    rng = np.random.default_rng(T)
    K = 4
    x = rng.standard_normal((2, 3, T))
    st = oc.last_tokens(x, K)
    n = min(T, K)
    assert st.shape == (2, 3, K)
    np.testing.assert_array_equal(st[:, :, K - n:], x[:, :, T - n:])
    assert np.all(st[:, :, : K - n] == 0)


@pytest.mark.parametrize("T,K", [(1, 4), (3, 4), (12, 4), (9, 1), (10, 6)])
def test_decode_chain_equals_prefill(T, K):
    """Token-by-token decode from a zero window == prefill (output and state)."""
    rng = np.random.default_rng(100 + T * 10 + K)
    B, C = 2, 3
    x = rng.standard_normal((B, C, T))
    w = rng.standard_normal((C, K))
    out, st = oc.conv1d_prefill(x, w)
    s = np.zeros((B, C, K))
    for t in range(T):
        y, s = oc.conv1d_decode(x[:, :, t:t + 1], s, w)
        np.testing.assert_allclose(y[:, :, 0], out[:, :, t], rtol=1e-13, atol=1e-14)
    np.testing.assert_array_equal(s, st)
