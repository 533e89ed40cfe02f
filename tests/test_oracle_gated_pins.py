"""Pins of the gated decode oracle (``oracle.gated_decode``): its gate mapping
against closed forms (softplus(0) = ln 2, sigmoid(0) = 1/2), its core against
the separately pinned recurrence oracle (the direction of the normalised
output), and its epilogue against invariants of RMSNormGated (unit RMS before
the gate, a zero gate giving zero, scale invariance of the L2-normalised
inputs)."""
import math

import numpy as np
import pytest

import oracle
from oracle import gated_decode as og

B, Hk, Hv, Dk, Dv = 2, 2, 4, 8, 6


def _raw(rng, state=True):
    qkv = rng.standard_normal((B, 2 * Hk * Dk + Hv * Dv))
    z = rng.standard_normal((B, Hv * Dv))
    a = rng.standard_normal((B, Hv))
    b = rng.standard_normal((B, Hv))
    A_log = np.log(rng.uniform(1.0, 16.0, Hv))
    dt_bias = rng.uniform(-4.0, -1.0, Hv)
    w = 1.0 + 0.1 * rng.standard_normal(Dv)
    st = 0.2 * rng.standard_normal((B, Hv, Dk, Dv)) if state else None
    return qkv, z, a, b, A_log, dt_bias, w, st


def test_gate_closed_forms():
    # a + dt_bias = 0 and A_log = 0 -> g = -softplus(0) = -ln 2, i.e. a decay factor of exactly 1/2
    g, beta = og.gates(np.zeros((1, 3)), np.zeros((1, 3)), np.zeros(3), np.zeros(3))
    np.testing.assert_allclose(g, -math.log(2.0), rtol=1e-15)
    np.testing.assert_allclose(beta, 0.5, rtol=0)
    # A_log scales the decay rate: g = -e^{A_log} ln 2
    g2, _ = og.gates(np.zeros((1, 1)), np.zeros((1, 1)), np.array([math.log(3.0)]), np.zeros(1))
    np.testing.assert_allclose(g2, -3.0 * math.log(2.0), rtol=1e-14)
    # large arguments: softplus(x) -> x, sigmoid(-x) -> 0
    g3, beta3 = og.gates(np.array([[50.0]]), np.array([[-60.0]]), np.zeros(1), np.zeros(1))
    np.testing.assert_allclose(g3, -50.0, rtol=1e-15)
    assert beta3[0, 0] < 1e-25


def test_pure_decay_halves_the_state():
    """beta -> 0 (b = -80) and g = -ln 2: the new state is exactly half the old one."""
    rng = np.random.default_rng(1)
    qkv, z, a, b, A_log, dt_bias, w, st = _raw(rng)
    a[:] = 0.0
    b[:] = -80.0
    _, st2 = og.decode_gated(qkv, z, a, b, np.zeros(Hv), np.zeros(Hv), w, 0.5, st, Hk, Hv, Dk, Dv)
    np.testing.assert_allclose(st2, 0.5 * st, rtol=1e-14, atol=1e-30)


def test_core_is_the_pinned_recurrence():
    """y / (norm_weight silu(z)) is parallel to the recurrence oracle's output for the
    g, beta the gates produce, on the L2-normalised q, k."""
    rng = np.random.default_rng(2)
    qkv, z, a, b, A_log, dt_bias, w, st = _raw(rng)
    scale = 1.0 / math.sqrt(Dk)
    y, st2 = og.decode_gated(qkv, z, a, b, A_log, dt_bias, w, scale, st, Hk, Hv, Dk, Dv)
    kd = Hk * Dk
    nrm = lambda x: x / np.sqrt(np.sum(x * x, -1, keepdims=True) + og.EPS_L2)
    q = nrm(qkv[:, :kd].reshape(B, Hk, Dk))
    k = nrm(qkv[:, kd:2 * kd].reshape(B, Hk, Dk))
    v = qkv[:, 2 * kd:].reshape(B, Hv, Dv)
    g = -np.exp(A_log)[None] * np.log1p(np.exp(a + dt_bias[None]))
    beta = 1.0 / (1.0 + np.exp(-b))
    o, s_ref = oracle.recurrence(q[:, :, None], k[:, :, None], v[:, :, None], g[:, :, None], beta[:, :, None],
                                 scale, st)
    np.testing.assert_allclose(st2, s_ref, rtol=1e-12, atol=1e-14)
    gate = (w[None, None, :] * og.silu(z.reshape(B, Hv, Dv)))
    r = y.reshape(B, Hv, Dv) / gate
    o = o[:, :, 0, :]
    cos = np.sum(r * o, -1) / (np.linalg.norm(r, axis=-1) * np.linalg.norm(o, axis=-1))
    np.testing.assert_allclose(cos, 1.0, rtol=0, atol=1e-12)
    # and its RMS is 1 up to the epsilon
    ms = np.mean(o * o, -1)
    np.testing.assert_allclose(np.sqrt(np.mean(r * r, -1)), np.sqrt(ms / (ms + og.EPS_RMS)), rtol=1e-12)


def test_zero_gate_gives_zero_and_the_state_still_updates():
    rng = np.random.default_rng(3)
    qkv, z, a, b, A_log, dt_bias, w, st = _raw(rng)
    y, st2 = og.decode_gated(qkv, np.zeros_like(z), a, b, A_log, dt_bias, w, 0.3, st, Hk, Hv, Dk, Dv)
    assert np.all(y == 0.0)
    assert not np.allclose(st2, st)


def test_qk_scale_invariance():
    """Positive rescaling of q or k before the L2 normalisation changes nothing (up to eps)."""
    rng = np.random.default_rng(4)
    qkv, z, a, b, A_log, dt_bias, w, st = _raw(rng)
    y, st2 = og.decode_gated(qkv, z, a, b, A_log, dt_bias, w, 0.3, st, Hk, Hv, Dk, Dv)
    qkv2 = qkv.copy()
    qkv2[:, : 2 * Hk * Dk] *= 7.0
    y2, st3 = og.decode_gated(qkv2, z, a, b, A_log, dt_bias, w, 0.3, st, Hk, Hv, Dk, Dv)
    # the epsilon makes the invariance approximate: ~eps / |x|^2 ~ 1e-7 relative per input
    np.testing.assert_allclose(y2, y, rtol=1e-5, atol=1e-8)
    np.testing.assert_allclose(st3, st2, rtol=1e-5, atol=1e-8)


@pytest.mark.parametrize("state", [True, False])
def test_gqa_blocks_and_zero_state(state):
    """Value heads 0, 1 read key head 0 and 2, 3 key head 1 (blocked); zeroing key head 1's
    q/k/v inputs changes only value heads 2, 3."""
    rng = np.random.default_rng(5)
    qkv, z, a, b, A_log, dt_bias, w, st = _raw(rng, state)
    y, _ = og.decode_gated(qkv, z, a, b, A_log, dt_bias, w, 0.3, st, Hk, Hv, Dk, Dv)
    qkv2 = qkv.copy()
    qkv2[:, Dk:2 * Dk] = 3.0           # q of key head 1
    qkv2[:, Hk * Dk + Dk:2 * Hk * Dk] = -2.0  # k of key head 1
    y2, _ = og.decode_gated(qkv2, z, a, b, A_log, dt_bias, w, 0.3, st, Hk, Hv, Dk, Dv)
    yh, y2h = y.reshape(B, Hv, Dv), y2.reshape(B, Hv, Dv)
    np.testing.assert_array_equal(yh[:, :2], y2h[:, :2])
    assert not np.allclose(yh[:, 2:], y2h[:, 2:])
