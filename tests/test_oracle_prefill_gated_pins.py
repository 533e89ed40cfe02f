"""Pins of the gated prefill oracle (``oracle.prefill_gated``) against the
separately pinned gated decode oracle: a prefill of S tokens with q, k already
of unit norm and g, beta given directly must produce, token by token, what S
single gated decode steps produce when their raw gate inputs are chosen so that
the gates come out as those g and beta (softplus and sigmoid inverted in closed
form).  A dropped decay, a transposed state or a norm over the wrong axis shows
up as a mismatch."""
import math

import numpy as np

import oracle
from oracle import gated_decode as og
from oracle import prefill_gated as opg


def test_prefill_gated_is_a_sequence_of_gated_decode_steps():
    rng = np.random.default_rng(11)
    B, Hk, Hv, S, Dk, Dv = 2, 1, 2, 5, 6, 4
    q = rng.standard_normal((B, Hk, S, Dk))
    k = rng.standard_normal((B, Hk, S, Dk))
    q /= np.linalg.norm(q, axis=-1, keepdims=True)
    k /= np.linalg.norm(k, axis=-1, keepdims=True)
    v = rng.standard_normal((B, Hv, S, Dv))
    z = rng.standard_normal((B, Hv, S, Dv))
    g = rng.uniform(-0.8, -0.05, (B, Hv, S))
    beta = rng.uniform(0.1, 0.9, (B, Hv, S))
    w = 1.0 + 0.1 * rng.standard_normal(Dv)
    st0 = 0.3 * rng.standard_normal((B, Hv, Dk, Dv))
    scale = 1.0 / math.sqrt(Dk)
    y, st = opg.prefill_gated(q, k, v, g, beta, z, w, scale, st0)

    # the same tokens through the decode oracle: A_log = dt_bias = 0 gives g = -softplus(a),
    # so a = log(e^{-g} - 1); beta = sigmoid(b) gives b = log(beta / (1 - beta))
    a_raw = np.log(np.expm1(-g))
    b_raw = np.log(beta / (1.0 - beta))
    cur = st0.copy()
    for t in range(S):
        qkv = np.concatenate([q[:, :, t].reshape(B, -1), k[:, :, t].reshape(B, -1), v[:, :, t].reshape(B, -1)], axis=1)
        yt, cur = og.decode_gated(qkv, z[:, :, t].reshape(B, -1), a_raw[:, :, t], b_raw[:, :, t], np.zeros(Hv),
                                  np.zeros(Hv), w, scale, cur, Hk, Hv, Dk, Dv)
        # the decode oracle re-normalises q and k with eps 1e-6: a relative 5e-7 difference
        np.testing.assert_allclose(y[:, :, t].reshape(B, -1), yt, rtol=2e-5, atol=1e-7)
    np.testing.assert_allclose(st, cur, rtol=2e-5, atol=1e-7)


def test_unit_rms_before_the_gate():
    """With norm_weight = 1 and z large (silu(z) = z to double precision), y / z has unit
    RMS over Dv for every token (up to the epsilon)."""
    rng = np.random.default_rng(12)
    B, Hk, Hv, S, Dk, Dv = 1, 1, 1, 7, 4, 8
    q = rng.standard_normal((B, Hk, S, Dk))
    k = rng.standard_normal((B, Hk, S, Dk))
    v = rng.standard_normal((B, Hv, S, Dv))
    g = rng.uniform(-0.5, -0.1, (B, Hv, S))
    beta = rng.uniform(0.2, 0.8, (B, Hv, S))
    z = np.full((B, Hv, S, Dv), 60.0)
    y, _ = opg.prefill_gated(q, k, v, g, beta, z, np.ones(Dv), 0.5, None)
    o, _ = oracle.recurrence(q, k, v, g, beta, 0.5, None)
    rms = np.sqrt(np.mean((y / 60.0) ** 2, axis=-1))
    expect = np.sqrt(np.mean(o ** 2, axis=-1) / (np.mean(o ** 2, axis=-1) + 1e-6))
    np.testing.assert_allclose(rms, expect, rtol=1e-12)
