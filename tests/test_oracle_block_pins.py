"""Pins of the decode-block oracle (``oracle.decode_block``): with identity
projections the block must equal the separately pinned conv1d and gated-step
oracles applied to the hidden state itself (checks the split into q|k|v, z, a,
b and the order of the stages), and a zero hidden state gives zero projections
(a zero token shifted into the conv window, a zero output through the zero gate)."""
import math

import numpy as np

from oracle import conv1d as oc
from oracle import decode_block as ob
from oracle import gated_decode as og

B, Hk, Hv, Dk, Dv, K = 2, 1, 2, 4, 3, 3
C = 2 * Hk * Dk + Hv * Dv


def _params(rng):
    conv_w = rng.standard_normal((C, K))
    conv_st = rng.standard_normal((B, C, K))
    A_log = np.log(rng.uniform(1, 16, Hv))
    dt_bias = rng.uniform(-4, -1, Hv)
    nw = 1 + 0.1 * rng.standard_normal(Dv)
    st = 0.2 * rng.standard_normal((B, Hv, Dk, Dv))
    return conv_w, conv_st, A_log, dt_bias, nw, st


def test_identity_projections_reduce_to_the_stages():
    rng = np.random.default_rng(0)
    H = C + Hv * Dv + 2 * Hv
    hidden = rng.standard_normal((B, 1, H))
    eye = np.eye(H)
    W_qkv, W_z = eye[:, :C], eye[:, C:C + Hv * Dv]
    W_a, W_b = eye[:, C + Hv * Dv:C + Hv * Dv + Hv], eye[:, C + Hv * Dv + Hv:]
    conv_w, conv_st, A_log, dt_bias, nw, st = _params(rng)
    y, cst, s2 = ob.decode_block(hidden, W_qkv, W_z, W_a, W_b, conv_w, conv_st, A_log, dt_bias, nw, st,
                                 Hk, Hv, Dk, Dv)
    h = hidden[:, 0, :]
    co, cst_ref = oc.conv1d_decode(h[:, :C, None], conv_st, conv_w)
    y_ref, s_ref = og.decode_gated(co[:, :, 0], h[:, C:C + Hv * Dv], h[:, C + Hv * Dv:C + Hv * Dv + Hv],
                                   h[:, C + Hv * Dv + Hv:], A_log, dt_bias, nw, 1 / math.sqrt(Dk), st,
                                   Hk, Hv, Dk, Dv)
    np.testing.assert_allclose(y[:, 0], y_ref, rtol=1e-13, atol=1e-15)
    np.testing.assert_array_equal(cst, cst_ref)
    np.testing.assert_allclose(s2, s_ref, rtol=1e-13, atol=1e-15)


def test_zero_hidden_state_projects_to_zero():
    """hidden = 0: the conv sees a zero token (the window shifts in a 0), z = 0 gives y = 0,
    and a = b = 0 gives beta = 1/2 and g = -exp(A_log) softplus(dt_bias)."""
    rng = np.random.default_rng(1)
    H = 5
    conv_w, conv_st, A_log, dt_bias, nw, st = _params(rng)
    Ws = [rng.standard_normal((H, n)) for n in (C, Hv * Dv, Hv, Hv)]
    y, cst, _ = ob.decode_block(np.zeros((B, 1, H)), *Ws, conv_w, conv_st, A_log, dt_bias, nw, st, Hk, Hv, Dk, Dv)
    assert np.all(y == 0)
    np.testing.assert_array_equal(cst[:, :, :-1], conv_st[:, :, 1:])
    assert np.all(cst[:, :, -1] == 0)
