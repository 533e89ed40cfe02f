"""Pins of the fp64 oracle to facts fixed by the pages and by the mathematics.

Every test here runs on the CPU.  None of them re-types the oracle's formula:
each compares it with a hand-worked example, a closed form, an invariant, or a
second formulation (the chunk algebra) that a plausible mistake (a dropped
term, a wrong sign or index, a transposed operand, the pre-update state used
for the output, a modulo head mapping) would break.
"""
import json
import os

import numpy as np
import pytest

import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _rand_inputs(rng, B=2, Hk=2, Hv=4, S=37, Dk=5, Dv=3, state=True, g_lo=-0.5, g_hi=-0.005):
    def unit(shape):
        x = rng.standard_normal(shape)
        return x / np.linalg.norm(x, axis=-1, keepdims=True)

    q = unit((B, Hk, S, Dk))
    k = unit((B, Hk, S, Dk))
    v = rng.standard_normal((B, Hv, S, Dv))
    g = rng.uniform(g_lo, g_hi, (B, Hv, S))
    beta = 1.0 / (1.0 + np.exp(-rng.standard_normal((B, Hv, S))))
    st = 0.3 * rng.standard_normal((B, Hv, Dk, Dv)) if state else None
    return q, k, v, g, beta, st


@pytest.mark.parametrize("fname", ["hand_worked_2x2.json", "hand_worked_scalar.json"])
def test_hand_worked_examples(fname):
    """Values derived by hand in the fixture (see its 'derivation' field)."""
    with open(os.path.join(GOLDEN, fname)) as f:
        d = json.load(f)
    g = np.log(np.array(d["a"], dtype=np.float64))
    out, st = oracle.recurrence(np.array(d["q"]), np.array(d["k"]), np.array(d["v"]), g,
                                np.array(d["beta"]), d["scale"], np.array(d["state_in"]))
    np.testing.assert_allclose(out, np.array(d["out"]), rtol=0, atol=1e-12)
    np.testing.assert_allclose(st, np.array(d["state_out"]), rtol=0, atol=1e-12)


def test_beta_zero_is_pure_decay():
    """beta = 0: no update, so S_T = exp(sum g) S0 and o_t = scale exp(G_t) S0^T q_t."""
    rng = np.random.default_rng(1)
    q, k, v, g, beta, st0 = _rand_inputs(rng)
    beta = np.zeros_like(beta)
    scale = 0.37
    out, st = oracle.recurrence(q, k, v, g, beta, scale, st0)
    B, Hk, S, Dk = q.shape
    Hv = v.shape[1]
    G = Hv // Hk
    for b in range(B):
        for h in range(Hv):
            Gcum = np.cumsum(g[b, h])
            np.testing.assert_allclose(st[b, h], np.exp(Gcum[-1]) * st0[b, h], rtol=1e-12, atol=1e-14)
            expect = scale * np.exp(Gcum)[:, None] * (q[b, h // G] @ st0[b, h])
            np.testing.assert_allclose(out[b, h], expect, rtol=1e-11, atol=1e-13)


def test_writes_value_into_orthonormal_key_direction():
    """g = 0, beta = 1, orthonormal keys, zero start: S = sum_i k_i v_i^T, and
    querying with q_t = k_t returns exactly scale * v_t (the output reads the
    post-update state; the pre-update state would give 0 at t = 0)."""
    rng = np.random.default_rng(2)
    Dk, Dv, n = 7, 4, 6
    Qm, _ = np.linalg.qr(rng.standard_normal((Dk, Dk)))
    keys = Qm[:, :n].T  # n orthonormal rows
    k = keys[None, None]
    q = k.copy()
    v = rng.standard_normal((1, 1, n, Dv))
    g = np.zeros((1, 1, n))
    beta = np.ones((1, 1, n))
    scale = 0.5
    out, st = oracle.recurrence(q, k, v, g, beta, scale, None)
    np.testing.assert_allclose(st[0, 0], keys.T @ v[0, 0], atol=1e-12)
    np.testing.assert_allclose(out[0, 0], scale * v[0, 0], atol=1e-12)


def test_delta_rule_correction_per_step():
    """For a unit key: S_t^T k_t = exp(g)(1 - beta) S_{t-1}^T k_t + beta v_t."""
    rng = np.random.default_rng(3)
    Dk, Dv = 6, 5
    for trial in range(5):
        q, k, v, g, beta, st0 = _rand_inputs(rng, B=1, Hk=1, Hv=1, S=1, Dk=Dk, Dv=Dv)
        _, st = oracle.recurrence(q, k, v, g, beta, 1.0, st0)
        kt = k[0, 0, 0]
        lhs = st[0, 0].T @ kt
        rhs = np.exp(g[0, 0, 0]) * (1 - beta[0, 0, 0]) * (st0[0, 0].T @ kt) + beta[0, 0, 0] * v[0, 0, 0]
        np.testing.assert_allclose(lhs, rhs, rtol=1e-12, atol=1e-13)


@pytest.mark.parametrize("chunk", [4, 16, 64])
@pytest.mark.parametrize("with_state", [False, True])
def test_chunked_equals_sequential(chunk, with_state):
    """The chunk algebra the GPU kernels use reproduces the per-token recurrence
    (S = 150 leaves a ragged last chunk for every chunk size)."""
    rng = np.random.default_rng(4 + chunk)
    q, k, v, g, beta, st0 = _rand_inputs(rng, B=1, Hk=2, Hv=4, S=150, Dk=8, Dv=6, state=with_state,
                                         g_lo=-2.0, g_hi=-0.001)
    o1, s1 = oracle.recurrence(q, k, v, g, beta, 0.25, st0)
    o2, s2 = oracle.chunked(q, k, v, g, beta, 0.25, st0, chunk=chunk)
    np.testing.assert_allclose(o2, o1, rtol=1e-9, atol=1e-11)
    np.testing.assert_allclose(s2, s1, rtol=1e-9, atol=1e-11)


def test_two_halves_chained_equal_one_pass():
    """The in/out state carries the sequence: two halves chained through it give
    the same final state and outputs as one pass (Parameters / recurrent_state)."""
    rng = np.random.default_rng(5)
    q, k, v, g, beta, st0 = _rand_inputs(rng, S=40)
    o, s = oracle.recurrence(q, k, v, g, beta, 0.3, st0)
    m = 17
    oa, sa = oracle.recurrence(q[:, :, :m], k[:, :, :m], v[:, :, :m], g[:, :, :m], beta[:, :, :m], 0.3, st0)
    ob, sb = oracle.recurrence(q[:, :, m:], k[:, :, m:], v[:, :, m:], g[:, :, m:], beta[:, :, m:], 0.3, sa)
    np.testing.assert_allclose(np.concatenate([oa, ob], axis=2), o, rtol=1e-12, atol=1e-13)
    np.testing.assert_allclose(sb, s, rtol=1e-12, atol=1e-13)


def test_gqa_mapping_is_blocked_not_modulo():
    """Value head h reads key/query head h // (Hv // Hk) (Notes): the result equals
    the run with q, k expanded by repeat_interleave, and differs from the tiled
    (modulo) expansion."""
    rng = np.random.default_rng(6)
    q, k, v, g, beta, st0 = _rand_inputs(rng, B=2, Hk=2, Hv=6, S=9)
    grp = 3
    o, s = oracle.recurrence(q, k, v, g, beta, 0.5, st0)
    qi, ki = np.repeat(q, grp, axis=1), np.repeat(k, grp, axis=1)
    o2, s2 = oracle.recurrence(qi, ki, v, g, beta, 0.5, st0)
    np.testing.assert_allclose(o2, o, rtol=1e-13, atol=1e-14)
    np.testing.assert_allclose(s2, s, rtol=1e-13, atol=1e-14)
    qt, kt = np.tile(q, (1, grp, 1, 1)), np.tile(k, (1, grp, 1, 1))
    o3, _ = oracle.recurrence(qt, kt, v, g, beta, 0.5, st0)
    assert np.abs(o3 - o).max() > 1e-3


def test_linear_in_v_and_scale():
    """With a zero start the update is linear in v (every term carries one factor
    of v), and the output is proportional to scale."""
    rng = np.random.default_rng(7)
    q, k, v, g, beta, _ = _rand_inputs(rng, state=False)
    v2 = rng.standard_normal(v.shape)
    o1, s1 = oracle.recurrence(q, k, v, g, beta, 1.0, None)
    o2, s2 = oracle.recurrence(q, k, v2, g, beta, 1.0, None)
    o3, s3 = oracle.recurrence(q, k, 2.0 * v - 3.0 * v2, g, beta, 1.0, None)
    np.testing.assert_allclose(o3, 2.0 * o1 - 3.0 * o2, rtol=1e-10, atol=1e-12)
    np.testing.assert_allclose(s3, 2.0 * s1 - 3.0 * s2, rtol=1e-10, atol=1e-12)
    o4, s4 = oracle.recurrence(q, k, v, g, beta, 0.125, None)
    np.testing.assert_allclose(o4, 0.125 * o1, rtol=1e-13, atol=1e-15)
    np.testing.assert_allclose(s4, s1, rtol=0, atol=0)


def test_zero_start_equals_explicit_zero_state():
    """The omitted state is a zero start (Parameters / recurrent_state)."""
    rng = np.random.default_rng(8)
    q, k, v, g, beta, st0 = _rand_inputs(rng)
    o1, s1 = oracle.recurrence(q, k, v, g, beta, 0.7, None)
    o2, s2 = oracle.recurrence(q, k, v, g, beta, 0.7, np.zeros_like(st0))
    np.testing.assert_array_equal(o1, o2)
    np.testing.assert_array_equal(s1, s2)


def test_empty_sequence_keeps_state():
    rng = np.random.default_rng(9)
    q, k, v, g, beta, st0 = _rand_inputs(rng, S=0)
    o, s = oracle.recurrence(q, k, v, g, beta, 0.7, st0)
    assert o.shape == (2, 4, 0, 3)
    np.testing.assert_array_equal(s, st0)


@pytest.mark.parametrize("g_range", [(-0.5, -0.005), (-1e-4, 0.0)])
def test_final_state_is_affine_in_the_start_state(g_range):
    """The fact the split prefill rests on: over a segment, the final state is M S0 + X, with X
    the final state from a zero start and M the final state from S0 = I with v = 0 (Dk = Dv),
    for any S0; and the outputs likewise split into a part linear in S0 and the zero-start
    part.  Checked against the recurrence from random start states, including almost no decay
    (where M is far from zero)."""
    rng = np.random.default_rng(23)
    D = 6
    q, k, v, g, beta, _ = _rand_inputs(rng, B=1, Hk=1, Hv=2, S=29, Dk=D, Dv=D, state=False,
                                       g_lo=g_range[0], g_hi=g_range[1])
    _, X = oracle.recurrence(q, k, v, g, beta, 1.0, None)
    eye = np.broadcast_to(np.eye(D), (1, 2, D, D)).copy()
    _, M = oracle.recurrence(q, k, np.zeros_like(v), g, beta, 1.0, eye)
    o0, _ = oracle.recurrence(q, k, v, g, beta, 1.0, None)
    oM, _ = oracle.recurrence(q, k, np.zeros_like(v), g, beta, 1.0, eye)
    assert np.abs(M).max() > 1e-5  # the map is not trivially zero over 29 tokens
    for _ in range(3):
        S0 = rng.standard_normal((1, 2, D, D))
        o, S = oracle.recurrence(q, k, v, g, beta, 1.0, S0)
        np.testing.assert_allclose(S, np.einsum("bhij,bhjk->bhik", M, S0) + X, rtol=1e-10, atol=1e-12)
        # out_t = (M_t S0)^T q_t + out_t(zero start); with v = 0 from I the output is (M_t)^T q_t
        np.testing.assert_allclose(o, np.einsum("bhtj,bhjk->bhtk", oM, S0) + o0, rtol=1e-10, atol=1e-12)
