"""fp64 CPU oracle for the gated single-token step: the decode prologue (L2
normalisation of q and k, the decay g and update strength beta from the raw
gate inputs) and the RMSNormGated output epilogue around one token of the
recurrence -- the per-token work of gdn_tkg inside the fused decode block
("GDN Block TKG Kernel API Reference": gdn_block_tkg Parameters A_log,
dt_bias, norm_weight, W_in_z / W_in_a / W_in_b, Returns "RMSNormGated decode
output", and the data flow "split conv_out + GQA-repeat q,k -> gdn_tkg
(l2norm/beta/g/RMSNormGated + single-token recurrence)").

TEST INFRASTRUCTURE, NOT PRODUCT CODE: only ``tests/``, ``__graft_entry__.smoke()``
and the CPU-baseline leg of ``bench.py`` may use it.  It shares no code with the
CUDA library.

The page names these inputs but prints no formulas.  The readings (assumptions,
the plainest ones the names support):
  * q, k: x / sqrt(sum(x^2) + eps_l2) over the head dim, eps_l2 = 1e-6;
  * g = -exp(A_log[h]) * softplus(a[b, h] + dt_bias[h]),  softplus(x) = log(1 + e^x);
  * beta = sigmoid(b[b, h]);
  * the token's output o (the recurrence's, with the query scale) is normalised
    per value head over Dv and gated:
        y = o / sqrt(mean(o^2) + eps_rms) * norm_weight * silu(z),  eps_rms = 1e-6;
  * the post-conv activations arrive packed as q | k | v along the channel axis
    (the page's conv_dim = 2 * key_dim + value_dim), each head-major.
"""
from __future__ import annotations

import numpy as np

from . import recurrence

EPS_L2 = 1e-6
EPS_RMS = 1e-6


def _f64(x):
    if hasattr(x, "detach"):
        x = x.detach().to("cpu").double().numpy()
    return np.asarray(x, dtype=np.float64)


def l2norm(x, eps: float = EPS_L2):
    x = _f64(x)
    return x / np.sqrt(np.sum(x * x, axis=-1, keepdims=True) + eps)


def softplus(x):
    return np.logaddexp(0.0, _f64(x))


def sigmoid(x):
    return 1.0 / (1.0 + np.exp(-_f64(x)))


def silu(x):
    x = _f64(x)
    return x * sigmoid(x)


def gates(a, b, A_log, dt_bias):
    """(g, beta) [B, Hv] from the raw gate inputs a, b [B, Hv] and the per-head A_log, dt_bias [Hv]."""
    a, b, A_log, dt_bias = _f64(a), _f64(b), _f64(A_log), _f64(dt_bias)
    g = -np.exp(A_log)[None, :] * softplus(a + dt_bias[None, :])
    return g, sigmoid(b)


def rms_norm_gated(o, z, norm_weight, eps: float = EPS_RMS):
    """o, z [..., Dv]: o / sqrt(mean(o^2) + eps) * norm_weight * silu(z)."""
    o, z, w = _f64(o), _f64(z), _f64(norm_weight)
    return o / np.sqrt(np.mean(o * o, axis=-1, keepdims=True) + eps) * w * silu(z)


def decode_gated(qkv, z, a, b, A_log, dt_bias, norm_weight, scale, state, Hk, Hv, Dk, Dv):
    """One gated token.  qkv [B, 2 Hk Dk + Hv Dv] (q | k | v), z [B, Hv Dv], a, b [B, Hv],
    A_log, dt_bias [Hv], norm_weight [Dv], state [B, Hv, Dk, Dv] or None (zeros).
    Returns (y [B, Hv Dv], new state [B, Hv, Dk, Dv]), fp64."""
    qkv = _f64(qkv)
    B = qkv.shape[0]
    kd = Hk * Dk
    q = l2norm(qkv[:, :kd].reshape(B, Hk, Dk))
    k = l2norm(qkv[:, kd:2 * kd].reshape(B, Hk, Dk))
    v = qkv[:, 2 * kd:].reshape(B, Hv, Dv)
    g, beta = gates(a, b, A_log, dt_bias)
    o, st = recurrence(q[:, :, None, :], k[:, :, None, :], v[:, :, None, :], g[:, :, None], beta[:, :, None],
                       scale, state)
    y = rms_norm_gated(o[:, :, 0, :], _f64(z).reshape(B, Hv, Dv), norm_weight)
    return y.reshape(B, Hv * Dv), st
