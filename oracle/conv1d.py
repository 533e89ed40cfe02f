"""fp64 CPU oracle for the depthwise causal conv1d + SiLU that precedes the GDN
recurrence ("GDN Conv1D Kernel API Reference": gdn_conv1d_prefill,
gdn_conv1d_decode).

TEST INFRASTRUCTURE, NOT PRODUCT CODE: only ``tests/``, ``__graft_entry__.smoke()``
and the CPU-baseline leg of ``bench.py`` may use it.  It shares no code with the
CUDA library.

What the page fixes (Parameters, Returns, Notes of both entry points):
  * ``mixed`` / ``x`` is the raw, pre-convolution input, layout [B, C, T]
    (channels on the middle axis, tokens last); the weights are [C, K],
    depthwise: every channel is an independent K-tap FIR.
  * prefill returns silu(causal_conv1d(mixed)) [B, C, T] and, as the new
    conv_state, the last K raw tokens of ``mixed`` [B, C, K].
  * decode takes the current raw token x [B, C, 1] and the previous window
    conv_state [B, C, K]; the FIR reduces to a K-tap dot product over the
    shifted window, and the new conv_state is that shifted window.

Readings where the page is silent (assumptions, stated here and tested by the pins):
  * tap order is that of a depthwise ``Conv1d`` weight (a cross-correlation):
    weight[c, K - 1] multiplies the current token, weight[c, K - 1 - m] the
    token m steps back;
  * the prefill has no input conv_state, so tokens before the sequence are 0
    (causal left padding), and when T < K the new conv_state is the T tokens
    right-aligned behind K - T zeros;
  * the shifted window is the previous window without its oldest token,
    followed by the current token; silu(z) = z / (1 + exp(-z)).
"""
from __future__ import annotations

import numpy as np


def _f64(x) -> np.ndarray:
    if hasattr(x, "detach"):  # a torch tensor
        x = x.detach().to("cpu").double().numpy()
    return np.asarray(x, dtype=np.float64)


def silu(z):
    """SiLU (the "silu" of both Returns entries): z * sigmoid(z) = z / (1 + e^-z)."""
    z = _f64(z)
    return z / (1.0 + np.exp(-z))


def causal_conv1d(x, w):
    """Pre-activation depthwise causal conv (Notes: depthwise, groups == C).

    x [B, C, T], w [C, K] -> z [B, C, T] with
        z[b, c, t] = sum_{i=0}^{K-1} w[c, i] * x[b, c, t - (K - 1) + i],
    x taken as 0 before t = 0.  One pass per tap over a shifted copy of x.
    """
    x, w = _f64(x), _f64(w)
    B, C, T = x.shape
    K = w.shape[1]
    z = np.zeros((B, C, T))
    for i in range(K):
        shift = K - 1 - i  # tap i reads the token `shift` steps back
        if shift >= T:
            continue
        z[:, :, shift:] += w[None, :, i, None] * x[:, :, : T - shift]
    return z


def last_tokens(x, K: int):
    """New conv_state of the prefill (Returns, second entry): the last K raw
    tokens of x [B, C, T] -> [B, C, K], right-aligned behind zeros if T < K."""
    x = _f64(x)
    B, C, T = x.shape
    state = np.zeros((B, C, K))
    n = min(T, K)
    if n > 0:
        state[:, :, K - n:] = x[:, :, T - n:]
    return state


def conv1d_prefill(mixed, w):
    """gdn_conv1d_prefill: (silu(causal_conv1d(mixed)) [B, C, T], conv_state [B, C, K])."""
    K = _f64(w).shape[1]
    return silu(causal_conv1d(mixed, w)), last_tokens(mixed, K)


def conv1d_decode(x, conv_state, w):
    """gdn_conv1d_decode: one token.  x [B, C, 1], conv_state [B, C, K], w [C, K]
    -> (silu(sum_i w[c, i] hs[b, c, i]) [B, C, 1], hs [B, C, K]) where
    hs = (conv_state without its oldest token, then x) is the shifted window."""
    x, st, w = _f64(x), _f64(conv_state), _f64(w)
    hs = np.concatenate([st[:, :, 1:], x[:, :, :1]], axis=2)
    z = np.sum(w[None, :, :] * hs, axis=2, keepdims=True)
    return silu(z), hs
