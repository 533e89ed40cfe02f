"""fp64 CPU oracle for the whole decode block without its output projection
("GDN Block TKG Kernel API Reference": gdn_block_tkg Parameters, Returns and the
data flow "in_proj matmuls -> gdn_conv1d_decode (conv + silu + slide-window
state) -> split conv_out + GQA-repeat q,k -> gdn_tkg (l2norm/beta/g/RMSNormGated
+ single-token recurrence)").

TEST INFRASTRUCTURE, NOT PRODUCT CODE: only ``tests/``, ``__graft_entry__.smoke()``
and the CPU-baseline leg of ``bench.py`` may use it.  It shares no code with the
CUDA library.

Steps, in the page's order: the four input projections of the token's hidden
state (matrix products, a library primitive here), the conv1d decode step on the
q|k|v channels (``oracle.conv1d``), then the gated single-token step
(``oracle.gated_decode``).  Readings where the page is silent: the weights are
[H, N] (the page: "== nn.Linear.weight.T"), the projections are exact products
(the GPU rounds them to bf16, like every inter-stage activation), and the query
scale is 1 / sqrt(head_k_dim), the page giving no scale argument.
"""
from __future__ import annotations

import math

import numpy as np

from .conv1d import conv1d_decode
from .gated_decode import decode_gated


def _f64(x):
    if hasattr(x, "detach"):
        x = x.detach().to("cpu").double().numpy()
    return np.asarray(x, dtype=np.float64)


def decode_block(hidden, W_qkv, W_z, W_a, W_b, conv_weight, conv_state, A_log, dt_bias, norm_weight, state,
                 Hk, Hv, Dk, Dv):
    """hidden [B, 1, H]; W_qkv [H, 2 Hk Dk + Hv Dv], W_z [H, Hv Dv], W_a, W_b [H, Hv];
    conv_weight [C, K], conv_state [B, C, K]; A_log, dt_bias [Hv]; norm_weight [Dv];
    state [B, Hv, Dk, Dv] (None: zeros).  Returns (y [B, 1, Hv Dv], conv_state', state')."""
    x = _f64(hidden)[:, 0, :]
    qkv = x @ _f64(W_qkv)
    z = x @ _f64(W_z)
    a = x @ _f64(W_a)
    b = x @ _f64(W_b)
    conv_out, conv_state2 = conv1d_decode(qkv[:, :, None], conv_state, conv_weight)
    y, state2 = decode_gated(conv_out[:, :, 0], z, a, b, A_log, dt_bias, norm_weight, 1.0 / math.sqrt(Dk),
                             state, Hk, Hv, Dk, Dv)
    return y[:, None, :], conv_state2, state2
