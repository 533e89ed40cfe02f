"""fp64 CPU oracle for the gated prefill: the recurrence's output for every token
("GDN CTE Kernel API Reference": Returns, the un-normalised head-major output)
followed by the RMSNormGated epilogue per token and value head over Dv ("GDN
Block TKG Kernel API Reference": Returns, "RMSNormGated decode output", and the
norm_weight parameter).

TEST INFRASTRUCTURE, NOT PRODUCT CODE: only ``tests/``, ``__graft_entry__.smoke()``
and the CPU-baseline leg of ``bench.py`` may use it.  It shares no code with the
CUDA library.

Steps: ``oracle.recurrence`` (the pinned per-token recurrence), then
``oracle.gated_decode.rms_norm_gated`` on each token's output.  Reading (an
assumption where the page is silent): the page states the epilogue for the decode
block's single token;
here it is applied to every token of a prefill, with z laid out like the output,
[B, Hv, S, Dv].
"""
from __future__ import annotations

from . import recurrence
from .gated_decode import rms_norm_gated


def prefill_gated(q, k, v, g_log, beta, z, norm_weight, scale, state=None):
    """q, k [B, Hk, S, Dk]; v, z [B, Hv, S, Dv]; g_log, beta [B, Hv, S]; norm_weight [Dv];
    state [B, Hv, Dk, Dv] or None (zeros).  Returns (y [B, Hv, S, Dv], final state), fp64."""
    o, st = recurrence(q, k, v, g_log, beta, scale, state)
    return rms_norm_gated(o, z, norm_weight), st
