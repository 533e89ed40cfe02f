"""Gated delta-rule (GDN) recurrence on NVIDIA GB300 (sm_103a).

``prefill``      chunk-parallel prefill (C ABI: ``gdn_prefill``)
``decode_step``  one-token step (C ABI: ``gdn_decode_step``)
``conv1d_prefill`` / ``conv1d_decode``  the depthwise causal conv1d + SiLU in
                 front of the recurrence (C ABI: ``gdn_conv1d_prefill`` / ``gdn_conv1d_decode``)
``decode_gated`` the gated single-token step of the decode block: L2-normalised
                 q/k, gates from raw inputs, RMSNormGated output (C ABI: ``gdn_decode_gated``)
``decode_block``  one token through the decode block without its output projection:
                 input projections, conv1d decode, gated step (C ABI: ``gdn_decode_block``)
``decode_block_noalloc``  the same block step with its scratch in a fixed array inside the
                 library, for callers that cannot allocate device memory (C ABI:
                 ``gdn_decode_block_noalloc``)
``rmsnorm_gated`` the RMSNormGated output epilogue over rows (C ABI: ``gdn_rmsnorm_gated``)
``prefill_gated`` the prefill with RMSNormGated on every token's output (C ABI: ``gdn_prefill_gated``)

All run hand-written CUDA kernels from the in-tree ``libgdn.so``; build it
with ``gated_delta_rule_20_gb300.build.build()``.  There is no fallback: a
missing library raises.
"""
from ._binding import (EXPORTED, GDN_BF16, GDN_ERR_ALIGN, GDN_ERR_CUDA, GDN_ERR_DIMS, GDN_ERR_NULL,
                       GDN_ERR_TIMEOUT, GDN_ERR_UNSUPPORTED, GDN_ERR_WORKSPACE, GDN_F32, GDN_FORCE_FFMA, GDN_OK, GDN_SINGLE_PASS,
                       GDN_ZERO_INITIAL_STATE, LIB_PATH, GdnBlockDims, GdnConvDims, GdnDims, GdnError, conv1d_decode,
                       conv1d_prefill, decode_block, decode_block_noalloc, decode_block_workspace_bytes, decode_gated, decode_step,
                       device_status, kernels_per_call, lib, make_dims, prefill, prefill_gated, prefill_segment_starts,
                       prefill_segments,
                       prefill_workspace_bytes,
                       rmsnorm_gated,
                       status_string)

__all__ = ["prefill", "prefill_segments", "prefill_segment_starts", "decode_step", "conv1d_prefill", "conv1d_decode", "decode_gated", "decode_block",
           "decode_block_noalloc", "decode_block_workspace_bytes", "prefill_workspace_bytes", "rmsnorm_gated", "prefill_gated", "GdnBlockDims", "GdnConvDims",
           "device_status",
           "kernels_per_call", "lib", "make_dims", "status_string", "GdnDims", "GdnError", "EXPORTED", "LIB_PATH", "GDN_OK", "GDN_ERR_NULL", "GDN_ERR_DIMS",
           "GDN_ERR_UNSUPPORTED", "GDN_ERR_ALIGN", "GDN_ERR_CUDA", "GDN_ERR_TIMEOUT", "GDN_ERR_WORKSPACE", "GDN_F32", "GDN_BF16",
           "GDN_ZERO_INITIAL_STATE", "GDN_FORCE_FFMA", "GDN_SINGLE_PASS"]
