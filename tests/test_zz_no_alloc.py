"""gdn_decode_block_noalloc: the decode block for callers that cannot allocate device
memory (a runtime that owns the whole device, a plugin whose host code may not call the
CUDA allocator, a serving loop that may not risk an allocation while it runs).  Its
scratch (z, a, b and the head counter) lives in a fixed array inside the library instead
of a caller's workspace.

The GPU test compares it, through the C ABI, with gdn_decode_block (the workspace form)
on two tokens in a row at the decode-block workload's size: the second call finds the
first call's contents in the shared array and must not depend on them.  The bar is the
decode block's bf16 one, relative L2 <= 1e-2 on out, the conv window and the state.

This file is collected last on purpose, so that a run that stops at the first failure
has run every other test before it."""
import ctypes

import numpy as np
import pytest

torch = pytest.importorskip("torch")

import gated_delta_rule_20_gb300 as gdn  # noqa: E402
import workloads  # noqa: E402
from gated_delta_rule_20_gb300 import _binding  # noqa: E402

BF16_REL_L2 = 1e-2


def test_noalloc_host_checks():
    """Host-side checks only (no GPU): invalid dims, and dims whose scratch exceeds the fixed
    array, are refused before anything touches the device."""
    L = _binding.lib()
    p = ctypes.c_void_p(0x1000)

    def call(d):
        return L.gdn_decode_block_noalloc(p, p, p, p, p, p, p, p, p, p, p, p,
                                          ctypes.byref(d) if d is not None else None, None)

    D = lambda **kw: gdn.GdnBlockDims(kw.get("B", 2), kw.get("H", 128), kw.get("Hk", 2), kw.get("Hv", 8),
                                      kw.get("Dk", 64), kw.get("Dv", 64), kw.get("K", 4),
                                      kw.get("dtype", gdn.GDN_BF16), 0)
    assert call(None) == gdn.GDN_ERR_NULL
    assert call(D(dtype=gdn.GDN_F32)) == gdn.GDN_ERR_UNSUPPORTED
    assert call(D(B=0)) == gdn.GDN_OK
    # B = 256 tokens with value_dim = 64 * 128: z alone is 4 MiB, beyond the fixed array
    big = D(B=256, H=128, Hk=2, Hv=64, Dk=128, Dv=128)
    assert L.gdn_decode_block_workspace_bytes(ctypes.byref(big)) > _binding.NOALLOC_SCRATCH_BYTES
    assert call(big) == gdn.GDN_ERR_UNSUPPORTED
    # the decode-block workload fits
    fits = D(B=64, H=2048, Hk=16, Hv=32, Dk=128, Dv=128)
    assert L.gdn_decode_block_workspace_bytes(ctypes.byref(fits)) <= _binding.NOALLOC_SCRATCH_BYTES


def _rel(a, b):
    a = a.double().cpu().numpy()
    b = b.double().cpu().numpy()
    assert np.isfinite(a).all()
    return float(np.linalg.norm(a - b) / max(np.linalg.norm(b), 1e-30))


@pytest.mark.gpu
def test_noalloc_matches_workspace_form_two_calls():
    w = workloads.DECODE_BLOCK
    x = workloads.make_block_inputs(w, device="cuda")
    gen = torch.Generator(device="cpu").manual_seed(41)
    hiddens = [x["hidden"], torch.randn(x["hidden"].shape, generator=gen).to(torch.bfloat16).cuda()]
    args = lambda h: (h, x["W_qkv"], x["W_z"], x["W_a"], x["W_b"], x["conv_weight"])
    gates = (x["A_log"], x["dt_bias"], x["norm_weight"])
    heads = (w.Hk, w.Hv, w.Dk, w.Dv)

    # the existing entry point, with a workspace the caller allocates
    cst_ref, st_ref = x["conv_state"].clone(), x["state"].clone()
    refs = []
    for h in hiddens:
        o, cst_ref, st_ref = gdn.decode_block(*args(h), cst_ref, *gates, st_ref, *heads)
        refs.append((o.clone(), cst_ref.clone(), st_ref.clone()))

    # the fixed-scratch entry point, two calls in a row on one stream
    cst, st = x["conv_state"].clone(), x["state"].clone()
    out = torch.empty((w.B, 1, w.Hv * w.Dv), dtype=torch.bfloat16, device="cuda")
    for i, h in enumerate(hiddens):
        _binding.decode_block_noalloc(*args(h), cst, *gates, st, *heads, out)
        torch.cuda.synchronize()
        ro, rc, rs = refs[i]
        for what, got, ref in (("out", out, ro), ("conv_state", cst, rc), ("state", st, rs)):
            e = _rel(got, ref)
            assert e <= BF16_REL_L2, "call %d, %s: rel L2 %.3e against gdn_decode_block" % (i, what, e)
    assert gdn.device_status(0) == 0
