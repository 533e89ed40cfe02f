"""The C-ABI library loads, exports every symbol include/gdn.h declares, and its
host-side argument checks reject bad calls before any launch.  No call here
reaches a kernel, so this file runs without a GPU."""
import ctypes
import os
import re

import pytest
import torch

import gated_delta_rule_20_gb300 as gdn
from gated_delta_rule_20_gb300 import build as gbuild

HEADER = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "include", "gdn.h")


@pytest.fixture(scope="module")
def L():
    gbuild.build()
    return gdn.lib()


def declared_functions():
    src = open(HEADER).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"^\s*(?:const\s+)?[a-z_0-9]+\s*\*?\s*(gdn_[a-z_0-9]+)\s*\(", src, flags=re.M)))


def test_header_declares_the_boundary():
    names = declared_functions()
    assert "gdn_prefill" in names and "gdn_decode_step" in names
    assert set(names) == set(gdn.EXPORTED)


def test_library_exports_every_declared_symbol(L):
    for name in declared_functions():
        assert hasattr(L, name), name


def test_status_strings(L):
    for code in range(8):
        s = gdn.status_string(code)
        assert s.startswith("GDN_"), s
    assert "unknown" in gdn.status_string(99)


def test_workspace_query_without_a_device(L):
    # the split's scratch depends on the device's SM count: with no device to query, 0
    d = gdn.make_dims(1, 16, 32, 32768, 128, 128, gdn.GDN_BF16)
    if not torch.cuda.is_available():
        assert L.gdn_prefill_workspace_bytes(ctypes.byref(d)) == 0
    assert L.gdn_prefill_workspace_bytes(None) == 0
    assert gdn.kernels_per_call() == 1


def test_prefill_ws_argument_checks(L):
    def call(dims, ws, nbytes, state=16):
        p = ctypes.c_void_p(16)
        return L.gdn_prefill_ws(p, p, p, p, p, ctypes.c_float(1.0), ctypes.c_void_p(state), p,
                                ctypes.byref(dims) if dims is not None else None,
                                ctypes.c_void_p(ws) if ws is not None else None, ctypes.c_size_t(nbytes), None)
    good = gdn.make_dims(1, 1, 2, 256, 128, 128, gdn.GDN_BF16)
    assert call(None, 4096, 4096) == gdn.GDN_ERR_NULL
    assert call(gdn.make_dims(1, 2, 3, 256, 128, 128, gdn.GDN_BF16), 4096, 4096) == gdn.GDN_ERR_DIMS
    assert call(good, 4096, 4096, state=None) == gdn.GDN_ERR_NULL
    # a misaligned workspace is refused before anything runs (B = 0 would otherwise be a no-op)
    assert call(gdn.make_dims(0, 1, 2, 256, 128, 128, gdn.GDN_BF16), 4104, 4096) == gdn.GDN_ERR_ALIGN


def _call(L, name, dims, ptr=16, state=16):
    p = ctypes.c_void_p(ptr) if ptr is not None else None
    s = ctypes.c_void_p(state) if state is not None else None
    return getattr(L, name)(p, p, p, p, p, ctypes.c_float(1.0), s, p,
                            ctypes.byref(dims) if dims is not None else None, None)


@pytest.mark.parametrize("name", ["gdn_prefill", "gdn_decode_step"])
def test_argument_checks(L, name):
    S = 1 if name == "gdn_decode_step" else 64
    ok = dict(B=2, Hk=2, Hv=4, S=S, Dk=128, Dv=128, dtype=gdn.GDN_BF16)

    def dims(**kw):
        a = dict(ok)
        a.update(kw)
        return gdn.make_dims(a["B"], a["Hk"], a["Hv"], a["S"], a["Dk"], a["Dv"], a["dtype"], a.get("flags", 0))

    assert _call(L, name, None) == gdn.GDN_ERR_NULL
    assert _call(L, name, dims(), ptr=None) == gdn.GDN_ERR_NULL
    assert _call(L, name, dims(), state=None) == gdn.GDN_ERR_NULL
    assert _call(L, name, dims(Hv=3)) == gdn.GDN_ERR_DIMS          # Hv % Hk != 0
    assert _call(L, name, dims(Dk=129)) == gdn.GDN_ERR_DIMS        # > MAX_HEAD_DIM
    assert _call(L, name, dims(Dv=129)) == gdn.GDN_ERR_DIMS
    assert _call(L, name, dims(Dk=0)) == gdn.GDN_ERR_DIMS
    assert _call(L, name, dims(Hk=0)) == gdn.GDN_ERR_DIMS
    assert _call(L, name, dims(B=-1)) == gdn.GDN_ERR_DIMS
    assert _call(L, name, dims(S=-1)) == gdn.GDN_ERR_DIMS
    assert _call(L, name, dims(dtype=7)) == gdn.GDN_ERR_UNSUPPORTED
    assert _call(L, name, dims(flags=1 << 9)) == gdn.GDN_ERR_UNSUPPORTED
    assert _call(L, name, dims(), ptr=24) == gdn.GDN_ERR_ALIGN       # not 16-byte aligned
    assert _call(L, name, dims(), state=8) == gdn.GDN_ERR_ALIGN
    if name == "gdn_decode_step":
        assert _call(L, name, dims(S=2)) == gdn.GDN_ERR_DIMS


def test_empty_batch_is_a_no_op(L):
    # B = 0: nothing to compute, no CUDA call is made.
    d = gdn.make_dims(0, 2, 4, 64, 128, 128, gdn.GDN_BF16)
    assert _call(L, "gdn_prefill", d) == gdn.GDN_OK
    d = gdn.make_dims(0, 2, 4, 1, 128, 128, gdn.GDN_BF16)
    assert _call(L, "gdn_decode_step", d) == gdn.GDN_OK


def test_prefill_segments():
    """The split rule of gdn_prefill (host only): few long sequences split into 2 .. 16
    segments where the launch model predicts a saving; one pass off the tensor-core path or
    when asked for; 0 for invalid dims."""
    seg = gdn.prefill_segments
    assert seg(1, 16, 32, 32768, sm_count=152) == 6       # the long workload: 32 sequences
    assert seg(4, 16, 32, 4096, sm_count=152) == 1        # 128 sequences: one pass
    assert seg(16, 8, 32, 2048, sm_count=152) == 1        # 512 sequences: one pass
    assert seg(1, 1, 2, 32768, sm_count=152) == 16        # capped by the run table
    assert seg(2, 5, 25, 4096, sm_count=152) == 2         # 50 sequences: 150 CTAs in one wave
    assert seg(2, 5, 25, 1536, sm_count=152) == 1         # 24 chunks: the split's fixed costs outweigh it
    assert seg(1, 1, 1, 256, sm_count=152) == 1           # 4 chunks: too short to pay
    assert seg(1, 1, 2, 32768, dtype=gdn.GDN_F32, sm_count=152) == 1
    assert seg(1, 1, 2, 32768, Dk=64, Dv=64, sm_count=152) == 1
    assert seg(1, 1, 2, 32768, sm_count=152, single_pass=True) == 1
    assert seg(1, 1, 2, 32768, sm_count=152, force_ffma=True) == 1
    assert seg(0, 1, 2, 32768, sm_count=152) == 1 and seg(1, 1, 2, 0, sm_count=152) == 1
    assert seg(1, 2, 3, 4096, sm_count=152) == 0          # Hv % Hk != 0
    assert seg(1, 1, 2, 4096, Dk=129, sm_count=152) == 0
    assert seg(1, 1, 2, 4096, sm_count=0) == 0
    L = gdn.lib()
    assert L.gdn_prefill_segments(None, 152) == 0


def test_prefill_segment_starts():
    """Segment bounds of the split (host only): segment 0 from token 0, segments 1 .. P - 2
    of one multiple of 128 tokens, the last one ending at S (ragged S included); one pass
    gives [0, S]; the count agrees with gdn_prefill_segments on every shape."""
    st = gdn.prefill_segment_starts
    assert st(1, 16, 32, 32768, sm_count=152) == [0, 12928, 16896, 20864, 24832, 28800, 32768]
    assert st(4, 16, 32, 4096, sm_count=152) == [0, 4096]
    assert st(1, 1, 2, 4096, sm_count=152, single_pass=True) == [0, 4096]
    assert st(1, 2, 3, 4096, sm_count=152) == []
    for B, Hk, Hv, S in [(1, 1, 2, 2000), (1, 1, 1, 4608), (2, 2, 8, 3072), (1, 1, 2, 3000), (1, 2, 4, 2500),
                         (2, 5, 25, 4096), (2, 4, 32, 8192), (1, 1, 8, 16385), (1, 1, 64, 32768), (1, 1, 2, 32767)]:
        b = st(B, Hk, Hv, S, sm_count=152)
        assert len(b) - 1 == gdn.prefill_segments(B, Hk, Hv, S, sm_count=152) >= 2
        assert b[0] == 0 and b[-1] == S and all(x < y for x, y in zip(b, b[1:]))
        assert b[1] % 64 == 0
        mids = {y - x for x, y in zip(b[1:-2], b[2:-1])}
        assert len(mids) <= 1 and all(m % 128 == 0 for m in mids)
        if len(b) > 3:
            assert 0 < S - b[-2] <= b[2] - b[1]   # the last segment: at most one middle segment


def test_prefill_split_plans_are_valid():
    """Every plan the split rule returns (host only, many shapes and SM counts) tiles the
    sequence: segment 0 of whole chunks, the middle segments of one length in whole
    128-token tiles, the last one no longer than them and ending at S, at most 16 segments;
    and the same dims ask for the same plan again."""
    import random
    rng = random.Random(5)
    st = gdn.prefill_segment_starts
    for _ in range(300):
        Hk = rng.choice([1, 2, 4, 8, 16])
        Hv = Hk * rng.choice([1, 2, 4])
        B = rng.choice([1, 1, 2, 3, 4])
        S = rng.choice([rng.randint(1, 4096), rng.randint(4096, 70000)])
        sms = rng.choice([132, 148, 152])
        b = st(B, Hk, Hv, S, sm_count=sms)
        P = len(b) - 1
        assert P == gdn.prefill_segments(B, Hk, Hv, S, sm_count=sms) and 1 <= P <= 16
        assert b[0] == 0 and b[-1] == S and all(x < y for x, y in zip(b, b[1:]))
        if P > 1:
            assert b[1] % 64 == 0
            lens = [y - x for x, y in zip(b[1:], b[2:])]
            assert all(m == lens[0] and m % 128 == 0 for m in lens[:-1])
            assert 0 < lens[-1] <= lens[0] if len(lens) > 1 else lens[0] > 0
        assert st(B, Hk, Hv, S, sm_count=sms) == b


def test_prefill_flags_known(L):
    # every documented flag passes validation (B = 0: no CUDA call); the next bit does not
    for f in (gdn.GDN_ZERO_INITIAL_STATE, gdn.GDN_FORCE_FFMA, gdn.GDN_SINGLE_PASS,
              gdn.GDN_ZERO_INITIAL_STATE | gdn.GDN_SINGLE_PASS):
        assert _call(L, "gdn_prefill", gdn.make_dims(0, 2, 4, 64, 128, 128, gdn.GDN_BF16, f)) == gdn.GDN_OK
    assert _call(L, "gdn_prefill", gdn.make_dims(0, 2, 4, 64, 128, 128, gdn.GDN_BF16, 1 << 3)) == \
        gdn.GDN_ERR_UNSUPPORTED


def test_binding_requires_cuda_tensors():
    torch = pytest.importorskip("torch")
    q = torch.zeros(1, 1, 4, 8)
    with pytest.raises(ValueError):
        gdn.prefill(q, q, q, torch.zeros(1, 1, 4), torch.zeros(1, 1, 4), 1.0, torch.zeros(1, 1, 8, 8),
                    torch.zeros(1, 1, 4, 8))


def _conv(L, name, dims, x=0x1000, w=0x2000, st=0x3000, out=0x4000):
    c = lambda v: ctypes.c_void_p(v) if v is not None else None
    if name == "gdn_conv1d_prefill":
        return L.gdn_conv1d_prefill(c(x), c(w), c(out), c(st), ctypes.byref(dims) if dims is not None else None, None)
    return L.gdn_conv1d_decode(c(x), c(w), c(st), c(out), ctypes.byref(dims) if dims is not None else None, None)


@pytest.mark.parametrize("name", ["gdn_conv1d_prefill", "gdn_conv1d_decode"])
def test_conv1d_argument_checks(L, name):
    """Host-side checks of the conv1d entry points (they run before any launch, so
    no GPU is needed): every failure returns its code and launches nothing."""
    D = lambda B=2, C=16, T=1, K=4, dtype=gdn.GDN_BF16, flags=0: gdn.GdnConvDims(B, C, T, K, dtype, flags)
    assert _conv(L, name, None) == gdn.GDN_ERR_NULL
    assert _conv(L, name, D(dtype=7)) == gdn.GDN_ERR_UNSUPPORTED
    assert _conv(L, name, D(flags=1)) == gdn.GDN_ERR_UNSUPPORTED
    assert _conv(L, name, D(K=9)) == gdn.GDN_ERR_UNSUPPORTED
    assert _conv(L, name, D(K=0)) == gdn.GDN_ERR_DIMS
    assert _conv(L, name, D(C=0)) == gdn.GDN_ERR_DIMS
    assert _conv(L, name, D(B=-1)) == gdn.GDN_ERR_DIMS
    assert _conv(L, name, D(), w=None) == gdn.GDN_ERR_NULL
    assert _conv(L, name, D(), st=None) == gdn.GDN_ERR_NULL
    assert _conv(L, name, D(), x=None) == gdn.GDN_ERR_NULL
    assert _conv(L, name, D(), x=0x1001) == gdn.GDN_ERR_ALIGN        # bf16 needs 2-byte alignment
    assert _conv(L, name, D(dtype=gdn.GDN_F32), out=0x4002) == gdn.GDN_ERR_ALIGN
    assert _conv(L, name, D(B=0)) == gdn.GDN_OK                      # nothing to do, nothing launched
    if name == "gdn_conv1d_decode":
        assert _conv(L, name, D(T=2)) == gdn.GDN_ERR_DIMS             # one token only


def test_decode_gated_argument_checks(L):
    """Host-side checks of gdn_decode_gated (no launch happens, so no GPU is needed)."""
    p = ctypes.c_void_p(0x1000)
    call = lambda d, st=p, a=p: L.gdn_decode_gated(p, p, a, p, p, p, p, ctypes.c_float(1.0), st, p,
                                                   ctypes.byref(d) if d is not None else None, None)
    D = lambda **kw: gdn.make_dims(kw.get("B", 2), kw.get("Hk", 2), kw.get("Hv", 4), kw.get("S", 1), kw.get("Dk", 128),
                                   kw.get("Dv", 128), kw.get("dtype", gdn.GDN_BF16), kw.get("flags", 0))
    assert call(None) == gdn.GDN_ERR_NULL
    assert call(D(S=2)) == gdn.GDN_ERR_DIMS
    assert call(D(Dk=129)) == gdn.GDN_ERR_DIMS
    assert call(D(Hv=3)) == gdn.GDN_ERR_DIMS
    assert call(D(dtype=5)) == gdn.GDN_ERR_UNSUPPORTED
    assert call(D(flags=gdn.GDN_FORCE_FFMA)) == gdn.GDN_ERR_UNSUPPORTED
    assert call(D(), st=None) == gdn.GDN_ERR_NULL
    assert call(D(), a=ctypes.c_void_p(0x1001)) == gdn.GDN_ERR_ALIGN
    assert call(D(B=0)) == gdn.GDN_OK


def test_decode_block_argument_checks(L):
    """Host-side checks of gdn_decode_block and its workspace query (no GPU needed)."""
    p = ctypes.c_void_p(0x1000)
    D = lambda **kw: gdn.GdnBlockDims(kw.get("B", 2), kw.get("H", 128), kw.get("Hk", 2), kw.get("Hv", 8),
                                      kw.get("Dk", 64), kw.get("Dv", 64), kw.get("K", 4),
                                      kw.get("dtype", gdn.GDN_BF16), kw.get("flags", 0))
    call = lambda d, ws=1 << 30, hid=p: L.gdn_decode_block(hid, p, p, p, p, p, p, p, p, p, p, p, p, ctypes.c_size_t(ws),
                                                          ctypes.byref(d) if d is not None else None, None)
    assert call(None) == gdn.GDN_ERR_NULL
    assert call(D(dtype=gdn.GDN_F32)) == gdn.GDN_ERR_UNSUPPORTED
    assert call(D(H=100)) == gdn.GDN_ERR_UNSUPPORTED       # H % 64
    assert call(D(B=300)) == gdn.GDN_ERR_UNSUPPORTED       # B > 256
    assert call(D(K=9)) == gdn.GDN_ERR_UNSUPPORTED
    assert call(D(Hv=4)) == gdn.GDN_ERR_UNSUPPORTED        # Hv % 8 (16-byte rows of W_a, W_b)
    assert call(D(Dk=129)) == gdn.GDN_ERR_DIMS
    assert call(D(), ws=16) == gdn.GDN_ERR_DIMS            # workspace too small
    assert call(D(), hid=ctypes.c_void_p(0x1008)) == gdn.GDN_ERR_ALIGN
    assert call(D(B=0)) == gdn.GDN_OK
    need = L.gdn_decode_block_workspace_bytes(ctypes.byref(D(B=64, H=2048, Hk=16, Hv=32, Dk=128, Dv=128)))
    assert need >= 64 * (4096 + 64) * 2   # z, a, b in bf16
    assert L.gdn_decode_block_workspace_bytes(ctypes.byref(D(dtype=gdn.GDN_F32))) == 0


def test_rmsnorm_and_gated_prefill_argument_checks(L):
    """Host-side checks of gdn_rmsnorm_gated and gdn_prefill_gated (no GPU needed)."""
    p = ctypes.c_void_p(0x1000)
    norm = lambda x=p, rows=4, D=128, dtype=gdn.GDN_BF16, w=p: L.gdn_rmsnorm_gated(x, p, w, p, rows, D, dtype, None)
    assert norm(rows=0) == gdn.GDN_OK
    assert norm(dtype=5) == gdn.GDN_ERR_UNSUPPORTED
    assert norm(D=0) == gdn.GDN_ERR_DIMS and norm(rows=-1) == gdn.GDN_ERR_DIMS
    assert norm(x=None) == gdn.GDN_ERR_NULL
    assert norm(x=ctypes.c_void_p(0x1001)) == gdn.GDN_ERR_ALIGN          # a bf16 row off by a byte
    assert norm(w=ctypes.c_void_p(0x1002)) == gdn.GDN_ERR_ALIGN          # fp32 weights
    d = lambda **kw: gdn.make_dims(kw.get("B", 2), 2, 4, kw.get("S", 64), 128, kw.get("Dv", 128), gdn.GDN_BF16)
    gp = lambda dims, z=p, w=p: L.gdn_prefill_gated(p, p, p, p, p, z, w, ctypes.c_float(1.0), p, p,
                                                    ctypes.byref(dims) if dims is not None else None, None)
    assert gp(None) == gdn.GDN_ERR_NULL
    assert gp(d(), z=None) == gdn.GDN_ERR_NULL                             # checked before the prefill launches
    assert gp(d(), w=ctypes.c_void_p(0x1002)) == gdn.GDN_ERR_ALIGN
    assert gp(d(Dv=129)) == gdn.GDN_ERR_DIMS
    assert gp(d(B=0)) == gdn.GDN_OK
