"""ctypes binding of ``libgdn.so`` (declared in ``include/gdn.h``).

Argument marshalling only: every step of the computation runs in the library's
CUDA kernels.  Tensors are PyTorch CUDA tensors (PyTorch supplies device memory
and streams); the library is called on the current torch stream.  If the
shared library is missing the binding raises instead of falling back to
anything else.
"""
from __future__ import annotations

import ctypes
import os

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "libgdn.so")

GDN_OK = 0
GDN_ERR_NULL = 1
GDN_ERR_DIMS = 2
GDN_ERR_UNSUPPORTED = 3
GDN_ERR_ALIGN = 4
GDN_ERR_CUDA = 5
GDN_ERR_TIMEOUT = 6
GDN_ERR_WORKSPACE = 7

GDN_F32 = 0
GDN_BF16 = 1

GDN_ZERO_INITIAL_STATE = 1 << 0
GDN_FORCE_FFMA = 1 << 1
GDN_SINGLE_PASS = 1 << 2

# Every symbol include/gdn.h declares.
EXPORTED = ("gdn_prefill", "gdn_decode_step", "gdn_prefill_workspace_bytes", "gdn_status_string",
            "gdn_device_status", "gdn_kernels_per_call", "gdn_conv1d_prefill", "gdn_conv1d_decode",
            "gdn_decode_gated", "gdn_decode_block_workspace_bytes", "gdn_decode_block", "gdn_rmsnorm_gated",
            "gdn_prefill_gated", "gdn_prefill_segments", "gdn_decode_block_noalloc",
            "gdn_set_wait_limit_ns", "gdn_test_stall_prefill", "gdn_prefill_ws", "gdn_prefill_segment_starts")


class GdnDims(ctypes.Structure):
    _fields_ = [("B", ctypes.c_int64), ("Hk", ctypes.c_int64), ("Hv", ctypes.c_int64), ("S", ctypes.c_int64),
                ("Dk", ctypes.c_int64), ("Dv", ctypes.c_int64), ("dtype", ctypes.c_int32),
                ("flags", ctypes.c_uint32)]


class GdnConvDims(ctypes.Structure):
    _fields_ = [("B", ctypes.c_int64), ("C", ctypes.c_int64), ("T", ctypes.c_int64), ("K", ctypes.c_int64),
                ("dtype", ctypes.c_int32), ("flags", ctypes.c_uint32)]


class GdnBlockDims(ctypes.Structure):
    _fields_ = [("B", ctypes.c_int64), ("H", ctypes.c_int64), ("Hk", ctypes.c_int64), ("Hv", ctypes.c_int64),
                ("Dk", ctypes.c_int64), ("Dv", ctypes.c_int64), ("K", ctypes.c_int64), ("dtype", ctypes.c_int32),
                ("flags", ctypes.c_uint32)]


class GdnError(RuntimeError):
    def __init__(self, code: int, msg: str):
        super().__init__(msg)
        self.code = code


_lib = None


def lib() -> ctypes.CDLL:
    """Load ``libgdn.so`` (raises if it has not been built)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError("libgdn.so is not built (%s); run __graft_entry__.build() or "
                               "python gated_delta_rule_20_gb300/build.py" % LIB_PATH)
        L = ctypes.CDLL(LIB_PATH)
        vp, fp = ctypes.c_void_p, ctypes.c_void_p
        sig = [vp, vp, vp, fp, fp, ctypes.c_float, fp, vp, ctypes.POINTER(GdnDims), vp]
        for name in ("gdn_prefill", "gdn_decode_step"):
            f = getattr(L, name)
            f.restype = ctypes.c_int
            f.argtypes = sig
        L.gdn_prefill_ws.restype = ctypes.c_int
        L.gdn_prefill_ws.argtypes = sig[:-1] + [vp, ctypes.c_size_t, vp]
        L.gdn_prefill_workspace_bytes.restype = ctypes.c_size_t
        L.gdn_prefill_workspace_bytes.argtypes = [ctypes.POINTER(GdnDims)]
        L.gdn_status_string.restype = ctypes.c_char_p
        L.gdn_status_string.argtypes = [ctypes.c_int]
        L.gdn_device_status.restype = ctypes.c_int
        L.gdn_device_status.argtypes = [ctypes.c_int, ctypes.c_int, ctypes.POINTER(ctypes.c_int32)]
        L.gdn_set_wait_limit_ns.restype = ctypes.c_int
        L.gdn_set_wait_limit_ns.argtypes = [ctypes.c_int, ctypes.c_uint64]
        L.gdn_test_stall_prefill.restype = ctypes.c_int
        L.gdn_test_stall_prefill.argtypes = [ctypes.c_int, ctypes.c_int]
        L.gdn_kernels_per_call.restype = ctypes.c_int
        L.gdn_kernels_per_call.argtypes = []
        L.gdn_prefill_segments.restype = ctypes.c_int32
        L.gdn_prefill_segments.argtypes = [ctypes.POINTER(GdnDims), ctypes.c_int32]
        L.gdn_prefill_segment_starts.restype = ctypes.c_int32
        L.gdn_prefill_segment_starts.argtypes = [ctypes.POINTER(GdnDims), ctypes.c_int32,
                                                 ctypes.POINTER(ctypes.c_int64), ctypes.c_int32]
        L.gdn_decode_gated.restype = ctypes.c_int
        L.gdn_decode_gated.argtypes = [vp, vp, vp, vp, fp, fp, fp, ctypes.c_float, fp, vp, ctypes.POINTER(GdnDims),
                                       vp]
        L.gdn_decode_block_workspace_bytes.restype = ctypes.c_size_t
        L.gdn_decode_block_workspace_bytes.argtypes = [ctypes.POINTER(GdnBlockDims)]
        L.gdn_decode_block.restype = ctypes.c_int
        L.gdn_decode_block.argtypes = [vp, vp, vp, vp, vp, fp, vp, fp, fp, fp, fp, vp, vp, ctypes.c_size_t,
                                       ctypes.POINTER(GdnBlockDims), vp]
        L.gdn_decode_block_noalloc.restype = ctypes.c_int
        L.gdn_decode_block_noalloc.argtypes = [vp, vp, vp, vp, vp, fp, vp, fp, fp, fp, fp, vp,
                                               ctypes.POINTER(GdnBlockDims), vp]
        for name in ("gdn_conv1d_prefill", "gdn_conv1d_decode"):
            f = getattr(L, name)
            f.restype = ctypes.c_int
            f.argtypes = [vp, fp, vp, vp, ctypes.POINTER(GdnConvDims), vp]
        L.gdn_rmsnorm_gated.restype = ctypes.c_int
        L.gdn_rmsnorm_gated.argtypes = [vp, vp, fp, vp, ctypes.c_int64, ctypes.c_int64, ctypes.c_int32, vp]
        L.gdn_prefill_gated.restype = ctypes.c_int
        L.gdn_prefill_gated.argtypes = [vp, vp, vp, fp, fp, vp, fp, ctypes.c_float, fp, vp, ctypes.POINTER(GdnDims),
                                        vp]
        _lib = L
    return _lib


def set_wait_limit_ns(device: int, ns: int) -> None:
    """``gdn_set_wait_limit_ns``: the give-up time of the tensor-core prefill's waits on ``device``
    (0 restores the default second).  Meant for exercising the timeout path."""
    _check(lib().gdn_set_wait_limit_ns(int(device), int(ns)))


def test_stall_prefill(device: int, on: bool) -> None:
    """``gdn_test_stall_prefill``: while on, each tensor-core prefill CTA waits on a barrier that is
    never arrived at, so that its wait runs out (a test of the give-up path)."""
    _check(lib().gdn_test_stall_prefill(int(device), 1 if on else 0))


def status_string(code: int) -> str:
    return lib().gdn_status_string(int(code)).decode()


def make_dims(B, Hk, Hv, S, Dk, Dv, dtype, flags=0) -> GdnDims:
    return GdnDims(int(B), int(Hk), int(Hv), int(S), int(Dk), int(Dv), int(dtype), int(flags))


def _check(code: int):
    if code != GDN_OK:
        raise GdnError(code, status_string(code))


def _torch():
    import torch
    return torch


def _dtype_code(t) -> int:
    torch = _torch()
    if t.dtype == torch.bfloat16:
        return GDN_BF16
    if t.dtype == torch.float32:
        return GDN_F32
    raise TypeError("q/k/v must be bfloat16 or float32, got %s" % t.dtype)


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _call(name, q, k, v, g_log, beta, scale, state, out, zero_initial_state, force_ffma, stream, single_pass=False,
          workspace=None):
    torch = _torch()
    for nm, t in (("q", q), ("k", k), ("v", v), ("g_log", g_log), ("beta", beta), ("state", state), ("out", out)):
        if not t.is_cuda:
            raise ValueError("%s must be a CUDA tensor" % nm)
        if not t.is_contiguous():
            raise ValueError("%s must be contiguous" % nm)
    if g_log.dtype != torch.float32 or beta.dtype != torch.float32 or state.dtype != torch.float32:
        raise TypeError("g_log, beta and state must be float32")
    dt = _dtype_code(q)
    if k.dtype != q.dtype or v.dtype != q.dtype or out.dtype != q.dtype:
        raise TypeError("q, k, v and out must share the compute dtype")
    if q.dim() != 4 or v.dim() != 4:
        raise ValueError("q/k must be [B,Hk,S,Dk] and v [B,Hv,S,Dv]")
    B, Hk, S, Dk = q.shape
    Hv, Dv = v.shape[1], v.shape[3]
    if tuple(k.shape) != tuple(q.shape) or tuple(v.shape[:3]) != (B, Hv, S) or \
            tuple(g_log.shape) != (B, Hv, S) or tuple(beta.shape) != (B, Hv, S) or \
            tuple(state.shape) != (B, Hv, Dk, Dv) or tuple(out.shape) != (B, Hv, S, Dv):
        raise ValueError("inconsistent shapes")
    flags = (GDN_ZERO_INITIAL_STATE if zero_initial_state else 0) | (GDN_FORCE_FFMA if force_ffma else 0) | \
        (GDN_SINGLE_PASS if single_pass else 0)
    dims = make_dims(B, Hk, Hv, S, Dk, Dv, dt, flags)
    if stream is None:
        stream = torch.cuda.current_stream(q.device)
    args = [_ptr(q), _ptr(k), _ptr(v), _ptr(g_log), _ptr(beta), ctypes.c_float(scale), _ptr(state), _ptr(out),
            ctypes.byref(dims)]
    if workspace is not None:  # gdn_prefill_ws: a device buffer of workspace.numel() bytes
        if not workspace.is_cuda or workspace.dtype != torch.uint8 or not workspace.is_contiguous():
            raise ValueError("workspace must be a contiguous uint8 CUDA tensor")
        name = "gdn_prefill_ws"
        args += [_ptr(workspace), ctypes.c_size_t(workspace.numel())]
    with torch.cuda.device(q.device):
        code = getattr(lib(), name)(*args, ctypes.c_void_p(stream.cuda_stream))
    _check(code)
    return out, state


def prefill(q, k, v, g_log, beta, scale, state=None, out=None, *, force_ffma=False, single_pass=False, stream=None,
            workspace=None):
    """Chunked prefill (``gdn_prefill``).

    ``state`` [B,Hv,Dk,Dv] fp32 is updated in place and returned; ``None`` means
    the zero-start form (a new zero-initialised tensor receives the final
    state).  ``single_pass`` sets ``GDN_SINGLE_PASS`` (no split into segments).
    ``workspace``: a uint8 CUDA tensor of at least ``prefill_workspace_bytes``
    bytes for a split's scratch (``gdn_prefill_ws``), so that the call allocates
    nothing.  Returns ``(out, state)``.
    """
    torch = _torch()
    B, Hk, S, Dk = q.shape
    Hv, Dv = v.shape[1], v.shape[3]
    zero = state is None
    if zero:
        state = torch.empty((B, Hv, Dk, Dv), dtype=torch.float32, device=q.device)
    if out is None:
        out = torch.empty((B, Hv, S, Dv), dtype=q.dtype, device=q.device)
    return _call("gdn_prefill", q, k, v, g_log, beta, scale, state, out, zero, force_ffma, stream, single_pass,
                 workspace)


def prefill_workspace_bytes(B, Hk, Hv, S, Dk, Dv, dtype=GDN_BF16, *, force_ffma=False, single_pass=False) -> int:
    """``gdn_prefill_workspace_bytes`` on the current CUDA device (0 for one pass or without a device)."""
    flags = (GDN_FORCE_FFMA if force_ffma else 0) | (GDN_SINGLE_PASS if single_pass else 0)
    return int(lib().gdn_prefill_workspace_bytes(ctypes.byref(make_dims(B, Hk, Hv, S, Dk, Dv, dtype, flags))))


def rmsnorm_gated(x, z, norm_weight, out=None, *, stream=None):
    """RMSNormGated over the last dimension (``gdn_rmsnorm_gated``): x, z [..., D] in the compute
    dtype, norm_weight [D] fp32; ``out`` may be ``x``.  Returns ``out``."""
    torch = _torch()
    if out is None:
        out = torch.empty_like(x)
    for nm, t in (("x", x), ("z", z), ("norm_weight", norm_weight), ("out", out)):
        if not t.is_cuda or not t.is_contiguous():
            raise ValueError("%s must be a contiguous CUDA tensor" % nm)
    if z.shape != x.shape or out.shape != x.shape or z.dtype != x.dtype or out.dtype != x.dtype:
        raise ValueError("x, z and out must share shape and dtype")
    if norm_weight.dtype != torch.float32 or norm_weight.shape != (x.shape[-1],):
        raise ValueError("norm_weight must be float32 [D]")
    D = x.shape[-1]
    rows = x.numel() // D if D else 0
    if stream is None:
        stream = torch.cuda.current_stream(x.device)
    with torch.cuda.device(x.device):
        _check(lib().gdn_rmsnorm_gated(_ptr(x), _ptr(z), _ptr(norm_weight), _ptr(out), rows, D, _dtype_code(x),
                                       ctypes.c_void_p(stream.cuda_stream)))
    return out


def prefill_gated(q, k, v, g_log, beta, z, norm_weight, scale, state=None, out=None, *, force_ffma=False,
                  stream=None):
    """``gdn_prefill_gated``: the prefill with RMSNormGated on its output, z [B,Hv,S,Dv] in the
    compute dtype, norm_weight [Dv] fp32.  Returns ``(out, state)`` as ``prefill``."""
    torch = _torch()
    B, Hk, S, Dk = q.shape
    Hv, Dv = v.shape[1], v.shape[3]
    zero = state is None
    if zero:
        state = torch.empty((B, Hv, Dk, Dv), dtype=torch.float32, device=q.device)
    if out is None:
        out = torch.empty((B, Hv, S, Dv), dtype=q.dtype, device=q.device)
    for nm, t in (("q", q), ("k", k), ("v", v), ("g_log", g_log), ("beta", beta), ("z", z),
                  ("norm_weight", norm_weight), ("state", state), ("out", out)):
        if not t.is_cuda or not t.is_contiguous():
            raise ValueError("%s must be a contiguous CUDA tensor" % nm)
    if z.dtype != q.dtype or tuple(z.shape) != (B, Hv, S, Dv):
        raise ValueError("z must be [B,Hv,S,Dv] in the compute dtype")
    if norm_weight.dtype != torch.float32 or tuple(norm_weight.shape) != (Dv,):
        raise ValueError("norm_weight must be float32 [Dv]")
    flags = (GDN_ZERO_INITIAL_STATE if zero else 0) | (GDN_FORCE_FFMA if force_ffma else 0)
    dims = make_dims(B, Hk, Hv, S, Dk, Dv, _dtype_code(q), flags)
    if stream is None:
        stream = torch.cuda.current_stream(q.device)
    with torch.cuda.device(q.device):
        _check(lib().gdn_prefill_gated(_ptr(q), _ptr(k), _ptr(v), _ptr(g_log), _ptr(beta), _ptr(z),
                                       _ptr(norm_weight), ctypes.c_float(scale), _ptr(state), _ptr(out),
                                       ctypes.byref(dims), ctypes.c_void_p(stream.cuda_stream)))
    return out, state


def decode_step(q, k, v, g_log, beta, scale, state, out=None, *, stream=None):
    """One token (``gdn_decode_step``): q, k [B,Hk,1,Dk], v [B,Hv,1,Dv],
    g_log / beta [B,Hv,1]; ``state`` is updated in place.  Returns ``(out, state)``."""
    torch = _torch()
    if out is None:
        out = torch.empty(v.shape, dtype=q.dtype, device=q.device)
    return _call("gdn_decode_step", q, k, v, g_log, beta, scale, state, out, False, False, stream)


def device_status(device: int = 0, clear: bool = True) -> int:
    """Kernel-side status word of ``device`` (0 = no kernel reported a problem)."""
    code = ctypes.c_int32(0)
    _check(lib().gdn_device_status(int(device), 1 if clear else 0, ctypes.byref(code)))
    return int(code.value)


def kernels_per_call() -> int:
    return int(lib().gdn_kernels_per_call())


def prefill_segments(B, Hk, Hv, S, Dk=128, Dv=128, dtype=GDN_BF16, sm_count=None, *, single_pass=False,
                     force_ffma=False) -> int:
    """``gdn_prefill_segments``: the segments gdn_prefill splits each sequence into (1: one
    pass) on a device with ``sm_count`` SMs (default: the current CUDA device's)."""
    if sm_count is None:
        sm_count = _torch().cuda.get_device_properties(_torch().cuda.current_device()).multi_processor_count
    flags = (GDN_FORCE_FFMA if force_ffma else 0) | (GDN_SINGLE_PASS if single_pass else 0)
    d = make_dims(B, Hk, Hv, S, Dk, Dv, dtype, flags)
    return int(lib().gdn_prefill_segments(ctypes.byref(d), int(sm_count)))


def prefill_segment_starts(B, Hk, Hv, S, Dk=128, Dv=128, dtype=GDN_BF16, sm_count=None, *, single_pass=False,
                           force_ffma=False) -> list:
    """``gdn_prefill_segment_starts``: the first token of every segment of gdn_prefill's split,
    then S (``[0, S]`` for one pass); ``[]`` for invalid dims."""
    if sm_count is None:
        sm_count = _torch().cuda.get_device_properties(_torch().cuda.current_device()).multi_processor_count
    flags = (GDN_FORCE_FFMA if force_ffma else 0) | (GDN_SINGLE_PASS if single_pass else 0)
    d = make_dims(B, Hk, Hv, S, Dk, Dv, dtype, flags)
    buf = (ctypes.c_int64 * 17)()
    P = int(lib().gdn_prefill_segment_starts(ctypes.byref(d), int(sm_count), buf, 17))
    return [int(buf[j]) for j in range(P + 1)] if P > 0 else []


def _conv_call(name, a, weight, b, c, dims, stream):
    torch = _torch()
    if stream is None:
        stream = torch.cuda.current_stream(weight.device)
    with torch.cuda.device(weight.device):
        code = getattr(lib(), name)(_ptr(a), _ptr(weight), _ptr(b), _ptr(c), ctypes.byref(dims),
                                    ctypes.c_void_p(stream.cuda_stream))
    _check(code)


def _conv_checks(tensors, dtype):
    torch = _torch()
    for nm, t in tensors:
        if not t.is_cuda:
            raise ValueError("%s must be a CUDA tensor" % nm)
        if not t.is_contiguous():
            raise ValueError("%s must be contiguous" % nm)
        if nm == "weight":
            if t.dtype != torch.float32:
                raise TypeError("weight must be float32")
        elif t.dtype != dtype:
            raise TypeError("x, out and conv_state must share the activation dtype")


def conv1d_prefill(x, weight, out=None, conv_state=None, *, stream=None):
    """Depthwise causal conv1d + SiLU over a sequence (``gdn_conv1d_prefill``):
    x [B,C,T] bf16/fp32, weight [C,K] fp32.  Returns ``(out [B,C,T], conv_state [B,C,K])``,
    the new conv_state being the last K raw tokens."""
    torch = _torch()
    B, C, T = x.shape
    K = weight.shape[1]
    if out is None:
        out = torch.empty_like(x)
    if conv_state is None:
        conv_state = torch.empty((B, C, K), dtype=x.dtype, device=x.device)
    _conv_checks((("x", x), ("weight", weight), ("out", out), ("conv_state", conv_state)), x.dtype)
    if tuple(weight.shape) != (C, K) or tuple(out.shape) != (B, C, T) or tuple(conv_state.shape) != (B, C, K):
        raise ValueError("inconsistent shapes")
    dims = GdnConvDims(B, C, T, K, _dtype_code(x), 0)
    _conv_call("gdn_conv1d_prefill", x, weight, out, conv_state, dims, stream)
    return out, conv_state


def conv1d_decode(x, weight, conv_state, out=None, *, stream=None):
    """One token (``gdn_conv1d_decode``): x [B,C,1], weight [C,K] fp32; ``conv_state``
    [B,C,K] is shifted in place.  Returns ``(out [B,C,1], conv_state)``."""
    torch = _torch()
    B, C, T = x.shape
    K = weight.shape[1]
    if out is None:
        out = torch.empty_like(x)
    _conv_checks((("x", x), ("weight", weight), ("out", out), ("conv_state", conv_state)), x.dtype)
    if tuple(weight.shape) != (C, K) or tuple(out.shape) != (B, C, T) or tuple(conv_state.shape) != (B, C, K):
        raise ValueError("inconsistent shapes")
    dims = GdnConvDims(B, C, T, K, _dtype_code(x), 0)
    _conv_call("gdn_conv1d_decode", x, weight, conv_state, out, dims, stream)
    return out, conv_state


def decode_gated(qkv, z, a, b, A_log, dt_bias, norm_weight, scale, state, Hk, Hv, Dk, Dv, out=None, *,
                 zero_initial_state=False, stream=None):
    """The gated single-token step (``gdn_decode_gated``): qkv [B, 2 Hk Dk + Hv Dv], z [B, Hv Dv],
    a, b [B, Hv] in the compute dtype; A_log, dt_bias [Hv], norm_weight [Dv] and ``state``
    [B, Hv, Dk, Dv] fp32 (updated in place).  Returns ``(out [B, Hv Dv], state)``."""
    torch = _torch()
    B = qkv.shape[0]
    if out is None:
        out = torch.empty((B, Hv * Dv), dtype=qkv.dtype, device=qkv.device)
    for nm, t in (("qkv", qkv), ("z", z), ("a", a), ("b", b), ("A_log", A_log), ("dt_bias", dt_bias),
                  ("norm_weight", norm_weight), ("state", state), ("out", out)):
        if not t.is_cuda or not t.is_contiguous():
            raise ValueError("%s must be a contiguous CUDA tensor" % nm)
    for nm, t in (("z", z), ("a", a), ("b", b), ("out", out)):
        if t.dtype != qkv.dtype:
            raise TypeError("%s must share the compute dtype of qkv" % nm)
    for nm, t in (("A_log", A_log), ("dt_bias", dt_bias), ("norm_weight", norm_weight), ("state", state)):
        if t.dtype != torch.float32:
            raise TypeError("%s must be float32" % nm)
    if tuple(qkv.shape) != (B, 2 * Hk * Dk + Hv * Dv) or tuple(z.shape) != (B, Hv * Dv) or \
            tuple(a.shape) != (B, Hv) or tuple(b.shape) != (B, Hv) or tuple(A_log.shape) != (Hv,) or \
            tuple(dt_bias.shape) != (Hv,) or tuple(norm_weight.shape) != (Dv,) or \
            tuple(state.shape) != (B, Hv, Dk, Dv) or tuple(out.shape) != (B, Hv * Dv):
        raise ValueError("inconsistent shapes")
    dims = make_dims(B, Hk, Hv, 1, Dk, Dv, _dtype_code(qkv), GDN_ZERO_INITIAL_STATE if zero_initial_state else 0)
    if stream is None:
        stream = torch.cuda.current_stream(qkv.device)
    with torch.cuda.device(qkv.device):
        code = lib().gdn_decode_gated(_ptr(qkv), _ptr(z), _ptr(a), _ptr(b), _ptr(A_log), _ptr(dt_bias),
                                      _ptr(norm_weight), ctypes.c_float(scale), _ptr(state), _ptr(out),
                                      ctypes.byref(dims), ctypes.c_void_p(stream.cuda_stream))
    _check(code)
    return out, state


def decode_block_workspace_bytes(B, H, Hk, Hv, Dk, Dv, K) -> int:
    return int(lib().gdn_decode_block_workspace_bytes(ctypes.byref(GdnBlockDims(B, H, Hk, Hv, Dk, Dv, K, GDN_BF16, 0))))


def decode_block(hidden, W_qkv, W_z, W_a, W_b, conv_weight, conv_state, A_log, dt_bias, norm_weight, state,
                 Hk, Hv, Dk, Dv, out=None, workspace=None, *, stream=None):
    """One token through the decode block (``gdn_decode_block``): hidden [B, 1, H] bf16, the four
    in_proj weights [H, N] bf16, conv_weight [C, K] fp32; ``conv_state`` [B, C, K] bf16 and ``state``
    [B, Hv, Dk, Dv] fp32 are updated in place.  ``workspace`` (uint8, optional) must hold
    ``decode_block_workspace_bytes`` bytes.  Returns ``(out [B, 1, Hv Dv], conv_state, state)``."""
    torch = _torch()
    B, _, H = hidden.shape
    K = conv_weight.shape[1]
    dims = GdnBlockDims(B, H, Hk, Hv, Dk, Dv, K, _dtype_code(hidden), 0)
    need = int(lib().gdn_decode_block_workspace_bytes(ctypes.byref(dims)))
    if workspace is None:
        workspace = torch.empty(max(need, 16), dtype=torch.uint8, device=hidden.device)
    if out is None:
        out = torch.empty((B, 1, Hv * Dv), dtype=hidden.dtype, device=hidden.device)
    for nm, t in (("hidden", hidden), ("W_qkv", W_qkv), ("W_z", W_z), ("W_a", W_a), ("W_b", W_b),
                  ("conv_weight", conv_weight), ("conv_state", conv_state), ("A_log", A_log), ("dt_bias", dt_bias),
                  ("norm_weight", norm_weight), ("state", state), ("out", out), ("workspace", workspace)):
        if not t.is_cuda or not t.is_contiguous():
            raise ValueError("%s must be a contiguous CUDA tensor" % nm)
    if stream is None:
        stream = torch.cuda.current_stream(hidden.device)
    with torch.cuda.device(hidden.device):
        code = lib().gdn_decode_block(_ptr(hidden), _ptr(W_qkv), _ptr(W_z), _ptr(W_a), _ptr(W_b), _ptr(conv_weight),
                                      _ptr(conv_state), _ptr(A_log), _ptr(dt_bias), _ptr(norm_weight), _ptr(state),
                                      _ptr(out), _ptr(workspace), ctypes.c_size_t(workspace.numel()),
                                      ctypes.byref(dims), ctypes.c_void_p(stream.cuda_stream))
    _check(code)
    return out, conv_state, state


# Bytes of the fixed scratch array gdn_decode_block_noalloc uses (GDN_NOALLOC_SCRATCH_BYTES).
NOALLOC_SCRATCH_BYTES = 4 << 20


def decode_block_noalloc(hidden, W_qkv, W_z, W_a, W_b, conv_weight, conv_state, A_log, dt_bias, norm_weight, state,
                         Hk, Hv, Dk, Dv, out, *, stream=None):
    """``gdn_decode_block_noalloc``: one token through the decode block with the inter-stage
    scratch in the library's fixed array (no workspace, no allocation by the library).
    ``out`` [B, 1, Hv Dv] bf16 is supplied by the caller; ``conv_state`` and ``state`` are
    updated in place.  Calls that may overlap on the GPU must be serialised on one stream."""
    torch = _torch()
    B, _, H = hidden.shape
    K = conv_weight.shape[1]
    dims = GdnBlockDims(B, H, Hk, Hv, Dk, Dv, K, _dtype_code(hidden), 0)
    for nm, t in (("hidden", hidden), ("W_qkv", W_qkv), ("W_z", W_z), ("W_a", W_a), ("W_b", W_b),
                  ("conv_weight", conv_weight), ("conv_state", conv_state), ("A_log", A_log), ("dt_bias", dt_bias),
                  ("norm_weight", norm_weight), ("state", state), ("out", out)):
        if not t.is_cuda or not t.is_contiguous():
            raise ValueError("%s must be a contiguous CUDA tensor" % nm)
    if stream is None:
        stream = torch.cuda.current_stream(hidden.device)
    with torch.cuda.device(hidden.device):
        code = lib().gdn_decode_block_noalloc(_ptr(hidden), _ptr(W_qkv), _ptr(W_z), _ptr(W_a), _ptr(W_b),
                                              _ptr(conv_weight), _ptr(conv_state), _ptr(A_log), _ptr(dt_bias),
                                              _ptr(norm_weight), _ptr(state), _ptr(out), ctypes.byref(dims),
                                              ctypes.c_void_p(stream.cuda_stream))
    _check(code)
    return out, conv_state, state
