"""fp64 CPU oracle for the gated delta-rule (GDN) recurrence.

TEST INFRASTRUCTURE, NOT PRODUCT CODE.  Only ``tests/``, ``__graft_entry__.smoke()``
and the CPU-baseline leg of ``bench.py`` may import this package.  It shares no
code with the CUDA library (``gated_delta_rule_20_gb300``) and neither imports
the other; both consume the same seeded inputs from ``workloads.py``.

Two functions compute the method:

``recurrence``
    The plain definition: the per-token recurrence in fp64, written out in C
    (``gdn_oracle.c``), one token after another for every (batch, value head).
    This is the oracle every GPU result is compared with.  It follows the
    "GDN CTE Kernel API Reference" page: Parameters (layouts of query/key/value,
    g_log, beta, scale and the optional in/out recurrent_state), Returns
    (head-major, un-normalised output; fp32 final state) and Notes (value head h
    reads key/query head h // (Hv // Hk)).

``chunked``
    The chunk-parallel form of the same recurrence in fp64 numpy, used only to
    pin the chunk algebra that the GPU kernels implement against the plain
    definition (the page's "chunk-parallel form", Background section).  Its
    derivation, for a chunk with start state S0, token decays g_r, G_r = sum of
    g over the chunk up to r, gamma_r = exp(G_r):

        A[r, j] = beta_r exp(G_r - G_j) (k_r . k_j)   for j < r, else 0
        T       = (I + A)^-1
        U       = T diag(beta) V
        W       = T diag(beta * gamma) K
        Delta   = U - W S0                      (row r = the update delta_r)
        O       = scale (diag(gamma) Q S0 + (M o Q K^T) Delta),  M[r, j] = exp(G_r - G_j) for j <= r
        S_end   = gamma_last S0 + (diag(exp(G_last - G)) K)^T Delta

The inverse is taken with ``numpy.linalg.solve`` (a library primitive).
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "gdn_oracle.c")
_SO = os.path.join(_HERE, "_gdn_oracle.so")
_lib_handle = None


def build(force: bool = False) -> str:
    """Compile the C oracle into ``oracle/_gdn_oracle.so`` (plain gcc, OpenMP)."""
    if force or not os.path.exists(_SO) or os.path.getmtime(_SO) < os.path.getmtime(_SRC):
        tmp = _SO + ".tmp.%d" % os.getpid()
        cmd = ["gcc", "-O2", "-fopenmp", "-fPIC", "-shared", "-o", tmp, _SRC, "-lm"]
        subprocess.run(cmd, check=True)
        os.replace(tmp, _SO)
    return _SO


def _lib():
    global _lib_handle
    if _lib_handle is None:
        build()
        lib = ctypes.CDLL(_SO)
        dp = ctypes.POINTER(ctypes.c_double)
        lib.gdn_oracle_recurrence.restype = ctypes.c_int
        lib.gdn_oracle_recurrence.argtypes = [dp, dp, dp, dp, dp, ctypes.c_double, dp] + \
            [ctypes.c_long] * 6 + [dp, dp]
        lib.gdn_oracle_max_threads.restype = ctypes.c_int
        lib.gdn_oracle_set_threads.argtypes = [ctypes.c_int]
        _lib_handle = lib
    return _lib_handle


def _as_f64(x) -> np.ndarray:
    """Exact fp64 copy of an array (numpy or a CPU/GPU torch tensor of any float dtype)."""
    if hasattr(x, "detach"):  # a torch tensor; bf16 widens exactly to fp64
        x = x.detach().to("cpu").double().numpy()
    return np.ascontiguousarray(np.asarray(x, dtype=np.float64))


def _ptr(a: np.ndarray):
    return a.ctypes.data_as(ctypes.POINTER(ctypes.c_double))


def max_threads() -> int:
    return int(_lib().gdn_oracle_max_threads())


def set_threads(n: int) -> None:
    _lib().gdn_oracle_set_threads(int(n))


def recurrence(q, k, v, g_log, beta, scale, state=None):
    """Per-token fp64 recurrence.  Returns ``(out [B,Hv,S,Dv], state [B,Hv,Dk,Dv])``.

    ``state=None`` is the page's "omitted" recurrent_state: a zero start.
    """
    q, k, v = _as_f64(q), _as_f64(k), _as_f64(v)
    g_log, beta = _as_f64(g_log), _as_f64(beta)
    B, Hk, S, Dk = q.shape
    Hv, Dv = v.shape[1], v.shape[3]
    if k.shape != q.shape or v.shape[:3] != (B, Hv, S) or g_log.shape != (B, Hv, S) \
            or beta.shape != (B, Hv, S) or Hv % Hk != 0:
        raise ValueError("inconsistent shapes")
    st_in = None
    if state is not None:
        st_in = _as_f64(state)
        if st_in.shape != (B, Hv, Dk, Dv):
            raise ValueError("state shape")
    out = np.zeros((B, Hv, S, Dv), dtype=np.float64)
    st = np.zeros((B, Hv, Dk, Dv), dtype=np.float64)
    rc = _lib().gdn_oracle_recurrence(
        _ptr(q), _ptr(k), _ptr(v), _ptr(g_log), _ptr(beta), float(scale),
        _ptr(st_in) if st_in is not None else None,
        B, Hk, Hv, S, Dk, Dv, _ptr(out), _ptr(st))
    if rc != 0:
        raise RuntimeError("oracle failed with code %d" % rc)
    return out, st


def chunked(q, k, v, g_log, beta, scale, state=None, chunk: int = 16):
    """Chunk-parallel fp64 form (see the module docstring).  A last chunk shorter
    than ``chunk`` is processed at its own length."""
    q, k, v = _as_f64(q), _as_f64(k), _as_f64(v)
    g_log, beta = _as_f64(g_log), _as_f64(beta)
    B, Hk, S, Dk = q.shape
    Hv, Dv = v.shape[1], v.shape[3]
    grp = Hv // Hk
    out = np.zeros((B, Hv, S, Dv))
    st = np.zeros((B, Hv, Dk, Dv)) if state is None else _as_f64(state).copy()
    for b in range(B):
        for h in range(Hv):
            S0 = st[b, h]
            for c0 in range(0, S, chunk):
                sl = slice(c0, min(c0 + chunk, S))
                K, Q, V = k[b, h // grp, sl], q[b, h // grp, sl], v[b, h, sl]
                gg, bb = g_log[b, h, sl], beta[b, h, sl]
                n = K.shape[0]
                Gc = np.cumsum(gg)
                gamma = np.exp(Gc)
                lower = np.tril(np.ones((n, n), dtype=bool))
                strict = np.tril(np.ones((n, n), dtype=bool), -1)
                decay = np.exp(np.where(lower, Gc[:, None] - Gc[None, :], -np.inf))
                A = np.where(strict, bb[:, None] * decay * (K @ K.T), 0.0)
                T = np.linalg.solve(np.eye(n) + A, np.eye(n))
                U = T @ (bb[:, None] * V)
                W = T @ ((bb * gamma)[:, None] * K)
                Delta = U - W @ S0
                P = decay * (Q @ K.T)
                out[b, h, sl] = scale * (gamma[:, None] * (Q @ S0) + P @ Delta)
                Ktil = np.exp(Gc[-1] - Gc)[:, None] * K
                S0 = gamma[-1] * S0 + Ktil.T @ Delta
            st[b, h] = S0
    return out, st
