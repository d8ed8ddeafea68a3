"""The oracle: plain, slow, obviously correct CPU implementations of the Kimi
Delta Attention gated delta-rule scan, in fp64.

TEST INFRASTRUCTURE. Only tests/, __graft_entry__.smoke() and bench.py's
CPU-baseline leg may import anything under oracle/. The product path (the CUDA
library and its Python binding) never imports it, and the oracle imports
nothing from the product package.

Three independent formulations live here, each written from the pages:

* ``scan`` / ``decode_step`` — the token-by-token definition
  ("Understanding Kimi Delta Attention", box "KDA: Retain, predict, correct";
  "Demystifying Kimi Delta Attention", opening KDA equations for the query
  scale), in plain C (kda_scan.c), threaded over (sequence, head).
* ``chunkwise.chunkwise_scan`` — the chunkwise/WY form derived in
  "Understanding Kimi Delta Attention", sections "The triangular system" and
  "Putting the chunks together", in numpy.
* ``dense.dense_scan`` — the explicit product of diagonal-plus-low-rank
  transitions, "Understanding Kimi Delta Attention", box "KDA as a structured
  state transition", in numpy.

Parity status: every function here is pinned by tests/test_oracle_pins.py
against worked examples, closed forms, special cases and each other.
"""
import ctypes
import os

import numpy as np

from . import build as _build

_lib = None


def _load():
    global _lib
    if _lib is None:
        path = _build.build()
        lib = ctypes.CDLL(path)
        dp = ctypes.POINTER(ctypes.c_double)
        lib.kda_oracle_scan.argtypes = [dp, dp, dp, dp, dp, ctypes.c_double, dp,
                                        ctypes.POINTER(ctypes.c_int64), ctypes.c_int,
                                        ctypes.c_int, ctypes.c_int, ctypes.c_int, dp, dp,
                                        ctypes.c_int]
        lib.kda_oracle_scan.restype = ctypes.c_int
        lib.kda_oracle_hw_threads.argtypes = []
        lib.kda_oracle_hw_threads.restype = ctypes.c_int
        _lib = lib
    return _lib


def hw_threads() -> int:
    """Threads the oracle uses by default (online processors of this host)."""
    return int(_load().kda_oracle_hw_threads())


def _f64(x):
    return np.ascontiguousarray(np.asarray(x, dtype=np.float64))


def _ptr(a):
    return a.ctypes.data_as(ctypes.POINTER(ctypes.c_double))


def scan(q, k, v, g, beta, scale, init_state=None, cu_seqlens=None, nthreads=0):
    """Token-by-token fp64 scan.

    Shapes: q, k, g ``[B, T, H, d_k]``; v ``[B, T, H, d_v]``; beta ``[B, T, H]``.
    Without ``cu_seqlens`` the B rows are B sequences of length T. With
    ``cu_seqlens`` (length N+1) B must be 1 and sequence n spans tokens
    ``cu_seqlens[n]:cu_seqlens[n+1]``. ``g`` is the per-token log-decay
    log a_t (not cumulative). ``init_state`` is ``[N, H, d_k, d_v]`` or None
    (zeros). Returns ``(out [B, T, H, d_v], final_state [N, H, d_k, d_v])``.
    """
    q, k, v, g, beta = (_f64(x) for x in (q, k, v, g, beta))
    if q.ndim != 4:
        raise ValueError("q must be [B, T, H, d_k]")
    B, T, H, dk = q.shape
    dv = v.shape[-1]
    if k.shape != q.shape or g.shape != q.shape or v.shape != (B, T, H, dv):
        raise ValueError("q, k, g, v shapes disagree")
    if beta.shape != (B, T, H):
        raise ValueError("beta must be [B, T, H]")
    if cu_seqlens is None:
        cu = np.arange(B + 1, dtype=np.int64) * T
    else:
        if B != 1:
            raise ValueError("cu_seqlens requires B == 1")
        cu = np.ascontiguousarray(np.asarray(cu_seqlens, dtype=np.int64))
        if cu[0] != 0 or cu[-1] != T or np.any(np.diff(cu) < 0):
            raise ValueError("cu_seqlens must rise from 0 to T")
    N = len(cu) - 1
    init = None if init_state is None else _f64(init_state)
    if init is not None and init.shape != (N, H, dk, dv):
        raise ValueError("init_state must be [N, H, d_k, d_v]")
    out = np.zeros((B, T, H, dv), dtype=np.float64)
    final = np.zeros((N, H, dk, dv), dtype=np.float64)
    lib = _load()
    rc = lib.kda_oracle_scan(_ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta), float(scale),
                             None if init is None else _ptr(init),
                             cu.ctypes.data_as(ctypes.POINTER(ctypes.c_int64)), N, H, dk, dv,
                             _ptr(out), _ptr(final), int(nthreads))
    if rc != 0:
        raise RuntimeError("oracle scan failed with code %d" % rc)
    return out, final


def decode_step(q, k, v, g, beta, scale, state, nthreads=0):
    """One recurrent step for N independent sequences.

    q, k, g ``[N, H, d_k]``; v ``[N, H, d_v]``; beta ``[N, H]``; state
    ``[N, H, d_k, d_v]``. Returns ``(out [N, H, d_v], new_state)``; the input
    state is not modified. A decode step is the scan over one token
    ("Kimi Delta Attention: How It Works, Step by Step", section 11).
    """
    q = _f64(q)
    N, H, dk = q.shape
    out, final = scan(q[None], _f64(k)[None], _f64(v)[None], _f64(g)[None], _f64(beta)[None],
                      scale, init_state=state, cu_seqlens=np.arange(N + 1), nthreads=nthreads)
    return out[0], final
