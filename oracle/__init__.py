"""fp64 CPU oracle for exact attention (forward and backward).

TEST INFRASTRUCTURE ONLY.  Only the tests, the smoke check and the bench's
cpu_baseline / reference leg may import this package.  The product library
(``exact_attention_36_gb300``) never imports it and has no CPU fallback.

The arithmetic lives in ``attn_oracle.c`` (the textbook definition of softmax
attention and of its chain-rule backward, in double precision).  This module
only marshals arrays: it converts the bf16 inputs to float64 exactly, cuts out
one (batch, head) slice at a time and calls the C routines.

Layout conventions follow the library's: Q/K/V/O/dO are [B, S, H, D];
LSE is [B, H, S].
"""
from __future__ import annotations

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
        lp = ctypes.POINTER(ctypes.c_long)
        L, I, Dd = ctypes.c_long, ctypes.c_int, ctypes.c_double
        lib.fa_oracle_fwd.argtypes = [dp, dp, dp, L, L, I, Dd, lp, L, dp, dp]
        lib.fa_oracle_fwd.restype = I
        lib.fa_oracle_bwd_stats.argtypes = [dp, dp, dp, dp, L, L, I, Dd, lp, L, dp, dp, dp]
        lib.fa_oracle_bwd_stats.restype = I
        lib.fa_oracle_bwd_dq.argtypes = [dp, dp, dp, dp, dp, dp, L, L, I, Dd, lp, L, dp]
        lib.fa_oracle_bwd_dq.restype = I
        lib.fa_oracle_bwd_dkdv.argtypes = [dp, dp, dp, dp, dp, dp, L, L, I, Dd, lp, L, dp, dp]
        lib.fa_oracle_bwd_dkdv.restype = I
        lib.fa_oracle_exp2.argtypes = [dp, dp, L]
        lib.fa_oracle_exp2.restype = None
        lib.fa_oracle_threads.argtypes = []
        lib.fa_oracle_threads.restype = I
        _lib = lib
    return _lib


def threads() -> int:
    """OpenMP threads the oracle uses."""
    return int(_load().fa_oracle_threads())


def _f64(x) -> np.ndarray:
    """Exact float64 copy of a torch tensor (any float dtype) or array."""
    try:
        import torch
        if isinstance(x, torch.Tensor):
            return x.detach().to("cpu", torch.float64).contiguous().numpy()
    except ImportError:  # pragma: no cover
        pass
    return np.ascontiguousarray(np.asarray(x, dtype=np.float64))


def _ptr(a: np.ndarray):
    return a.ctypes.data_as(ctypes.POINTER(ctypes.c_double))


def _lptr(a):
    if a is None:
        return None
    return a.ctypes.data_as(ctypes.POINTER(ctypes.c_long))


def _idx(a):
    if a is None:
        return None, 0
    a = np.ascontiguousarray(np.asarray(a, dtype=np.int64))
    return a, int(a.size)


def _head(x64: np.ndarray, b: int, h: int) -> np.ndarray:
    return np.ascontiguousarray(x64[b, :, h, :])


def forward_head(q, k, v, causal: bool, scale: float, rows=None):
    """Oracle forward of one head.  q/k/v: [S, D] float64.

    Returns (o [n, D], lse [n]) for the listed rows (all rows if None).
    """
    q, k, v = _f64(q), _f64(k), _f64(v)
    S, D = q.shape
    rows_a, n = _idx(rows)
    if rows_a is None:
        n = S
    o = np.empty((n, D), np.float64)
    lse = np.empty((n,), np.float64)
    rc = _load().fa_oracle_fwd(_ptr(q), _ptr(k), _ptr(v), S, D, int(causal), float(scale),
                               _lptr(rows_a), n, _ptr(o), _ptr(lse))
    if rc != 0:
        raise MemoryError("oracle forward: allocation failed")
    return o, lse


def backward_head(q, k, v, dout, causal: bool, scale: float, rows=None, cols=None,
                  want_o: bool = False):
    """Oracle backward of one head.  All inputs [S, D] float64.

    Returns a dict with lse [S], delta [S], dq [len(rows), D] (rows of dQ),
    dk / dv [len(cols), D] (rows of dK / dV for the listed keys) and, if
    want_o, the exact forward output o [S, D].
    """
    q, k, v, dout = _f64(q), _f64(k), _f64(v), _f64(dout)
    S, D = q.shape
    lib = _load()
    lse = np.empty((S,), np.float64)
    delta = np.empty((S,), np.float64)
    o = np.empty((S, D), np.float64) if want_o else None
    rc = lib.fa_oracle_bwd_stats(_ptr(q), _ptr(k), _ptr(v), _ptr(dout), S, D, int(causal),
                                 float(scale), None, S, _ptr(lse), _ptr(delta),
                                 _ptr(o) if o is not None else None)
    if rc != 0:
        raise MemoryError("oracle backward stats: allocation failed")
    rows_a, nr = _idx(rows)
    if rows_a is None:
        nr = S
    cols_a, nc = _idx(cols)
    if cols_a is None:
        nc = S
    dq = np.empty((nr, D), np.float64)
    dk = np.empty((nc, D), np.float64)
    dv = np.empty((nc, D), np.float64)
    rc = lib.fa_oracle_bwd_dq(_ptr(q), _ptr(k), _ptr(v), _ptr(dout), _ptr(lse), _ptr(delta),
                              S, D, int(causal), float(scale), _lptr(rows_a), nr, _ptr(dq))
    if rc != 0:
        raise MemoryError("oracle dq: allocation failed")
    rc = lib.fa_oracle_bwd_dkdv(_ptr(q), _ptr(k), _ptr(v), _ptr(dout), _ptr(lse), _ptr(delta),
                                S, D, int(causal), float(scale), _lptr(cols_a), nc,
                                _ptr(dk), _ptr(dv))
    if rc != 0:
        raise MemoryError("oracle dk/dv: allocation failed")
    out = {"lse": lse, "delta": delta, "dq": dq, "dk": dk, "dv": dv}
    if want_o:
        out["o"] = o
    return out


def row_stats_head(q, k, v, dout, causal: bool, scale: float, rows):
    """LSE_i and Delta_i (= sum_j P_ij dP_ij) of one head for the listed rows.

    Returns (lse [n], delta [n]) as an (n,)-array pair.
    """
    q, k, v, dout = _f64(q), _f64(k), _f64(v), _f64(dout)
    S, D = q.shape
    rows_a, n = _idx(rows)
    lse = np.empty((n,), np.float64)
    delta = np.empty((n,), np.float64)
    rc = _load().fa_oracle_bwd_stats(_ptr(q), _ptr(k), _ptr(v), _ptr(dout), S, D, int(causal),
                                     float(scale), _lptr(rows_a), n, _ptr(lse), _ptr(delta), None)
    if rc != 0:
        raise MemoryError("oracle row stats: allocation failed")
    return lse, delta


def dq_rows_head(q, k, v, dout, lse_full, delta_full, causal: bool, scale: float, rows):
    """Rows of dQ of one head given LSE/Delta arrays indexed by row (only the
    listed rows' entries are read)."""
    q, k, v, dout = _f64(q), _f64(k), _f64(v), _f64(dout)
    S, D = q.shape
    rows_a, n = _idx(rows)
    lse_full = np.ascontiguousarray(lse_full, dtype=np.float64)
    delta_full = np.ascontiguousarray(delta_full, dtype=np.float64)
    dq = np.empty((n, D), np.float64)
    rc = _load().fa_oracle_bwd_dq(_ptr(q), _ptr(k), _ptr(v), _ptr(dout), _ptr(lse_full),
                                  _ptr(delta_full), S, D, int(causal), float(scale),
                                  _lptr(rows_a), n, _ptr(dq))
    if rc != 0:
        raise MemoryError("oracle dq: allocation failed")
    return dq


def forward(q, k, v, causal: bool, scale: float, heads=None, rows=None):
    """Oracle forward over [B, S, H, D] inputs.

    heads: list of (b, h) pairs (default: every head).  rows: optional query
    rows to evaluate (default: all).  Returns {(b, h): (o, lse)}.
    """
    q64, k64, v64 = _f64(q), _f64(k), _f64(v)
    B, S, H, D = q64.shape
    if heads is None:
        heads = [(b, h) for b in range(B) for h in range(H)]
    out = {}
    for (b, h) in heads:
        out[(b, h)] = forward_head(_head(q64, b, h), _head(k64, b, h), _head(v64, b, h),
                                   causal, scale, rows)
    return out


def backward(q, k, v, dout, causal: bool, scale: float, heads=None, rows=None, cols=None,
             want_o: bool = False):
    """Oracle backward over [B, S, H, D] inputs; returns {(b, h): dict}."""
    q64, k64, v64, d64 = _f64(q), _f64(k), _f64(v), _f64(dout)
    B, S, H, D = q64.shape
    if heads is None:
        heads = [(b, h) for b in range(B) for h in range(H)]
    out = {}
    for (b, h) in heads:
        out[(b, h)] = backward_head(_head(q64, b, h), _head(k64, b, h), _head(v64, b, h),
                                    _head(d64, b, h), causal, scale, rows, cols, want_o)
    return out


def exp2(x) -> np.ndarray:
    """2**x in double precision through the C library, elementwise."""
    x = np.ascontiguousarray(np.asarray(x, dtype=np.float64)).ravel()
    y = np.empty_like(x)
    _load().fa_oracle_exp2(_ptr(x), _ptr(y), x.size)
    return y
