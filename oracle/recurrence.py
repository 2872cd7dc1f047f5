"""ctypes front end of the C per-token recurrence (the oracle).

TEST INFRASTRUCTURE ONLY.  See ``ssd_oracle.c`` for what is computed and the
readings taken where the pages leave a step open.
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional

import numpy as np

from . import build as _build

_lib = None


def lib() -> ctypes.CDLL:
    global _lib
    if _lib is None:
        path = _build.build()
        _lib = ctypes.CDLL(path)
        f = _lib.ssd_oracle_varlen_fwd
        f.restype = ctypes.c_int
        f.argtypes = ([ctypes.c_void_p] * 12
                      + [ctypes.c_int64, ctypes.c_int32, ctypes.c_int32, ctypes.c_int32,
                         ctypes.c_int32, ctypes.c_int32, ctypes.c_int64, ctypes.c_int32,
                         ctypes.c_void_p, ctypes.c_int32, ctypes.c_int32, ctypes.c_int32])
        _lib.ssd_oracle_max_threads.restype = ctypes.c_int
    return _lib


def max_threads() -> int:
    return int(lib().ssd_oracle_max_threads())


def _ptr(a: Optional[np.ndarray]):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _c(a, dtype):
    return None if a is None else np.ascontiguousarray(a, dtype=dtype)


def ssd_varlen_fwd(*, x, dt, A, B, C, D, dt_bias, ssm_pool, query_start_loc,
                   has_initial_state, cache_indices, dt_softplus: bool = True,
                   seq_select=None, heads=None, num_threads: int = 0):
    """Run the fp64 recurrence.

    Arguments are NumPy arrays with the op's shapes (bf16 tensors as uint16
    bit patterns).  ``ssm_pool`` is not modified: a copy is updated and
    returned.  ``seq_select`` (bool per sequence) and ``heads`` (a (begin, end)
    range) restrict the work; outputs of unselected work are NaN in ``y`` and
    unchanged in the pool.

    Returns ``(y, pool_out)``: ``y`` fp64 (T, H, P), ``pool_out`` fp32.
    """
    x = _c(x, np.uint16)
    dt = _c(dt, np.uint16)
    A = _c(A, np.float32)
    B = _c(B, np.uint16)
    C = _c(C, np.uint16)
    D = _c(D, np.float32)
    dt_bias = _c(dt_bias, np.float32)
    pool = np.array(ssm_pool, dtype=np.float32, copy=True, order="C")
    qsl = _c(query_start_loc, np.int32)
    hinit = _c(has_initial_state, np.uint8)
    cidx = _c(cache_indices, np.uint32)
    sel = _c(seq_select, np.uint8)
    T, H, P = x.shape
    G, N = B.shape[1], B.shape[2]
    batch = qsl.shape[0] - 1
    h0, h1 = (0, H) if heads is None else heads
    y = np.full((T, H, P), np.nan, dtype=np.float64)
    rc = lib().ssd_oracle_varlen_fwd(
        _ptr(y), _ptr(pool), _ptr(x), _ptr(dt), _ptr(A), _ptr(B), _ptr(C), _ptr(D),
        _ptr(dt_bias), _ptr(qsl), _ptr(hinit), _ptr(cidx),
        T, batch, H, P, G, N, pool.shape[0], int(bool(dt_softplus)),
        _ptr(sel), h0, h1, int(num_threads))
    if rc != 0:
        raise ValueError(f"oracle rejected its arguments (code {rc})")
    return y, pool


def run_workload(w, **kw):
    """Convenience: run the oracle on a ``Workload``-like object."""
    return ssd_varlen_fwd(x=w.x, dt=w.dt, A=w.A, B=w.B, C=w.C, D=w.D, dt_bias=w.dt_bias,
                          ssm_pool=w.ssm_pool, query_start_loc=w.query_start_loc,
                          has_initial_state=w.has_initial_state,
                          cache_indices=w.cache_indices, dt_softplus=w.dt_softplus, **kw)
