"""ctypes front end of the C oracle (``mla_verify_ref.c``) -- test infrastructure.

The C file is compiled with plain ``gcc -O2 -fopenmp`` (no fast-math, so
IEEE fp64 arithmetic in source order) into ``liboracle.so`` next to it.
"""

from __future__ import annotations

import ctypes
import os
import subprocess
import threading
from typing import Optional, Sequence

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "mla_verify_ref.c")
_LIB = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile the oracle if the library is missing or older than its source."""
    if (not force and os.path.exists(_LIB)
            and os.path.getmtime(_LIB) >= os.path.getmtime(_SRC)):
        return _LIB
    tmp = _LIB + ".tmp%d" % os.getpid()
    cmd = ["gcc", "-O2", "-fopenmp", "-fPIC", "-shared", "-std=c11", "-o", tmp, _SRC, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    with _lock:
        if _lib is None:
            build()
            lib = ctypes.CDLL(_LIB)
            P = ctypes.c_void_p
            i32, i64, f64 = ctypes.c_int, ctypes.c_int64, ctypes.c_double
            lib.oracle_mla_verify.argtypes = [i32, i32, i32, P, P, P, P, i64, P, P, P, P, P, f64,
                                              P, i64, P, P, i32, i32]
            lib.oracle_mla_verify.restype = i32
            lib.oracle_mla_verify_split_merge.argtypes = [i32, i32, i32, P, P, P, P, i64, P, P, P, P, P,
                                                          f64, i32, i64, i64, P, i64, P, P, i32]
            lib.oracle_mla_verify_split_merge.restype = i32
            lib.oracle_max_threads.argtypes = []
            lib.oracle_max_threads.restype = i32
            _lib = lib
    return _lib


def max_threads() -> int:
    return int(_load().oracle_max_threads())


def _c(a, dtype):
    a = np.ascontiguousarray(a, dtype=dtype)
    return a, a.ctypes.data_as(ctypes.c_void_p)


def _common(wl):
    keep = []
    ptrs = []
    for key, dt in (("q_nope", np.uint16), ("q_rope", np.uint16), ("pool", np.uint16),
                    ("kv_indptr", np.int32), ("kv_indices", np.int32), ("out_cache_loc", np.int32),
                    ("custom_mask", np.uint8), ("mask_indptr", np.int32)):
        arr = wl[key]
        if arr.size == 0:
            arr = np.zeros(1, dtype=dt)
        a, p = _c(arr, dt)
        keep.append(a)
        ptrs.append(p)
    return keep, ptrs


def _qo(wl):
    """qo_indptr (request token offsets) of a varlen call, else None (uniform T)."""
    qo = wl.get("qo_indptr")
    if qo is None:
        return None, None
    a, p = _c(qo, np.int32)
    return a, p


def n_token_rows(wl) -> int:
    qo = wl.get("qo_indptr")
    return int(qo[-1]) if qo is not None else wl["B"] * wl["T"]


def _rows(wl, rows):
    n_all = n_token_rows(wl) * wl["H"]
    if rows is None:
        return None, None, n_all
    r = np.ascontiguousarray(np.asarray(rows, dtype=np.int64))
    return r, r.ctypes.data_as(ctypes.c_void_p), int(r.size)


def verify(wl: dict, rows: Optional[Sequence[int]] = None, nthreads: int = 0, mutation: int = 0,
           sm_scale: Optional[float] = None):
    """Direct fp64 evaluation; returns (O [n,512] float64, LSE [n] float64)."""
    lib = _load()
    keep, (qn, qr, pool, indptr, idx, ocl, mask, mindptr) = _common(wl)
    r, rp, n = _rows(wl, rows)
    o = np.zeros((n, 512), dtype=np.float64)
    lse = np.zeros(n, dtype=np.float64)
    scale = wl["sm_scale"] if sm_scale is None else sm_scale
    qo_keep, qo = _qo(wl)
    rc = lib.oracle_mla_verify(wl["B"], wl["H"], wl["T"], qo, qn, qr, pool, wl["pool"].shape[0], indptr, idx,
                               ocl, mask, mindptr, float(scale), rp, n,
                               o.ctypes.data_as(ctypes.c_void_p), lse.ctypes.data_as(ctypes.c_void_p),
                               int(nthreads), int(mutation))
    if rc != 0:
        raise ValueError("oracle: a referenced pool row is out of range")
    del keep
    return o, lse


def verify_split_merge(wl: dict, nsplit: int, granule: int = 1, min_chunk: int = 1,
                       rows: Optional[Sequence[int]] = None, nthreads: int = 0):
    """Split-then-merge fp64 evaluation (same quantity, organised per split)."""
    lib = _load()
    keep, (qn, qr, pool, indptr, idx, ocl, mask, mindptr) = _common(wl)
    r, rp, n = _rows(wl, rows)
    o = np.zeros((n, 512), dtype=np.float64)
    lse = np.zeros(n, dtype=np.float64)
    qo_keep, qo = _qo(wl)
    rc = lib.oracle_mla_verify_split_merge(wl["B"], wl["H"], wl["T"], qo, qn, qr, pool, wl["pool"].shape[0],
                                           indptr, idx, ocl, mask, mindptr, float(wl["sm_scale"]),
                                           int(nsplit), int(granule), int(min_chunk), rp, n,
                                           o.ctypes.data_as(ctypes.c_void_p),
                                           lse.ctypes.data_as(ctypes.c_void_p), int(nthreads))
    if rc != 0:
        raise ValueError("oracle split/merge failed (%d)" % rc)
    del keep
    return o, lse
