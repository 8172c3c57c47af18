"""CPU oracle for the sparse-weight direct convolution (TEST INFRASTRUCTURE).

A plain, slow, fp64 C implementation (``spconv_oracle.c``) reached through
ctypes.  Only the tests, the smoke check and the benchmark's CPU-baseline leg
use it; the library under ``sparse_weight_direct_gb300`` never imports it and
shares no code with it.

Functions:

* ``out_dim``   -- Tuteja et al., "Theoretical and Empirical Analysis of Sparse
  Convolution", Sec. 3 Eq.(2): floor((H + 2P - K) / s) + 1.
* ``dense7``    -- Escoin (arXiv 1802.10280), "CONV layer" Algorithm 1: the
  seven-loop nest over a dense M x C x R x S filter, with Eq.(1)'s clipped
  kernel range (zero padding, no flip).
* ``csr``       -- Escoin "Sparse weights" CSR and Algorithm 2 (walk each row's
  nonzeros over every output position), i.e. Tuteja et al. Eq.(3).
* ``csr_points``-- Eq.(3) evaluated one output element at a time.

Each returns ``abs_sum`` = sum |w * x| over the same terms alongside the result.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_LIB_PATH = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_lib = None

_i32p = np.ctypeslib.ndpointer(dtype=np.int32, flags="C_CONTIGUOUS")
_i64p = np.ctypeslib.ndpointer(dtype=np.int64, flags="C_CONTIGUOUS")
_f64p = np.ctypeslib.ndpointer(dtype=np.float64, flags="C_CONTIGUOUS")
_int = ctypes.c_int


def build() -> str:
    """Compile liboracle.so with the Makefile beside this file."""
    subprocess.run(["make", "-s", "-C", _HERE], check=True)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        src = os.path.join(_HERE, "spconv_oracle.c")
        if (not os.path.exists(_LIB_PATH)
                or os.path.getmtime(_LIB_PATH) < os.path.getmtime(src)):
            build()
        lib = ctypes.CDLL(_LIB_PATH)
        dims = [_int] * 9
        lib.oracle_out_dim.argtypes = [_int] * 4
        lib.oracle_out_dim.restype = _int
        lib.oracle_num_cpus.argtypes = []
        lib.oracle_num_cpus.restype = _int
        lib.oracle_dense7.argtypes = dims + [_f64p, _f64p, _f64p, _f64p]
        lib.oracle_dense7.restype = _int
        lib.oracle_csr.argtypes = dims + [_i32p, _i32p, _f64p, _f64p, _f64p, _f64p, _int]
        lib.oracle_csr.restype = _int
        lib.oracle_csr_points.argtypes = dims + [_i32p, _i32p, _f64p, _f64p,
                                                 ctypes.c_int64, _i64p, _f64p, _f64p]
        lib.oracle_csr_points.restype = _int
        _lib = lib
        return lib


def out_dim(size: int, k: int, stride: int, pad: int) -> int:
    return int(_load().oracle_out_dim(size, k, stride, pad))


def num_cpus() -> int:
    return int(_load().oracle_num_cpus())


def _f64(a) -> np.ndarray:
    return np.ascontiguousarray(np.asarray(a, dtype=np.float64))


def _i32(a) -> np.ndarray:
    return np.ascontiguousarray(np.asarray(a, dtype=np.int32))


def dense7(x, w, stride: int, pad: int):
    """x: (N, C, H, W); w: (M, C, R, S) dense.  Returns (y, abs_sum), fp64."""
    x = _f64(x)
    w = _f64(w)
    N, C, H, W = x.shape
    M, C2, R, S = w.shape
    if C2 != C:
        raise ValueError("channel mismatch")
    E, F = out_dim(H, R, stride, pad), out_dim(W, S, stride, pad)
    y = np.zeros((N, M, max(E, 0), max(F, 0)))
    a = np.zeros_like(y)
    rc = _load().oracle_dense7(N, C, H, W, M, R, S, stride, pad, x, w, y, a)
    if rc != 0:
        raise ValueError(f"oracle_dense7 rejected its arguments ({rc})")
    return y, a


def csr(x, rowptr, colidx, value, M: int, R: int, S: int, stride: int, pad: int,
        threads: int = 0, return_threads: bool = False):
    """CSR walker.  Returns (y, abs_sum) [, threads used]."""
    x = _f64(x)
    N, C, H, W = x.shape
    E, F = out_dim(H, R, stride, pad), out_dim(W, S, stride, pad)
    y = np.zeros((N, M, max(E, 0), max(F, 0)))
    a = np.zeros_like(y)
    rc = _load().oracle_csr(N, C, H, W, M, R, S, stride, pad, _i32(rowptr), _i32(colidx),
                            _f64(value), x, y, a, threads)
    if rc < 1:
        raise ValueError(f"oracle_csr rejected its arguments ({rc})")
    return (y, a, rc) if return_threads else (y, a)


def csr_points(x, rowptr, colidx, value, M: int, R: int, S: int, stride: int, pad: int,
               flat_idx):
    """Eq.(3) at the given flat NMEF output indices.  Returns (y, abs_sum)."""
    x = _f64(x)
    N, C, H, W = x.shape
    idx = np.ascontiguousarray(np.asarray(flat_idx, dtype=np.int64))
    y = np.zeros(idx.size)
    a = np.zeros(idx.size)
    rc = _load().oracle_csr_points(N, C, H, W, M, R, S, stride, pad, _i32(rowptr),
                                   _i32(colidx), _f64(value), x, idx.size, idx, y, a)
    if rc != 0:
        raise ValueError(f"oracle_csr_points rejected its arguments ({rc})")
    return y, a


def csr_to_dense(rowptr, colidx, value, M: int, C: int, R: int, S: int) -> np.ndarray:
    """Scatter CSR back into a dense (M, C, R, S) fp64 filter (no arithmetic)."""
    w = np.zeros((M, C * R * S))
    rowptr = np.asarray(rowptr)
    for m in range(M):
        lo, hi = int(rowptr[m]), int(rowptr[m + 1])
        np.add.at(w[m], np.asarray(colidx[lo:hi]), np.asarray(value[lo:hi], dtype=np.float64))
    return w.reshape(M, C, R, S)
