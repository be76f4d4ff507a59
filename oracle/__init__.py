"""CPU oracle for CSR SpMM / SDDMM — test infrastructure only.

A plain fp64 restatement of what the kernels of "Sparse GPU Kernels for Deep
Learning" (Gale et al., SC 2020) compute, used to check the CUDA library.
Only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline
and reference arms may import it.  The product path never calls it, and it
imports nothing from the CUDA package (nor the reverse).

Every function here marshals numpy arrays into ``usm_oracle.c`` (compiled
with gcc, OpenMP over rows, fp64 accumulation in CSR order).  Inputs are
widened exactly to fp64 first: fp32 by a cast, bf16 by placing its 16 bits
above 16 zero bits.

Parity pins (tests/test_oracle.py): dense brute force through numpy's
matmul, identity and permutation matrices, SDDMM ≡ mask ⊙ (X·Yᵀ), the adjoint
identity, integer-valued exactness, swizzle against a lexicographic sort,
hand-computed worked examples under tests/golden/.  Nothing is "parity
unpinned" except the pages' aggregate V100 ratios, which are not computed.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "usm_oracle.c")
_BUILD_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD_DIR, "liboracle.so")
_lock = threading.Lock()
_lib = None

_i32p = ctypes.POINTER(ctypes.c_int32)
_f64p = ctypes.POINTER(ctypes.c_double)
_u16p = ctypes.POINTER(ctypes.c_uint16)


def build(force: bool = False) -> str:
    """Compile usm_oracle.c into oracle/_build/liboracle.so (host compiler)."""
    os.makedirs(_BUILD_DIR, exist_ok=True)
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-fopenmp", "-ffp-contract=off", "-fno-fast-math", "-shared", "-fPIC",
           "-std=c11", _SRC, "-o", tmp, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _configure(lib):
    i64, i32 = ctypes.c_int64, ctypes.c_int
    lib.oracle_csr_check.argtypes = [i32, i32, i64, _i32p, _i32p]
    lib.oracle_csr_check.restype = ctypes.c_int
    lib.oracle_spmm.argtypes = [i32, i32, i32, _i32p, _i32p, _f64p, _f64p, i64, _f64p, i64, i32]
    lib.oracle_sddmm.argtypes = [i32, i32, i32, _i32p, _i32p, _f64p, i64, _f64p, i64, _f64p, i32]
    lib.oracle_sddmm_general.argtypes = [i32, i32, i32, _i32p, _i32p, _f64p, i32, _f64p, i64,
                                         _f64p, i64, i32, _f64p, i32]
    lib.oracle_row_swizzle.argtypes = [i32, i32, _i32p, _i32p]
    lib.oracle_csr_transpose.argtypes = [i32, i32, _i32p, _i32p, _f64p, _i32p, _i32p, _f64p]
    lib.oracle_csr_softmax.argtypes = [i32, _i32p, _f64p, _f64p, i32]
    lib.oracle_round_to_bf16.argtypes = [i64, _f64p, _u16p]
    lib.oracle_max_threads.restype = ctypes.c_int
    return lib


def _L():
    global _lib
    with _lock:
        if _lib is None:
            _lib = _configure(ctypes.CDLL(build()))
    return _lib


def _p(a, t):
    return a.ctypes.data_as(t)


def _i32(a):
    return np.ascontiguousarray(a, dtype=np.int32)


def _f64(a):
    return np.ascontiguousarray(a, dtype=np.float64)


def max_threads() -> int:
    return int(_L().oracle_max_threads())


# ---------------------------------------------------------------------------
# Widening of the stored inputs (exact)
# ---------------------------------------------------------------------------
def widen(x: np.ndarray, dtype: str) -> np.ndarray:
    """fp32 array or bf16 bit pattern (uint16) -> fp64, exactly."""
    if dtype == "bf16":
        bits = np.ascontiguousarray(x, dtype=np.uint16).astype(np.uint32) << 16
        return bits.view(np.float32).astype(np.float64)
    return np.asarray(x, dtype=np.float32).astype(np.float64)


def round_to_bf16(x: np.ndarray) -> np.ndarray:
    """fp64 -> bf16 bits, round to nearest even, one rounding step."""
    x = _f64(x).ravel()
    out = np.empty(x.size, dtype=np.uint16)
    _L().oracle_round_to_bf16(x.size, _p(x, _f64p), _p(out, _u16p))
    return out


# ---------------------------------------------------------------------------
# Operations
# ---------------------------------------------------------------------------
def csr_check(M: int, K: int, row_offsets, col_indices, nnz: int | None = None) -> int:
    """0 for a valid CSR, else the negative code of the first violation
    (usm_oracle.c).  nnz defaults to the length of col_indices."""
    ro, ci = _i32(row_offsets), _i32(col_indices)
    if ro.size != M + 1:
        return -7
    nnz = ci.size if nnz is None else nnz
    if nnz > ci.size:
        return -7
    return int(_L().oracle_csr_check(M, K, nnz, _p(ro, _i32p), _p(ci, _i32p)))


def spmm(M: int, K: int, row_offsets, col_indices, values64, B64, nthreads: int = 0) -> np.ndarray:
    """C = A·B in fp64; A given by CSR arrays and fp64 values, B fp64 K×N."""
    ro, ci, a = _i32(row_offsets), _i32(col_indices), _f64(values64)
    B = _f64(B64)
    N = B.shape[1] if B.ndim == 2 else 0
    C = np.empty((M, N), dtype=np.float64)
    if M == 0:
        return C
    _L().oracle_spmm(M, K, N, _p(ro, _i32p), _p(ci, _i32p), _p(a, _f64p), _p(B, _f64p), N,
                     _p(C, _f64p), N, nthreads)
    return C


def spmm_error_scale(M, K, row_offsets, col_indices, values64, B64, nthreads: int = 0):
    """S[r][j] = sum_p |a_p|·|B[col_p][j]|: the scale the fp32/bf16 error
    bound multiplies (it is SpMM of the absolute values)."""
    return spmm(M, K, row_offsets, col_indices, np.abs(_f64(values64)), np.abs(_f64(B64)), nthreads)


def sddmm(M: int, K: int, row_offsets, col_indices, X64, Y64, nthreads: int = 0) -> np.ndarray:
    """out[p] = X[r]·Y[col_p] (no scaling by values; Y is K×D)."""
    ro, ci = _i32(row_offsets), _i32(col_indices)
    X, Y = _f64(X64), _f64(Y64)
    D = X.shape[1]
    out = np.empty(int(ro[-1]), dtype=np.float64)
    if M == 0 or out.size == 0:
        return out
    _L().oracle_sddmm(M, K, D, _p(ro, _i32p), _p(ci, _i32p), _p(X, _f64p), D, _p(Y, _f64p),
                      Y.shape[1], _p(out, _f64p), nthreads)
    return out


def sddmm_error_scale(M, K, row_offsets, col_indices, X64, Y64, nthreads: int = 0):
    return sddmm(M, K, row_offsets, col_indices, np.abs(_f64(X64)), np.abs(_f64(Y64)), nthreads)


def sddmm_general(M: int, K: int, row_offsets, col_indices, values64, scale_by_values: bool,
                  X64, Y64, y_transposed: bool, nthreads: int = 0) -> np.ndarray:
    ro, ci = _i32(row_offsets), _i32(col_indices)
    a = _f64(values64) if values64 is not None else np.zeros(int(ro[-1]), dtype=np.float64)
    X, Y = _f64(X64), _f64(Y64)
    D = X.shape[1]
    out = np.empty(int(ro[-1]), dtype=np.float64)
    if M == 0 or out.size == 0:
        return out
    _L().oracle_sddmm_general(M, K, D, _p(ro, _i32p), _p(ci, _i32p), _p(a, _f64p),
                              int(bool(scale_by_values)), _p(X, _f64p), X.shape[1], _p(Y, _f64p),
                              Y.shape[1], int(bool(y_transposed)), _p(out, _f64p), nthreads)
    return out


def row_swizzle(row_offsets, seg_rows: int = 0) -> np.ndarray:
    ro = _i32(row_offsets)
    M = ro.size - 1
    perm = np.empty(M, dtype=np.int32)
    if M > 0:
        _L().oracle_row_swizzle(M, int(seg_rows), _p(ro, _i32p), _p(perm, _i32p))
    return perm


def csr_transpose(M: int, K: int, row_offsets, col_indices, values64):
    ro, ci, a = _i32(row_offsets), _i32(col_indices), _f64(values64)
    nnz = int(ro[-1])
    ro_t = np.empty(K + 1, dtype=np.int32)
    ci_t = np.empty(nnz, dtype=np.int32)
    a_t = np.empty(nnz, dtype=np.float64)
    _L().oracle_csr_transpose(M, K, _p(ro, _i32p), _p(ci, _i32p), _p(a, _f64p), _p(ro_t, _i32p),
                              _p(ci_t, _i32p), _p(a_t, _f64p))
    return ro_t, ci_t, a_t


def csr_softmax(row_offsets, scores64, nthreads: int = 0) -> np.ndarray:
    ro, s = _i32(row_offsets), _f64(scores64)
    out = np.zeros(s.size, dtype=np.float64)
    M = ro.size - 1
    if M > 0 and s.size:
        _L().oracle_csr_softmax(M, _p(ro, _i32p), _p(s, _f64p), _p(out, _f64p), nthreads)
    return out


# ---------------------------------------------------------------------------
# Row sampling for full-size parity: the sub-CSR of selected rows (indexing
# only, no arithmetic) so the oracle computes exactly those outputs.
# ---------------------------------------------------------------------------
def select_rows(row_offsets, col_indices, rows):
    ro = np.asarray(row_offsets, dtype=np.int64)
    rows = np.asarray(rows, dtype=np.int64)
    lens = ro[rows + 1] - ro[rows]
    sub_ro = np.zeros(rows.size + 1, dtype=np.int64)
    np.cumsum(lens, out=sub_ro[1:])
    pos = np.concatenate([np.arange(ro[r], ro[r + 1]) for r in rows]) if rows.size else np.zeros(0, np.int64)
    return sub_ro.astype(np.int32), np.asarray(col_indices)[pos].astype(np.int32), pos
