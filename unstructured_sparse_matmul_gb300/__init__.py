"""Python binding of libusm (CSR SpMM / SDDMM / row swizzle on GB300).

Argument marshalling only: every step runs in the library's CUDA kernels,
called through the C ABI declared in include/usm.h.  PyTorch supplies device
memory and the current stream.  There is no CPU fallback: if the library is
not built, or no CUDA device is present, calls raise.

Source of the operations: "Sparse GPU Kernels for Deep Learning" (Gale,
Zaharia, Young, Elsen, SC 2020), summary card ("Summary"; "Interesting ideas"
I3 for the SDDMM form, I4 for the row swizzle, I5 for plain CSR).
"""
from __future__ import annotations

import ctypes
import os
import threading

from . import build as _build

USM_F32 = 0
USM_BF16 = 1

STATUS = {
    0: "USM_OK", -1: "USM_ERR_INVALID_ARG", -2: "USM_ERR_ALIGNMENT", -3: "USM_ERR_UNSUPPORTED",
    -4: "USM_ERR_CUDA", -5: "USM_ERR_TIMEOUT", -6: "USM_ERR_WORKSPACE",
}

# Every symbol include/usm.h declares, with its ctypes signature.
_vp, _i, _sz, _ll = ctypes.c_void_p, ctypes.c_int, ctypes.c_size_t, ctypes.c_longlong
SIGNATURES = {
    "csr_spmm": (_i, [_i, _i, _i, _i, _vp, _vp, _vp, _vp, _i, _vp, _i, _vp, _i, _i, _vp]),
    "csr_sddmm_workspace_bytes": (_sz, [_i, _i, _i, _i, _i]),
    "csr_sddmm": (_i, [_i, _i, _i, _i, _vp, _vp, _vp, _i, _vp, _i, _vp, _i, _vp, _i, _i, _vp, _sz, _vp]),
    "row_swizzle_workspace_bytes": (_sz, [_i, _i]),
    "row_swizzle_build": (_i, [_i, _i, _i, _vp, _vp, _vp, _sz, _vp]),
    "usm_poll_status": (_i, [_vp]),
    "usm_status_string": (ctypes.c_char_p, [_i]),
    "usm_selftest_wait_timeout": (_i, [_ll, _vp]),
    "usm_set_schedule_override": (_i, [_i, _i, _i]),
    "csr_sddmm_static_scratch": (_i, [_i, _i, _i, _i, _vp, _vp, _vp, _i, _vp, _i, _vp, _i, _vp, _i, _i, _vp]),
    "csr_transpose_workspace_bytes": (_sz, [_i, _i, _i]),
    "csr_sddmm_general_workspace_bytes": (_sz, [_i, _i, _i, _i, _i, _i]),
    "csr_sddmm_general": (_i, [_i, _i, _i, _i, _vp, _vp, _vp, _vp, _i, _vp, _i, _vp, _i, _i, _vp, _i, _i, _vp,
                               _sz, _vp]),
    "csr_row_softmax": (_i, [_i, _i, _vp, _vp, _vp, _i, _vp]),
    "csr_transpose": (_i, [_i, _i, _i, _vp, _vp, _vp, _i, _vp, _vp, _vp, _vp, _vp, _sz, _vp]),
    "csr_permute_values": (_i, [_i, _vp, _vp, _i, _vp, _vp]),
    "csr_validate": (_i, [_i, _i, _i, _vp, _vp, _vp, _vp]),
    "csr_spmm_row_softmax": (_i, [_i, _i, _i, _i, _vp, _vp, _vp, _vp, _i, _vp, _i, _vp, _i, _i, _vp]),
}

# csr_validate result codes (usm_csr_check in include/usm.h).
CSR_CHECK = {0: "USM_CSR_VALID", 1: "USM_CSR_FIRST_OFFSET", 2: "USM_CSR_OFFSETS_DECREASE",
             3: "USM_CSR_LAST_OFFSET", 4: "USM_CSR_COLUMN_RANGE", 5: "USM_CSR_COLUMN_ORDER"}
CSR_VALIDATE_INTS = 8

_lib = None
_lock = threading.Lock()


class USMError(RuntimeError):
    def __init__(self, fn: str, code: int):
        super().__init__(f"{fn} returned {code} ({STATUS.get(code, 'unknown')})")
        self.code = code


def library_path() -> str:
    return _build.LIB


def load(build_if_missing: bool = True):
    """Load libusm.so (building it first if needed) and bind its symbols."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        if not os.path.exists(_build.LIB) or not _build.up_to_date():
            if not build_if_missing:
                raise RuntimeError(f"CUDA library not built: {_build.LIB}")
            _build.build_library()
        lib = ctypes.CDLL(_build.LIB)
        for name, (res, args) in SIGNATURES.items():
            fn = getattr(lib, name)
            fn.restype = res
            fn.argtypes = args
        _lib = lib
        return lib


def _check(fn: str, code: int):
    if code != 0:
        raise USMError(fn, code)


# ---------------------------------------------------------------------------
# torch helpers (memory and streams only)
# ---------------------------------------------------------------------------
def _torch():
    import torch
    if not torch.cuda.is_available():
        raise RuntimeError("no CUDA device: libusm has no CPU fallback")
    return torch


def _ptr(t) -> int | None:
    return None if t is None else t.data_ptr()


def _stream(stream=None):
    torch = _torch()
    s = stream if stream is not None else torch.cuda.current_stream()
    return ctypes.c_void_p(s.cuda_stream)


def _dtype_code(t) -> int:
    torch = _torch()
    if t.dtype == torch.float32:
        return USM_F32
    if t.dtype == torch.bfloat16:
        return USM_BF16
    raise TypeError(f"unsupported element type {t.dtype} (fp32 or bf16)")


def _require(t, name, dtypes=None, cuda=True):
    if t is None:
        raise ValueError(f"{name} is required")
    if cuda and not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if dtypes is not None and t.dtype not in dtypes:
        raise TypeError(f"{name} has dtype {t.dtype}, expected one of {dtypes}")


def _ld(t) -> int:
    if t.dim() != 2 or t.stride(1) != 1:
        raise ValueError("dense operands must be 2-D with unit column stride")
    return t.stride(0)


def _round_up(x: int, m: int) -> int:
    return (x + m - 1) // m * m


def _tma_ready(t):
    """The library reads dense inputs with TMA, which needs a 16-byte aligned
    base and a row pitch that is a multiple of 16 bytes.  Inputs that already
    satisfy this pass through untouched; others are copied once into a padded
    buffer (a marshalling copy; pass aligned tensors to avoid it)."""
    es = t.element_size()
    if (t.dim() == 2 and t.stride(1) == 1 and t.data_ptr() % 16 == 0
            and (t.stride(0) * es) % 16 == 0 and t.stride(0) >= t.shape[1]):
        return t
    torch = _torch()
    rows, cols = t.shape
    ld = _round_up(max(cols, 1), 16 // es)
    buf = torch.zeros((rows, ld), dtype=t.dtype, device=t.device)
    buf[:, :cols] = t
    return buf[:, :cols]


def _new_dense_out(rows: int, cols: int, device):
    """fp32 output with a row pitch that is a multiple of 4 elements."""
    torch = _torch()
    ld = _round_up(max(cols, 1), 4)
    return torch.empty((rows, ld), dtype=torch.float32, device=device)[:, :cols]


# ---------------------------------------------------------------------------
# Operations
# ---------------------------------------------------------------------------
def row_swizzle(row_offsets, K: int, seg_rows: int = 0, out=None, stream=None):
    """Row-swizzle order (int32[M]) of a CSR's rows; see row_swizzle_build."""
    torch = _torch()
    lib = load()
    _require(row_offsets, "row_offsets", (torch.int32,))
    M = row_offsets.numel() - 1
    out = out if out is not None else torch.empty(M, dtype=torch.int32, device=row_offsets.device)
    ws_bytes = lib.row_swizzle_workspace_bytes(M, K)
    ws = torch.empty(max(ws_bytes, 16), dtype=torch.uint8, device=row_offsets.device)
    _check("row_swizzle_build", lib.row_swizzle_build(M, K, seg_rows, _ptr(row_offsets), _ptr(out),
                                                      _ptr(ws), ws_bytes, _stream(stream)))
    return out


def spmm(row_offsets, col_indices, values, B, K: int | None = None, row_swizzle=None, out=None,
         stream=None, seg_rows: int = 0):
    """C = A·B (fp32 out).  values and B are both fp32 or both bf16."""
    torch = _torch()
    lib = load()
    _require(row_offsets, "row_offsets", (torch.int32,))
    _require(col_indices, "col_indices", (torch.int32,))
    _require(values, "values", (torch.float32, torch.bfloat16))
    _require(B, "B", (values.dtype,))
    M = row_offsets.numel() - 1
    K = B.shape[0] if K is None else K
    N = B.shape[1]
    B = _tma_ready(B)
    C = out if out is not None else _new_dense_out(M, N, B.device)
    _require(C, "out", (torch.float32,))
    code = lib.csr_spmm(M, K, N, col_indices.numel(), _ptr(row_offsets), _ptr(col_indices), _ptr(values),
                        _ptr(row_swizzle), seg_rows, _ptr(B), _ld(B), _ptr(C), _ld(C), _dtype_code(values),
                        _stream(stream))
    _check("csr_spmm", code)
    return C


def spmm_row_softmax(row_offsets, col_indices, scores, B, K: int | None = None, row_swizzle=None, out=None,
                     stream=None, seg_rows: int = 0):
    """C = softmax_rows(scores)·B (fp32 out): each row's stored fp32 scores
    turned into softmax probabilities, rounded to B's element type (fp32 or
    bf16), inside the product; see csr_spmm_row_softmax."""
    torch = _torch()
    lib = load()
    _require(row_offsets, "row_offsets", (torch.int32,))
    _require(col_indices, "col_indices", (torch.int32,))
    _require(scores, "scores", (torch.float32,))
    _require(B, "B", (torch.float32, torch.bfloat16))
    M = row_offsets.numel() - 1
    K = B.shape[0] if K is None else K
    N = B.shape[1]
    B = _tma_ready(B)
    C = out if out is not None else _new_dense_out(M, N, B.device)
    _require(C, "out", (torch.float32,))
    code = lib.csr_spmm_row_softmax(M, K, N, col_indices.numel(), _ptr(row_offsets), _ptr(col_indices), _ptr(scores),
                                    _ptr(row_swizzle), seg_rows, _ptr(B), _ld(B), _ptr(C), _ld(C), _dtype_code(B),
                                    _stream(stream))
    _check("csr_spmm_row_softmax", code)
    return C


def sddmm(row_offsets, col_indices, X, Y, row_swizzle=None, out=None, out_dtype=None, workspace=None,
          stream=None, seg_rows: int = 0):
    """out[p] = X[r]·Y[col_p] on the mask's nonzeros (CSR order)."""
    torch = _torch()
    lib = load()
    _require(row_offsets, "row_offsets", (torch.int32,))
    _require(col_indices, "col_indices", (torch.int32,))
    _require(X, "X", (torch.float32, torch.bfloat16))
    _require(Y, "Y", (X.dtype,))
    M = row_offsets.numel() - 1
    K, D = Y.shape[0], Y.shape[1]
    if X.shape[1] != D:
        raise ValueError("X and Y must have the same number of columns")
    X, Y = _tma_ready(X), _tma_ready(Y)
    nnz = col_indices.numel()
    if out is None:
        od = out_dtype if out_dtype is not None else torch.float32
        out = torch.empty(nnz, dtype=od, device=X.device)
    in_code = _dtype_code(X)
    out_code = _dtype_code(out)
    ws_bytes = lib.csr_sddmm_workspace_bytes(M, K, D, nnz, in_code)
    if ws_bytes and (workspace is None or workspace.numel() * workspace.element_size() < ws_bytes):
        workspace = torch.empty(ws_bytes, dtype=torch.uint8, device=X.device)
    code = lib.csr_sddmm(M, K, D, nnz, _ptr(row_offsets), _ptr(col_indices), _ptr(row_swizzle), seg_rows,
                         _ptr(X), _ld(X), _ptr(Y), _ld(Y), _ptr(out), in_code, out_code,
                         _ptr(workspace) if ws_bytes else None, ws_bytes, _stream(stream))
    _check("csr_sddmm", code)
    return out


def sddmm_general(row_offsets, col_indices, X, Y, values=None, y_transposed=True, row_swizzle=None, out=None,
                  out_dtype=None, stream=None, seg_rows: int = 0):
    """out[p] = (values[p] if given) · X[r]·Yop[col_p]; Yop = Y (K×D) when
    y_transposed, else Yᵀ with Y given D×K."""
    torch = _torch()
    lib = load()
    _require(row_offsets, "row_offsets", (torch.int32,))
    _require(col_indices, "col_indices", (torch.int32,))
    _require(X, "X", (torch.float32, torch.bfloat16))
    _require(Y, "Y", (X.dtype,))
    if values is not None:
        _require(values, "values", (X.dtype,))
    M = row_offsets.numel() - 1
    D = X.shape[1]
    K = Y.shape[0] if y_transposed else Y.shape[1]
    if (Y.shape[1] if y_transposed else Y.shape[0]) != D:
        raise ValueError("X and Y disagree on D")
    X = _tma_ready(X)
    if y_transposed:
        Y = _tma_ready(Y)
    elif Y.stride(1) != 1:
        Y = Y.contiguous()
    nnz = col_indices.numel()
    if out is None:
        out = torch.empty(nnz, dtype=out_dtype if out_dtype is not None else torch.float32, device=X.device)
    in_code = _dtype_code(X)
    ws_bytes = lib.csr_sddmm_general_workspace_bytes(M, K, D, nnz, in_code, int(bool(y_transposed)))
    ws = torch.empty(max(ws_bytes, 16), dtype=torch.uint8, device=X.device)
    code = lib.csr_sddmm_general(M, K, D, nnz, _ptr(row_offsets), _ptr(col_indices), _ptr(values),
                                 _ptr(row_swizzle), seg_rows, _ptr(X), _ld(X), _ptr(Y), Y.stride(0),
                                 int(bool(y_transposed)),
                                 _ptr(out), in_code, _dtype_code(out), _ptr(ws) if ws_bytes else None, ws_bytes,
                                 _stream(stream))
    _check("csr_sddmm_general", code)
    return out


def row_softmax(row_offsets, scores, out=None, out_dtype=None, stream=None):
    """Softmax over the stored entries of each CSR row (fp32 scores in)."""
    torch = _torch()
    lib = load()
    _require(row_offsets, "row_offsets", (torch.int32,))
    _require(scores, "scores", (torch.float32,))
    if out is None:
        out = torch.empty_like(scores, dtype=out_dtype if out_dtype is not None else torch.float32)
    code = lib.csr_row_softmax(row_offsets.numel() - 1, scores.numel(), _ptr(row_offsets), _ptr(scores), _ptr(out),
                               _dtype_code(out), _stream(stream))
    _check("csr_row_softmax", code)
    return out


def csr_validate(row_offsets, col_indices, K: int, stream=None):
    """Check the CSR contract on the device: (code, index), code one of
    CSR_CHECK (0 = valid), index the first offending row or nonzero (-1 when
    valid).  Reads the two result words back, so it waits for the stream."""
    torch = _torch()
    lib = load()
    _require(row_offsets, "row_offsets", (torch.int32,))
    _require(col_indices, "col_indices", (torch.int32,))
    result = torch.empty(CSR_VALIDATE_INTS, dtype=torch.int32, device=row_offsets.device)
    code = lib.csr_validate(row_offsets.numel() - 1, K, col_indices.numel(), _ptr(row_offsets), _ptr(col_indices),
                            _ptr(result), _stream(stream))
    _check("csr_validate", code)
    out = result[:2].cpu()
    return int(out[0]), int(out[1])


def csr_transpose(row_offsets, col_indices, values, K: int, with_perm: bool = False, stream=None):
    """Aᵀ in CSR: (row_offsets_t, col_indices_t, values_t[, perm])."""
    torch = _torch()
    lib = load()
    _require(row_offsets, "row_offsets", (torch.int32,))
    _require(col_indices, "col_indices", (torch.int32,))
    M = row_offsets.numel() - 1
    nnz = col_indices.numel()
    dev = row_offsets.device
    ro_t = torch.empty(K + 1, dtype=torch.int32, device=dev)
    ci_t = torch.empty(nnz, dtype=torch.int32, device=dev)
    v_t = torch.empty_like(values) if values is not None else None
    perm = torch.empty(nnz, dtype=torch.int32, device=dev) if with_perm else None
    code_dt = _dtype_code(values) if values is not None else USM_F32
    ws_bytes = lib.csr_transpose_workspace_bytes(M, K, nnz)
    ws = torch.empty(max(ws_bytes, 16), dtype=torch.uint8, device=dev)
    code = lib.csr_transpose(M, K, nnz, _ptr(row_offsets), _ptr(col_indices), _ptr(values), code_dt, _ptr(ro_t),
                             _ptr(ci_t), _ptr(v_t), _ptr(perm), _ptr(ws), ws_bytes, _stream(stream))
    _check("csr_transpose", code)
    return (ro_t, ci_t, v_t, perm) if with_perm else (ro_t, ci_t, v_t)


def csr_permute_values(perm, values, out=None, stream=None):
    """out[q] = values[perm[q]]."""
    lib = load()
    out = out if out is not None else values.new_empty(perm.numel())
    _check("csr_permute_values", lib.csr_permute_values(perm.numel(), _ptr(perm), _ptr(values), _dtype_code(values),
                                                        _ptr(out), _stream(stream)))
    return out


def poll_status(stream=None) -> int:
    return int(load().usm_poll_status(_stream(stream)))


def set_schedule_override(rows_per_warp: int = 0, tiles_per_block: int = 0, k_splits: int = 0) -> None:
    """Force the launch shape of later SpMM/SDDMM calls (0 = the library's
    choice); see usm_set_schedule_override."""
    _check("usm_set_schedule_override", load().usm_set_schedule_override(rows_per_warp, tiles_per_block, k_splits))


def status_string(code: int) -> str:
    return load().usm_status_string(code).decode()
