"""Host-side checks of the C ABI that need no GPU: the library builds for
sm_103a, loads, exports every function include/usm.h declares, and rejects
bad arguments before touching the device (no compute call is made here)."""
import ctypes
import os
import re

import pytest

import unstructured_sparse_matmul_gb300 as usm
from unstructured_sparse_matmul_gb300 import build as usm_build

HEADER = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "include", "usm.h")

# Fake, never-dereferenced device addresses (host code only checks them).
A16 = 0x10000
ODD = 0x10004


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    names = re.findall(r"^\s*(?:const\s+)?[A-Za-z_][A-Za-z0-9_]*\s*\*?\s*([A-Za-z_][A-Za-z0-9_]*)\s*\(",
                       text, flags=re.M)
    return sorted(set(names))


@pytest.fixture(scope="module")
def lib():
    return usm.load()


def test_header_declares_expected_entry_points():
    names = declared_functions()
    for n in ["csr_spmm", "csr_sddmm", "csr_sddmm_workspace_bytes", "row_swizzle_build",
              "row_swizzle_workspace_bytes", "usm_poll_status", "usm_status_string"]:
        assert n in names


def test_library_exports_every_declared_symbol(lib):
    names = declared_functions()
    assert names, "no declarations parsed"
    for n in names:
        assert hasattr(lib, n), f"{n} declared in usm.h but not exported"
        assert n in usm.SIGNATURES, f"{n} has no binding signature"


def test_library_is_built_for_sm103a():
    assert usm_build.ARCH == ["-gencode", "arch=compute_103a,code=sm_103a"]
    assert os.path.exists(usm_build.LIB)


def test_status_strings(lib):
    for code, name in usm.STATUS.items():
        assert lib.usm_status_string(code).decode() == name
    assert lib.usm_status_string(12345).decode() == "USM_UNKNOWN_STATUS"


def test_workspace_sizes(lib):
    assert lib.row_swizzle_workspace_bytes(0, 10) == 0
    assert lib.row_swizzle_workspace_bytes(4096, 1024) == 4096 * 4 + 256 * 2 * 4
    assert lib.csr_sddmm_workspace_bytes(10, 10, 64, 100, usm.USM_F32) == 0        # one strip
    assert lib.csr_sddmm_workspace_bytes(10, 10, 128, 100, usm.USM_F32) == 0
    assert lib.csr_sddmm_workspace_bytes(100, 10, 129, 100, usm.USM_F32) == 2 * 128 * 4  # 128-wide strips
    # masks at least a quarter full use 256-wide strips (bf16 too, unless D <= 64)
    assert lib.csr_sddmm_workspace_bytes(10, 10, 129, 100, usm.USM_F32) == 0
    assert lib.csr_sddmm_workspace_bytes(10, 10, 257, 25, usm.USM_F32) == 2 * 32 * 4  # strips 32-aligned
    assert lib.csr_sddmm_workspace_bytes(10, 10, 257, 24, usm.USM_F32) == 3 * 32 * 4
    assert lib.csr_sddmm_workspace_bytes(10, 10, 257, 100, usm.USM_BF16) == 2 * 128 * 4
    assert lib.csr_sddmm_workspace_bytes(100, 10, 257, 100, usm.USM_BF16) == 3 * 128 * 4
    assert lib.csr_sddmm_workspace_bytes(10, 10, 2048, 7, usm.USM_BF16) == 16 * 32 * 4
    assert lib.csr_sddmm_workspace_bytes(10, 10, 64, 7, usm.USM_BF16) == 0
    assert lib.csr_sddmm_workspace_bytes(10, 10, 0, 7, usm.USM_F32) == 0
    # general SDDMM: transposed-Y region (K x ld, 256-byte aligned) + strip partials
    assert lib.csr_sddmm_general_workspace_bytes(10, 10, 64, 7, usm.USM_F32, 1) == 0
    assert lib.csr_sddmm_general_workspace_bytes(10, 10, 64, 7, usm.USM_F32, 0) == 2560  # 10 x 64 x 4
    assert lib.csr_transpose_workspace_bytes(10, 10, 0) == 0
    assert lib.csr_transpose_workspace_bytes(10, 10, 100) == 512 * 2 + 1024 + 512


def spmm(lib, M=4, K=4, N=8, nnz=4, ro=A16, ci=A16, vals=A16, perm=None, B=A16, ldb=8, C=A16, ldc=8, dt=0):
    return lib.csr_spmm(M, K, N, nnz, ro, ci, vals, perm, 0, B, ldb, C, ldc, dt, None)


def test_spmm_rejects_bad_args_on_host(lib):
    assert spmm(lib, M=-1) == -1
    assert spmm(lib, N=-3) == -1
    assert spmm(lib, nnz=-1) == -1
    assert spmm(lib, dt=7) == -1
    assert spmm(lib, ldc=4) == -1                      # ldc < N
    assert spmm(lib, C=None) == -1
    assert spmm(lib, ro=None) == -1
    assert spmm(lib, C=ODD) == -2                      # C not 16-byte aligned
    assert spmm(lib, ldc=10) == -2                     # ldc not a multiple of 4
    assert spmm(lib, K=0) == -1                        # nonzeros with no columns
    assert spmm(lib, ci=None) == -1
    assert spmm(lib, ldb=4) == -1                      # ldb < N
    assert spmm(lib, B=ODD) == -2
    assert spmm(lib, ldb=9) == -2                      # row pitch 36 bytes
    assert spmm(lib, dt=1, ldb=12) == -2               # bf16 pitch 24 bytes
    # empty problems are no-ops that never touch the pointers
    assert spmm(lib, M=0, C=None, ro=None) == 0
    assert spmm(lib, N=0, C=None) == 0


def sddmm(lib, M=4, K=4, D=8, nnz=4, ro=A16, ci=A16, perm=None, X=A16, ldx=8, Y=A16, ldy=8, out=A16,
          it=0, ot=0, ws=None, wsb=0):
    return lib.csr_sddmm(M, K, D, nnz, ro, ci, perm, 0, X, ldx, Y, ldy, out, it, ot, ws, wsb, None)


def test_sddmm_rejects_bad_args_on_host(lib):
    assert sddmm(lib, M=-1) == -1
    assert sddmm(lib, D=-1) == -1
    assert sddmm(lib, it=2) == -1
    assert sddmm(lib, ot=5) == -1
    assert sddmm(lib, out=None) == -1
    assert sddmm(lib, K=0) == -1
    assert sddmm(lib, X=None) == -1
    assert sddmm(lib, ldx=4) == -1
    assert sddmm(lib, X=ODD) == -2
    assert sddmm(lib, ldy=9) == -2
    assert sddmm(lib, D=300, ldx=300, ldy=300) == -6   # needs workspace, none given
    assert sddmm(lib, D=300, ldx=300, ldy=300, ws=A16, wsb=10) == -6
    assert sddmm(lib, M=0) == 0
    assert sddmm(lib, nnz=0, out=None) == 0


def test_swizzle_rejects_bad_args_on_host(lib):
    assert lib.row_swizzle_build(-1, 4, 0, A16, A16, A16, 1 << 20, None) == -1
    assert lib.row_swizzle_build(4, -1, 0, A16, A16, A16, 1 << 20, None) == -1
    assert lib.row_swizzle_build(4, 4, 0, None, A16, A16, 1 << 20, None) == -1
    assert lib.row_swizzle_build(4, 4, 0, A16, A16, None, 1 << 20, None) == -6
    assert lib.row_swizzle_build(4, 4, 0, A16, A16, A16, 8, None) == -6
    assert lib.row_swizzle_build(0, 4, 0, None, None, None, 0, None) == 0


def test_next_rows_reject_bad_args_on_host(lib):
    assert lib.csr_transpose(-1, 4, 4, A16, A16, A16, 0, A16, A16, A16, None, A16, 1 << 20, None) == -1
    assert lib.csr_transpose(4, 0, 4, A16, A16, A16, 0, A16, A16, A16, None, A16, 1 << 20, None) == -1
    assert lib.csr_transpose(4, 4, 4, A16, A16, A16, 0, A16, A16, None, None, A16, 1 << 20, None) == -1
    assert lib.csr_transpose(4, 4, 4, A16, A16, A16, 0, A16, A16, A16, None, None, 0, None) == -6
    assert lib.csr_transpose(4, 4, 4, A16, A16, A16, 0, A16, A16, A16, None, A16 + 16, 1 << 20, None) == -2
    assert lib.csr_permute_values(-1, A16, A16, 0, A16, None) == -1
    assert lib.csr_permute_values(5, None, A16, 0, A16, None) == -1
    assert lib.csr_permute_values(0, None, None, 0, None, None) == 0
    g = lambda **k: lib.csr_sddmm_general(*[k.get(n, v) for n, v in [
        ("M", 4), ("K", 4), ("D", 8), ("nnz", 4), ("ro", A16), ("ci", A16), ("vals", None), ("perm", None), ("seg", 0),
        ("X", A16), ("ldx", 8), ("Y", A16), ("ldy", 8), ("ytr", 1), ("out", A16), ("it", 0), ("ot", 0),
        ("ws", None), ("wsb", 0), ("st", None)]])
    assert g(ytr=2) == -1
    assert g(ytr=0, ldy=3) == -1            # D x K operand needs ldy >= K
    assert g(ytr=0) == -6                   # transposed copy of Y needs workspace
    assert g(X=ODD) == -2
    assert g(M=0) == 0
    assert lib.csr_row_softmax(-1, 4, A16, A16, A16, 0, None) == -1
    assert lib.csr_row_softmax(4, 4, A16, A16, A16, 3, None) == -1
    assert lib.csr_row_softmax(4, 4, None, A16, A16, 0, None) == -1
    assert lib.csr_row_softmax(0, 4, None, None, None, 0, None) == 0


def test_selftest_rejects_bad_limit(lib):
    assert lib.usm_selftest_wait_timeout(10, None) == -1
    assert lib.usm_selftest_wait_timeout(10**12, None) == -1


def test_binding_refuses_without_gpu():
    torch = pytest.importorskip("torch")
    if torch.cuda.is_available():
        pytest.skip("a GPU is present")
    with pytest.raises(RuntimeError, match="no CUDA device"):
        usm.spmm(None, None, None, None)


def test_schedule_override_validation(lib):
    f = lib.usm_set_schedule_override
    INVALID = -1
    try:
        for bad in [(3, 0, 0), (64, 0, 0), (-1, 0, 0), (0, -1, 0), (0, 0, -1), (0, 0, 65536)]:
            assert f(*bad) == INVALID, bad
        for good in [(0, 0, 0), (1, 0, 0), (32, 5, 7), (4, 0, 65535), (16, 100000, 1)]:
            assert f(*good) == 0, good
    finally:
        assert f(0, 0, 0) == 0


def test_validate_rejects_bad_args_on_host(lib):
    v = lib.csr_validate
    assert v(-1, 4, 0, A16, A16, A16, None) == -1
    assert v(4, -1, 0, A16, A16, A16, None) == -1
    assert v(4, 4, -1, A16, A16, A16, None) == -1
    assert v(4, 4, 5, A16, None, A16, None) == -1       # nonzeros need col_indices
    assert v(4, 4, 5, None, A16, A16, None) == -1       # row_offsets always read
    assert v(4, 4, 5, A16, A16, None, None) == -1       # nowhere to write the result
    assert v(4, 4, 5, A16, A16, A16 + 2, None) == -2    # result not int-aligned
