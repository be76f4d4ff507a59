"""csr_sddmm_static_scratch, the SDDMM entry point for callers that cannot
allocate device memory (it takes its scratch from a fixed array inside the
library instead of a caller workspace), checked against csr_sddmm.

This file is named so pytest collects it last; it passes on its own in a
fresh process and after the rest of the suite."""
import ctypes

import numpy as np
import pytest

import workloads as W
from parity_util import TOL, assert_within, dev, host, oracle_sddmm

pytestmark = pytest.mark.gpu

STATIC_SCRATCH_BYTES = 32 << 20


def _call_static(lib, usm, ro, ci, csr, Xd, Yd, out, in_code, out_code):
    D = Xd.shape[1]
    return lib.csr_sddmm_static_scratch(
        csr.M, csr.K, D, csr.nnz, ro.data_ptr(), ci.data_ptr(), None, 0,
        Xd.data_ptr(), Xd.stride(0), Yd.data_ptr(), Yd.stride(0), out.data_ptr(), in_code, out_code,
        usm._stream())


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_static_scratch_matches_csr_sddmm_twice(usm, dtype):
    import torch
    lib = usm.load()
    code = 1 if dtype == "bf16" else 0
    # Two different problems in a row, both needing scratch (D spans several
    # strips); the second must not see anything the first left behind.
    for call, (M, K, D, seed) in enumerate([(700, 500, 300, 1), (900, 650, 520, 2)]):
        csr = W.random_csr([seed, 77], M, K, 0.15, dtype=dtype)
        rng = np.random.default_rng([seed, 78])
        X, Y = W.dense(rng, M, D, 1.0, dtype), W.dense(rng, K, D, 1.0, dtype)
        Xd, Yd = usm._tma_ready(dev(X, dtype)), usm._tma_ready(dev(Y, dtype))
        need = lib.csr_sddmm_workspace_bytes(M, K, D, csr.nnz, code)
        assert 0 < need <= STATIC_SCRATCH_BYTES
        ro, ci = dev(csr.row_offsets), dev(csr.col_indices)
        got = torch.full((csr.nnz,), float("nan"), device="cuda")
        assert _call_static(lib, usm, ro, ci, csr, Xd, Yd, got, code, 0) == 0
        want = usm.sddmm(ro, ci, Xd, Yd)
        assert usm.poll_status() == 0
        g, w = host(got).astype(np.float64), host(want).astype(np.float64)
        ref, S, _ = oracle_sddmm(csr, X, Y, dtype)
        assert_within(g, w, S, TOL[dtype], f"static scratch vs csr_sddmm, call {call + 1}")
        assert_within(g, ref, S, TOL[dtype], f"static scratch vs oracle, call {call + 1}")


def test_static_scratch_rejects_oversized_problem(usm):
    lib = usm.load()
    M, K, D = 4096, 4096, 4096      # a sparse mask (under 2% set): 32 strips of 128
    nnz = STATIC_SCRATCH_BYTES // (32 * 4) + 1
    assert lib.csr_sddmm_workspace_bytes(M, K, D, nnz, 0) > STATIC_SCRATCH_BYTES
    # Rejected on the host before any launch; the pointers are never read.
    fake = 0x10000
    code = lib.csr_sddmm_static_scratch(M, K, D, nnz, fake, fake, None, 0, fake, D, fake, D, fake, 0, 0,
                                        usm._stream())
    assert code == -3
