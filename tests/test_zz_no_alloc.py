"""csr_sddmm_static_scratch, the SDDMM entry point for callers that cannot
allocate device memory (a plugin that only receives raw pointers, a loop
whose memory was fixed at start-up): it takes its scratch from a fixed array
inside the library instead of a caller workspace.  Checked against
csr_sddmm, which runs the same kernels in the same order, so the two must
agree bit for bit, and against the oracle.

This file is named so pytest collects it last; it passes on its own in a
fresh process and after the rest of the suite."""
import numpy as np
import pytest

import workloads as W
from parity_util import TOL, assert_within, dev, host, oracle_sddmm

pytestmark = pytest.mark.gpu

STATIC_SCRATCH_BYTES = 32 << 20


def _call_static(lib, usm, ro, ci, csr, Xd, Yd, out, in_code, out_code, perm=None):
    D = Xd.shape[1]
    return lib.csr_sddmm_static_scratch(
        csr.M, csr.K, D, csr.nnz, ro.data_ptr(), ci.data_ptr(), None if perm is None else perm.data_ptr(), 0,
        Xd.data_ptr(), Xd.stride(0), Yd.data_ptr(), Yd.stride(0), out.data_ptr(), in_code, out_code,
        usm._stream())


def _bits(t):
    """Output bits for an exact comparison (bf16 as its 16-bit pattern)."""
    h = host(t)
    return h if h.dtype == np.uint16 else h.view(np.uint32)


# (M, K, D, seed, row swizzle, bf16 output): two different problems in a row,
# both needing scratch (D spans several strips), the second with a row
# swizzle and bf16 output; each must match csr_sddmm bit for bit, so nothing
# the previous call left in the shared array leaks into it.
CALLS = [(700, 500, 300, 1, False, False), (900, 650, 520, 2, True, True)]


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_static_scratch_matches_csr_sddmm_twice(usm, dtype):
    import torch
    lib = usm.load()
    code = 1 if dtype == "bf16" else 0
    for call, (M, K, D, seed, swz, out16) in enumerate(CALLS):
        csr = W.random_csr([seed, 77], M, K, 0.15, dtype=dtype)
        rng = np.random.default_rng([seed, 78])
        X, Y = W.dense(rng, M, D, 1.0, dtype), W.dense(rng, K, D, 1.0, dtype)
        Xd, Yd = usm._tma_ready(dev(X, dtype)), usm._tma_ready(dev(Y, dtype))
        need = lib.csr_sddmm_workspace_bytes(M, K, D, csr.nnz, code)
        assert 0 < need <= STATIC_SCRATCH_BYTES
        ro, ci = dev(csr.row_offsets), dev(csr.col_indices)
        perm = usm.row_swizzle(ro, K) if swz else None
        odt = torch.bfloat16 if out16 else torch.float32
        got = torch.full((csr.nnz,), float("nan"), dtype=odt, device="cuda")
        assert _call_static(lib, usm, ro, ci, csr, Xd, Yd, got, code, 1 if out16 else 0, perm) == 0
        torch.cuda.synchronize()
        # A repeat of the same call (its kernels are loaded now) allocates
        # nothing: neither torch's allocator nor the device's free memory moves.
        again = torch.full_like(got, float("nan"))
        torch.cuda.synchronize()
        free0, alloc0 = torch.cuda.mem_get_info()[0], torch.cuda.memory_allocated()
        assert _call_static(lib, usm, ro, ci, csr, Xd, Yd, again, code, 1 if out16 else 0, perm) == 0
        torch.cuda.synchronize()
        assert torch.cuda.mem_get_info()[0] == free0, "device memory taken by a repeated call"
        assert torch.cuda.memory_allocated() == alloc0
        want = usm.sddmm(ro, ci, Xd, Yd, row_swizzle=perm, out_dtype=odt)
        assert usm.poll_status() == 0
        assert np.array_equal(_bits(got), _bits(want)), f"call {call + 1}: differs from csr_sddmm"
        assert np.array_equal(_bits(again), _bits(want)), f"call {call + 1} repeated: differs from csr_sddmm"
        if not out16:
            ref, S, _ = oracle_sddmm(csr, X, Y, dtype)
            assert_within(host(got).astype(np.float64), ref, S, TOL[dtype], f"static scratch vs oracle, call {call + 1}")


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
