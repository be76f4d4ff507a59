"""CUDA path vs the CPU oracle, element by element, through the C ABI.

Every case is compared in full, every output element against the oracle:
small cases (several tiles, ragged tails, edge cases) and the five workload
configurations at full size, in the same launch configuration the benchmark
times.  Swizzles are compared bit-exactly; integer-valued inputs must match
bit-exactly too (every partial sum is an exact integer)."""
import numpy as np
import pytest

import oracle
import workloads as W
from parity_util import TOL, assert_within, dev, host, oracle_sddmm, oracle_spmm

pytestmark = pytest.mark.gpu


def csr_dev(csr):
    return dev(csr.row_offsets), dev(csr.col_indices), dev(csr.values, csr.dtype)


# ---------------------------------------------------------------------------
# Row swizzle (bit-exact)
# ---------------------------------------------------------------------------
SWIZZLE_CASES = [
    ("tiny", lambda: W.tiny().csr, 0),
    ("ragged", lambda: W.random_csr(1, 5000, 300, 0.1), 0),
    ("ragged_seg", lambda: W.random_csr(2, 5000, 300, 0.1), 1000),
    ("one_row", lambda: W.random_csr(3, 1, 10, 0.5), 0),
    ("all_empty", lambda: W.random_csr(4, 300, 10, 0.0), 0),
    ("equal_lengths", lambda: W.random_csr(5, 777, 64, 0.0, lengths=np.full(777, 5)), 0),
    ("long_tail", lambda: W.random_csr(6, 3000, 70000, 0.0, lengths=np.r_[np.zeros(2999, int), [65000]]), 0),
    ("multi_tile_seg", lambda: W.random_csr(7, 9000, 100, 0.2), 4096),
]


@pytest.mark.parametrize("name,make,seg", SWIZZLE_CASES, ids=[c[0] for c in SWIZZLE_CASES])
def test_swizzle_bit_exact(usm, name, make, seg):
    csr = make()
    got = host(usm.row_swizzle(dev(csr.row_offsets), csr.K, seg))
    assert np.array_equal(got, oracle.row_swizzle(csr.row_offsets, seg))


def test_swizzle_full_configs(usm):
    for csr, seg in [(W.resnet(with_sddmm=False).csr, 0), (W.lstm(90).csr, 0),
                     (W.ffn(4096, 1024, 90, with_spmm=False, with_sddmm=False).csr, 0),
                     (W.attention().csr, 4096)]:
        got = host(usm.row_swizzle(dev(csr.row_offsets), csr.K, seg))
        assert np.array_equal(got, oracle.row_swizzle(csr.row_offsets, seg))


# ---------------------------------------------------------------------------
# SpMM, small and ragged, compared in full
# ---------------------------------------------------------------------------
SPMM_SHAPES = [
    (1, 1, 1, 1.0), (5, 7, 3, 0.5), (37, 61, 64, 0.3), (130, 300, 129, 0.2), (257, 1000, 200, 0.1),
    (300, 129, 513, 0.05), (64, 4097, 128, 0.3), (1000, 50, 8, 0.9), (513, 2000, 4, 0.02),
]


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("M,K,N,density", SPMM_SHAPES)
@pytest.mark.parametrize("swz", [False, True])
def test_spmm_small(usm, dtype, M, K, N, density, swz):
    csr = W.random_csr([M, K, N, 31], M, K, density, dtype=dtype)
    B = W.dense(np.random.default_rng([M, K, N, 32]), K, N, 1.0, dtype)
    ro, ci, vals = csr_dev(csr)
    perm = usm.row_swizzle(ro, K) if swz else None
    C = host(usm.spmm(ro, ci, vals, dev(B, dtype), K=K, row_swizzle=perm))
    ref, S = oracle_spmm(csr, B, dtype)
    assert_within(C, ref, S, TOL[dtype], f"spmm {dtype} {M}x{K}x{N}")


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_spmm_row_length_mix(usm, dtype):
    # Every row length 0..9, then some long rows, every start residue.
    lengths = np.r_[np.arange(10).repeat(7), [500, 1999, 2000, 33, 64, 65, 127, 128, 129]]
    rng = np.random.default_rng(40)
    lengths = rng.permutation(lengths)
    M, K, N = lengths.size, 2000, 136
    csr = W.random_csr(41, M, K, 0.0, dtype=dtype, lengths=lengths)
    B = W.dense(np.random.default_rng(42), K, N, 1.0, dtype)
    ro, ci, vals = csr_dev(csr)
    C = host(usm.spmm(ro, ci, vals, dev(B, dtype), K=K, row_swizzle=usm.row_swizzle(ro, K)))
    ref, S = oracle_spmm(csr, B, dtype)
    assert_within(C, ref, S, TOL[dtype], "row length mix")


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("N", [64, 128, 300])
def test_spmm_integer_valued_bit_exact(usm, dtype, N):
    M, K = 300, 700
    csr = W.random_csr([M, K, 43], M, K, 0.2, dtype=dtype, int_valued=True)
    B = W.dense(np.random.default_rng(44), K, N, 1.0, dtype, int_valued=True)
    ro, ci, vals = csr_dev(csr)
    C = host(usm.spmm(ro, ci, vals, dev(B, dtype), K=K))
    ref, _ = oracle_spmm(csr, B, dtype)
    assert np.array_equal(C.astype(np.float64), ref)


def test_spmm_identity_and_permutation_bit_exact(usm):
    n, N = 1000, 72
    B = W.dense(np.random.default_rng(45), n, N)
    perm = np.random.default_rng(46).permutation(n).astype(np.int32)
    ro = np.arange(n + 1, dtype=np.int32)
    ones = np.ones(n, dtype=np.float32)
    for cols in (np.arange(n, dtype=np.int32), perm):
        C = host(usm.spmm(dev(ro), dev(cols), dev(ones), dev(B), K=n))
        assert np.array_equal(C, B[cols])


def test_spmm_empty_cases(usm):
    import torch
    # nnz = 0: C is zero-filled (the buffer starts as garbage)
    csr = W.random_csr(47, 50, 40, 0.0)
    B = W.dense(np.random.default_rng(48), 40, 24)
    out = torch.full((50, 24), float("nan"), device="cuda")
    ro, ci, vals = csr_dev(csr)
    C = host(usm.spmm(ro, ci, vals, dev(B), K=40, out=out))
    assert np.array_equal(C, np.zeros((50, 24), np.float32))
    # M = 0 and N = 0 are no-ops
    z = usm.spmm(dev(np.zeros(1, np.int32)), ci, vals, dev(B), K=40)
    assert z.shape == (0, 24)
    # rows that are all empty but one
    lengths = np.zeros(300, int)
    lengths[123] = 40
    csr = W.random_csr(49, 300, 40, 0.0, lengths=lengths)
    ro, ci, vals = csr_dev(csr)
    C = host(usm.spmm(ro, ci, vals, dev(B), K=40))
    ref, S = oracle_spmm(csr, B, "f32")
    assert_within(C, ref, S, TOL["f32"], "one nonempty row")


def test_spmm_leading_dimensions(usm):
    import torch
    M, K, N = 200, 300, 100
    csr = W.random_csr(50, M, K, 0.1)
    Bbig = W.dense(np.random.default_rng(51), K, 132)
    Bv = dev(Bbig)[:, :N]
    out = torch.zeros((M, 104), device="cuda")
    ro, ci, vals = csr_dev(csr)
    usm.spmm(ro, ci, vals, Bv, K=K, out=out[:, :N])
    ref, S = oracle_spmm(csr, np.ascontiguousarray(Bbig[:, :N]), "f32")
    C = host(out)
    assert_within(C[:, :N], ref, S, TOL["f32"], "ld")
    assert np.all(C[:, N:] == 0), "wrote outside the N columns"


@pytest.mark.parametrize("M,K,N,density,seg", [(900, 500, 300, 0.4, 0), (700, 2500, 257, 0.3, 0),
                                                (1000, 1000, 512, 0.6, 500), (300, 4097, 600, 0.3, 0),
                                                (800, 1500, 300, 0.17, 0)])
def test_spmm_tensor_memory_rows(usm, schedule, M, K, N, density, seg):
    """fp32 masks at least 15% set with N > 128 read the last 64 rows
    of every chunk from tensor memory, with chunks of 192 rows (K = 500,
    1500) and 208 (K = 1000, 2500, 4097: fewer chunks): ragged last chunks
    (some of those rows lie past K), several and ragged
    strips, block-diagonal schedules and forced schedules, every element
    against the oracle and forced schedules bit for bit."""
    if seg:
        K = M
        rng = np.random.default_rng([M, 151])
        lengths = rng.binomial(seg, density, M)
        base = (np.arange(M) // seg) * seg
        ro, ci = W.csr_from_lengths(rng, lengths, seg, col_base=base)
        csr = W.CSR(M, K, ro, ci, W.values_for(rng, int(ro[-1]), 1.0, "f32"), "f32", seg_rows=seg)
    else:
        csr = W.random_csr([M, K, N, 152], M, K, density)
    assert csr.nnz >= 0.15 * M * K
    B = W.dense(np.random.default_rng([M, K, 153]), K, N)
    rod, cid, vd = csr_dev(csr)
    Bd = dev(B)
    perm = usm.row_swizzle(rod, K, seg)
    outs = []
    for r, t, s_ in [(0, 0, 0), (2, 0, 0), (4, 0, 0), (0, 40, 0)]:
        schedule(r, t, s_)
        outs.append(host(usm.spmm(rod, cid, vd, Bd, K=K, row_swizzle=perm, seg_rows=seg)))
    for c in outs[1:]:
        assert np.array_equal(c, outs[0])
    ref, S = oracle_spmm(csr, B, "f32")
    assert_within(outs[0], ref, S, TOL["f32"], f"tensor-memory spmm {M}x{K}x{N}")
    assert usm.poll_status() == 0


# fp32 masks at least 55% set (256-wide strips for N > 128, 128-wide for
# 64 < N <= 128), K <= 6144, with 64-row tiles x strips covering at least half
# the SMs: the row-group kernel.  (Block-diagonal masks of two or more blocks
# are at most half set, so they never take it.)
ROW_GROUP_CASES = [(1300, 3000, 1000, 0.6, 0), (5000, 500, 300, 0.58, 0), (2560, 2560, 300, 1.0, 0),
                   (2500, 6144, 300, 0.58, 0), (5000, 1000, 100, 0.6, 0), (5000, 2500, 128, 0.58, 0),
                   (5000, 1500, 65, 0.9, 0)]


@pytest.mark.parametrize("M,K,N,density,seg", ROW_GROUP_CASES)
def test_spmm_row_groups(usm, schedule, M, K, N, density, seg):
    """Row groups (a staged row of B serves every row of a warp holding its
    column), on 256- and 128-wide strips: ragged strips and chunks, K under
    one chunk, fully dense rows (every slab reloads the windows),
    the largest K the kernel takes, and forced schedules bit for bit; every
    element against the oracle."""
    if seg:
        K = M
        rng = np.random.default_rng([M, 154])
        lengths = rng.binomial(seg, density, M)
        base = (np.arange(M) // seg) * seg
        ro, ci = W.csr_from_lengths(rng, lengths, seg, col_base=base)
        csr = W.CSR(M, K, ro, ci, W.values_for(rng, int(ro[-1]), 1.0, "f32"), "f32", seg_rows=seg)
    else:
        csr = W.random_csr([M, K, N, 155], M, K, density)
    import torch
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    strip = 256 if N > 128 else 128
    assert csr.nnz >= 0.55 * M * K
    assert 2 * ((M + 63) // 64) * ((N + strip - 1) // strip) >= sms
    B = W.dense(np.random.default_rng([M, K, 156]), K, N)
    rod, cid, vd = csr_dev(csr)
    Bd = dev(B)
    perm = usm.row_swizzle(rod, K, seg)
    outs = []
    for r, t, s_ in [(0, 0, 0), (2, 0, 0), (4, 0, 0), (0, 40, 0), (4, 200, 0)]:
        schedule(r, t, s_)
        outs.append(host(usm.spmm(rod, cid, vd, Bd, K=K, row_swizzle=perm, seg_rows=seg)))
    for c in outs[1:]:
        assert np.array_equal(c, outs[0])
    ref, S = oracle_spmm(csr, B, "f32")
    assert_within(outs[0], ref, S, TOL["f32"], f"row-group spmm {M}x{K}x{N}")
    assert usm.poll_status() == 0


@pytest.mark.parametrize("N", [100, 300])
def test_spmm_row_groups_schedule_arguments_do_not_change_bits(usm, N):
    """Fully dense diagonal blocks of 2048 rows, the last one ragged (1024
    rows and columns), so 56% of the mask is set: N = 300 takes 256-wide row
    groups, N = 100 the row kernel (48 tiles of one 128-wide strip cover under
    half the SMs).  No swizzle, a global swizzle, and per-block swizzles with
    and without seg_rows give the same bits."""
    seg = 2048
    M = K = 3 * seg // 2
    rng = np.random.default_rng([N, 163])
    base = (np.arange(M) // seg) * seg
    width = np.minimum(base + seg, K) - base
    ro = np.concatenate([[0], np.cumsum(width)]).astype(np.int32)
    ci = np.concatenate([np.arange(b, b + w) for b, w in zip(base, width)]).astype(np.int32)
    csr = W.CSR(M, K, ro, ci, W.values_for(rng, int(ro[-1]), 1.0, "f32"), "f32", seg_rows=seg)
    assert csr.nnz >= 0.55 * M * K
    B = W.dense(rng, K, N)
    rod, cid, vd = csr_dev(csr)
    Bd = dev(B)
    variants = [(None, 0), (usm.row_swizzle(rod, K), 0), (usm.row_swizzle(rod, K, seg), seg),
                (usm.row_swizzle(rod, K, seg), 0)]
    Cs = [host(usm.spmm(rod, cid, vd, Bd, K=K, row_swizzle=p, seg_rows=sr)) for p, sr in variants]
    for c in Cs[1:]:
        assert np.array_equal(c, Cs[0])
    ref, S = oracle_spmm(csr, B, "f32")
    assert_within(Cs[0], ref, S, TOL["f32"], f"dense blocks N={N}")


def test_spmm_row_groups_integer_valued_bit_exact(usm):
    M, K, N = 1300, 1000, 1000
    csr = W.random_csr([M, K, 157], M, K, 0.6, int_valued=True)
    B = W.dense(np.random.default_rng(158), K, N, 1.0, "f32", int_valued=True)
    ro, ci, vals = csr_dev(csr)
    C = host(usm.spmm(ro, ci, vals, dev(B), K=K))
    ref, _ = oracle_spmm(csr, B, "f32")
    assert np.array_equal(C.astype(np.float64), ref)


@pytest.mark.parametrize("N,ldb,ldc", [(300, 312, 304), (100, 132, 104)])
def test_spmm_row_groups_leading_dimensions(usm, N, ldb, ldc):
    """Row groups (256- and 128-wide strips) on B and C that are views of
    wider buffers: the right result, and nothing written past column N."""
    import torch
    M, K = 5000, 700
    csr = W.random_csr([N, 161], M, K, 0.6)
    Bbig = W.dense(np.random.default_rng([N, 162]), K, ldb)
    out = torch.zeros((M, ldc), device="cuda")
    ro, ci, vals = csr_dev(csr)
    usm.spmm(ro, ci, vals, dev(Bbig)[:, :N], K=K, out=out[:, :N])
    ref, S = oracle_spmm(csr, np.ascontiguousarray(Bbig[:, :N]), "f32")
    C = host(out)
    assert_within(C[:, :N], ref, S, TOL["f32"], f"row-group ld N={N}")
    assert np.all(C[:, N:] == 0), "wrote outside the N columns"


@pytest.mark.parametrize("density", [0.1, 0.6])
def test_spmm_non_finite_b_reaches_only_its_rows(usm, density):
    """Infinities and NaNs in B reach exactly the outputs whose rows hold
    those columns (no product of an absent entry is formed), for the row
    kernel (10% set) and the row-group kernel (60%), as in the oracle."""
    M, K, N = 1300, 1500, 1000
    csr = W.random_csr([M, K, 159], M, K, density)
    B = W.dense(np.random.default_rng(160), K, N)
    B[7, 3] = np.inf
    B[700, 500] = -np.inf
    B[1499, 999] = np.nan
    B[3, 0:4] = [np.inf, -np.inf, np.nan, np.inf]
    ro, ci, vals = csr_dev(csr)
    C = host(usm.spmm(ro, ci, vals, dev(B), K=K))
    ref = oracle.spmm(M, K, csr.row_offsets, csr.col_indices, oracle.widen(csr.values, "f32"),
                      oracle.widen(B, "f32"))
    fin = np.isfinite(ref)
    assert np.array_equal(np.isfinite(C), fin)
    assert np.array_equal(np.isnan(C), np.isnan(ref))
    assert np.array_equal(np.sign(C[np.isinf(ref)]), np.sign(ref[np.isinf(ref)]))
    Bf = np.where(np.isfinite(B), B, 0.0).astype(np.float32)
    ref_f, S = oracle_spmm(csr, Bf, "f32")
    assert_within(np.where(fin, C, 0.0), np.where(fin, ref_f, 0.0), S, TOL["f32"], "finite outputs")
    assert (~fin).sum() > 0


def test_spmm_long_k_fp32(usm):
    """fp32 with more than 128 chunks of K (K = 40000: 193 chunks of 208
    rows) takes the kernel with a second-level accumulator; with every
    value and every B element positive the rounding errors cannot cancel,
    and each element must still be within 1e-5 of its error scale."""
    M, K, N = 64, 40000, 256
    rng = np.random.default_rng(46)
    lengths = np.full(M, K // 2)
    lengths[:8] = K  # some dense rows: every chunk of K contributes
    csr = W.random_csr(47, M, K, 0.0, lengths=lengths)
    csr.values[:] = rng.uniform(0.5, 1.0, csr.nnz).astype(np.float32)
    B = rng.uniform(0.5, 1.0, (K, N)).astype(np.float32)
    ro, ci, vals = csr_dev(csr)
    C = host(usm.spmm(ro, ci, vals, dev(B), K=K, row_swizzle=usm.row_swizzle(ro, K)))
    ref, S = oracle_spmm(csr, B, "f32")
    assert_within(C, ref, S, TOL["f32"], "long-K fp32 spmm")


def test_spmm_swizzle_does_not_change_bits(usm):
    csr = W.random_csr(52, 3000, 800, 0.15)
    B = W.dense(np.random.default_rng(53), 800, 256)
    ro, ci, vals = csr_dev(csr)
    Bd = dev(B)
    a = host(usm.spmm(ro, ci, vals, Bd, K=800))
    b = host(usm.spmm(ro, ci, vals, Bd, K=800, row_swizzle=usm.row_swizzle(ro, 800)))
    c = host(usm.spmm(ro, ci, vals, Bd, K=800))
    assert np.array_equal(a, b) and np.array_equal(a, c)


# ---------------------------------------------------------------------------
# SDDMM, small and ragged, compared in full
# ---------------------------------------------------------------------------
SDDMM_SHAPES = [
    (1, 1, 1, 1.0), (7, 5, 3, 0.6), (37, 61, 64, 0.3), (130, 300, 129, 0.2), (257, 1000, 200, 0.1),
    (300, 129, 513, 0.05), (64, 2100, 128, 0.3), (1000, 50, 8, 0.9), (40, 70, 1000, 0.2),
    # masks at least a quarter full take 256-wide strips: several, the last one ragged
    (200, 500, 600, 0.3), (90, 2100, 300, 0.5),
]


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("M,K,D,density", SDDMM_SHAPES)
@pytest.mark.parametrize("swz", [False, True])
def test_sddmm_small(usm, dtype, M, K, D, density, swz):
    csr = W.random_csr([M, K, D, 61], M, K, density, dtype=dtype)
    rng = np.random.default_rng([M, K, D, 62])
    X = W.dense(rng, M, D, 1.0, dtype)
    Y = W.dense(rng, K, D, 1.0, dtype)
    ro, ci = dev(csr.row_offsets), dev(csr.col_indices)
    perm = usm.row_swizzle(ro, K) if swz else None
    out = host(usm.sddmm(ro, ci, dev(X, dtype), dev(Y, dtype), row_swizzle=perm))
    ref, S, _ = oracle_sddmm(csr, X, Y, dtype)
    assert_within(out, ref, S, TOL[dtype], f"sddmm {dtype} {M}x{K}x{D}")


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("D,density", [(64, 0.2), (128, 0.2), (300, 0.2), (600, 0.3)])
def test_sddmm_integer_valued_bit_exact(usm, dtype, D, density):
    M, K = 300, 700
    csr = W.random_csr([M, K, 63], M, K, density, dtype=dtype, int_valued=True)
    rng = np.random.default_rng(64)
    X = W.dense(rng, M, D, 1.0, dtype, int_valued=True)
    Y = W.dense(rng, K, D, 1.0, dtype, int_valued=True)
    out = host(usm.sddmm(dev(csr.row_offsets), dev(csr.col_indices), dev(X, dtype), dev(Y, dtype)))
    ref, _, _ = oracle_sddmm(csr, X, Y, dtype)
    assert np.array_equal(out.astype(np.float64), ref)


@pytest.mark.parametrize("D", [64 * 128, 65 * 128 + 3, 200 * 128])
def test_sddmm_many_strips_fp32(usm, D):
    """More than 64 column strips: the strip sum adds them in runs of 64,
    then the run totals (D = 65·128 + 3 leaves a ragged strip in a second
    run).  Positive operands so the rounding errors cannot cancel."""
    M, K = 40, 60
    csr = W.random_csr([D, 82], M, K, 0.1)
    rng = np.random.default_rng([D, 83])
    X = rng.uniform(0.5, 1.0, (M, D)).astype(np.float32)
    Y = rng.uniform(0.5, 1.0, (K, D)).astype(np.float32)
    ro, ci = dev(csr.row_offsets), dev(csr.col_indices)
    out = host(usm.sddmm(ro, ci, dev(X), dev(Y)))
    ref, S, _ = oracle_sddmm(csr, X, Y, "f32")
    assert_within(out, ref, S, TOL["f32"], f"sddmm D={D}")


def test_sddmm_bf16_output_rounding(usm):
    import torch
    M, K, D = 200, 300, 96
    csr = W.random_csr(65, M, K, 0.2)
    rng = np.random.default_rng(66)
    X, Y = W.dense(rng, M, D), W.dense(rng, K, D)
    ro, ci = dev(csr.row_offsets), dev(csr.col_indices)
    f32 = usm.sddmm(ro, ci, dev(X), dev(Y))
    b16 = host(usm.sddmm(ro, ci, dev(X), dev(Y), out_dtype=torch.bfloat16))
    # The bf16 output is the fp32 result rounded to nearest even.
    want = f32.to(torch.bfloat16).view(torch.int16).cpu().numpy().view(np.uint16)
    assert np.array_equal(b16, want)


def test_sddmm_row_length_mix_and_empty(usm):
    lengths = np.r_[np.arange(10).repeat(5), [0] * 20, [700, 1500, 32, 33, 31]]
    lengths = np.random.default_rng(67).permutation(lengths)
    M, K, D = lengths.size, 1500, 200
    csr = W.random_csr(68, M, K, 0.0, lengths=lengths)
    rng = np.random.default_rng(69)
    X, Y = W.dense(rng, M, D), W.dense(rng, K, D)
    ro, ci = dev(csr.row_offsets), dev(csr.col_indices)
    out = host(usm.sddmm(ro, ci, dev(X), dev(Y), row_swizzle=usm.row_swizzle(ro, K)))
    ref, S, _ = oracle_sddmm(csr, X, Y, "f32")
    assert_within(out, ref, S, TOL["f32"], "sddmm length mix")


def test_sddmm_adjoint_identity_on_gpu(usm):
    # sum(SpMM(S,B) ⊙ C) = sum(vals ⊙ SDDMM_S(C, B)), both sides from the GPU.
    M, K, N = 500, 400, 96
    csr = W.random_csr(70, M, K, 0.1)
    rng = np.random.default_rng(71)
    B, Cm = W.dense(rng, K, N), W.dense(rng, M, N)
    ro, ci, vals = csr_dev(csr)
    lhs = np.sum(host(usm.spmm(ro, ci, vals, dev(B), K=K)).astype(np.float64) * Cm)
    rhs = np.sum(csr.values.astype(np.float64) * host(usm.sddmm(ro, ci, dev(Cm), dev(B))))
    scale = np.sum(np.abs(csr.values)) * np.abs(B).max() * np.abs(Cm).max() * 4
    assert abs(lhs - rhs) <= 1e-5 * scale


# ---------------------------------------------------------------------------
# Full-size workloads, every element (same launch configuration as bench.py)
# ---------------------------------------------------------------------------
def _spmm_full(usm, p):
    csr = p.csr
    ro, ci, vals = csr_dev(csr)
    perm = usm.row_swizzle(ro, csr.K)
    C = host(usm.spmm(ro, ci, vals, dev(p.B, p.dtype), K=csr.K, row_swizzle=perm))
    ref, S = oracle_spmm(csr, p.B, p.dtype)
    assert_within(C, ref, S, TOL[p.dtype], p.name + " spmm")


def _sddmm_full(usm, p):
    csr = p.csr
    ro, ci = dev(csr.row_offsets), dev(csr.col_indices)
    perm = usm.row_swizzle(ro, csr.K)
    out = host(usm.sddmm(ro, ci, dev(p.X, p.dtype), dev(p.Y, p.dtype), row_swizzle=perm))
    ref, S, _ = oracle_sddmm(csr, p.X, p.Y, p.dtype)
    assert_within(out, ref, S, TOL[p.dtype], p.name + " sddmm")


@pytest.mark.slow
def test_tiny_config_full(usm):
    p = W.tiny()
    csr = p.csr
    ro, ci, vals = csr_dev(csr)
    perm = usm.row_swizzle(ro, csr.K)
    C = host(usm.spmm(ro, ci, vals, dev(p.B), K=csr.K, row_swizzle=perm))
    ref, S = oracle_spmm(csr, p.B, "f32")
    assert_within(C, ref, S, TOL["f32"], "tiny spmm")
    out = host(usm.sddmm(ro, ci, dev(p.X), dev(p.Y), row_swizzle=perm))
    ref, S, _ = oracle_sddmm(csr, p.X, p.Y, "f32")
    assert_within(out, ref, S, TOL["f32"], "tiny sddmm")


@pytest.mark.slow
def test_resnet_config(usm):
    p = W.resnet()
    _spmm_full(usm, p)
    _sddmm_full(usm, p)


@pytest.mark.slow
@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("shape", W.FFN_SHAPES, ids=["4096x1024", "1024x4096"])
@pytest.mark.parametrize("s", W.FFN_SPARSITIES)
def test_ffn_config(usm, dtype, shape, s):
    p = W.ffn(shape[0], shape[1], s, dtype)
    _spmm_full(usm, p)
    _sddmm_full(usm, p)


@pytest.mark.slow
@pytest.mark.parametrize("s", W.LSTM_SPARSITIES)
def test_lstm_config(usm, s):
    _spmm_full(usm, W.lstm(s))


@pytest.mark.slow
def test_attention_chain(usm):
    """SDDMM scores (fp32 accumulation, rounded to bf16), then SpMM of the
    scores with V: the sparse-attention use of the two kernels."""
    import torch
    p = W.attention()
    csr = p.csr
    ro, ci = dev(csr.row_offsets), dev(csr.col_indices)
    perm = usm.row_swizzle(ro, csr.K, seg_rows=p.meta["seq"])
    Q, Kt, V = dev(p.X, "bf16"), dev(p.Y, "bf16"), dev(p.V, "bf16")
    seg = p.meta["seq"]
    s32 = usm.sddmm(ro, ci, Q, Kt, row_swizzle=perm, seg_rows=seg)
    s16 = usm.sddmm(ro, ci, Q, Kt, row_swizzle=perm, out_dtype=torch.bfloat16, seg_rows=seg)
    O = host(usm.spmm(ro, ci, s16, V, K=csr.K, row_swizzle=perm, seg_rows=seg))
    # scores, every nonzero of the 32768-row stack
    ref_s, S_s, _ = oracle_sddmm(csr, p.X, p.Y, "bf16")
    assert_within(host(s32), ref_s, S_s, TOL["bf16"], "attention scores")
    # rounded scores: each is its fp32 score rounded to nearest even, bit for
    # bit (rounded here by the oracle's rounding of the widened fp32 value);
    # against the oracle's own rounding of the exact scores they agree except
    # where the fp32 sum and the exact sum fall on two sides of a rounding
    # boundary, or straddle zero in a cancelling sum
    got16 = host(s16)
    assert np.array_equal(got16, oracle.round_to_bf16(host(s32).astype(np.float64)))
    want16 = oracle.round_to_bf16(ref_s)
    assert np.mean(got16 == want16) > 0.99
    # chain output, every element: the SpMM against the oracle on the GPU's
    # own rounded scores (its actual inputs) ...
    Vw = oracle.widen(p.V, "bf16")
    ro_h, ci_h = csr.row_offsets, csr.col_indices
    g64 = oracle.widen(got16, "bf16")
    ref_o = oracle.spmm(csr.M, csr.K, ro_h, ci_h, g64, Vw)
    S_o = oracle.spmm_error_scale(csr.M, csr.K, ro_h, ci_h, g64, Vw)
    assert_within(O, ref_o, S_o, TOL["bf16"], "attention output")
    # ... and against the oracle's whole chain.  Its scores differ from the
    # GPU's by one bf16 ulp (at most 2^-7 of the score) in under 1% of the
    # entries, which moves an output by at most 2^-7 of its error scale.
    w64 = oracle.widen(want16, "bf16")
    ref_w = oracle.spmm(csr.M, csr.K, ro_h, ci_h, w64, Vw)
    S_w = oracle.spmm_error_scale(csr.M, csr.K, ro_h, ci_h, w64, Vw)
    assert_within(O, ref_w, S_w, TOL["bf16"] + 2.0 ** -7, "attention output vs the oracle chain")


# ---------------------------------------------------------------------------
# Status word and bounded waits
# ---------------------------------------------------------------------------
def test_bounded_wait_times_out_cleanly(usm):
    import torch
    lib = usm.load()
    assert usm.poll_status() == 0
    assert lib.usm_selftest_wait_timeout(2_000_000, usm._stream()) == 0   # 2 ms
    assert usm.poll_status() == -5
    assert usm.poll_status() == 0   # read-and-clear
    # the context is still usable
    x = torch.ones(10, device="cuda")
    assert float(x.sum()) == 10.0


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_calls_leave_csr_untouched(usm, dtype):
    """No call writes to the CSR arrays (or the swizzle, values and dense
    operands) it is given: all compare equal byte for byte afterwards."""
    import torch
    M, K, N, D = 700, 900, 300, 300
    csr = W.random_csr([M, K, 150], M, K, 0.1, dtype=dtype)
    rng = np.random.default_rng(151)
    B, X, Y = W.dense(rng, K, N, 1.0, dtype), W.dense(rng, M, D, 1.0, dtype), W.dense(rng, K, D, 1.0, dtype)
    rod, cid, vd = csr_dev(csr)
    Bd, Xd, Yd = dev(B, dtype), dev(X, dtype), dev(Y, dtype)
    perm = usm.row_swizzle(rod, K, 350)
    before = [t.clone() for t in (rod, cid, vd, Bd, Xd, Yd, perm)]
    usm.spmm(rod, cid, vd, Bd, K=K, row_swizzle=perm, seg_rows=350)
    s = usm.sddmm(rod, cid, Xd, Yd, row_swizzle=perm, seg_rows=350)
    usm.sddmm_general(rod, cid, Xd, Yd, values=vd, row_swizzle=perm, seg_rows=350)
    usm.row_softmax(rod, s)
    usm.csr_transpose(rod, cid, vd, K, with_perm=True)
    usm.csr_validate(rod, cid, K)
    torch.cuda.synchronize()
    for a, b in zip(before, (rod, cid, vd, Bd, Xd, Yd, perm)):
        assert torch.equal(a.view(torch.uint8) if a.dtype == torch.bfloat16 else a,
                           b.view(torch.uint8) if b.dtype == torch.bfloat16 else b)
    assert usm.poll_status() == 0


def test_concurrent_streams_match_one_stream(usm):
    """Independent problems dealt over three streams at once (as the bench
    runs its step) give the same bits as the same calls on one stream: the
    kernels keep no state outside their arguments."""
    import torch
    probs = []
    for i, (M, K, dt, dens) in enumerate([(600, 900, "f32", 0.3), (900, 600, "bf16", 0.1), (400, 1500, "f32", 0.05),
                                          (700, 700, "bf16", 0.3), (500, 800, "f32", 0.2), (300, 2000, "bf16", 0.25)]):
        csr = W.random_csr([M, K, 170 + i], M, K, dens, dtype=dt)
        rng = np.random.default_rng(180 + i)
        N = 300
        d = dict(csr=csr, dt=dt, K=K, B=dev(W.dense(rng, K, N, 1.0, dt), dt), X=dev(W.dense(rng, M, N, 1.0, dt), dt),
                 Y=dev(W.dense(rng, K, N, 1.0, dt), dt))
        d["ro"], d["ci"], d["v"] = csr_dev(csr)
        d["perm"] = usm.row_swizzle(d["ro"], K)
        probs.append(d)

    def run_all(streams):
        outs = [None] * len(probs)
        main = torch.cuda.current_stream()
        for s in streams:
            s.wait_stream(main)
        for j, d in enumerate(probs):
            with torch.cuda.stream(streams[j % len(streams)]):
                C = usm.spmm(d["ro"], d["ci"], d["v"], d["B"], K=d["K"], row_swizzle=d["perm"])
                S = usm.sddmm(d["ro"], d["ci"], d["X"], d["Y"], row_swizzle=d["perm"])
                outs[j] = (C, S)
        for s in streams:
            main.wait_stream(s)
        torch.cuda.synchronize()
        return [(host(C), host(S)) for C, S in outs]

    one = run_all([torch.cuda.current_stream()])
    many = run_all([torch.cuda.Stream() for _ in range(3)])
    for j, ((c1, s1), (c3, s3)) in enumerate(zip(one, many)):
        assert np.array_equal(c1, c3) and np.array_equal(s1, s3), j
    assert usm.poll_status() == 0


def test_misaligned_pointer_rejected(usm):
    import torch
    csr = W.random_csr(120, 10, 10, 0.3)
    ro, ci, vals = csr_dev(csr)
    B = torch.zeros((10, 9), device="cuda")[:, 1:]   # offset by 4 bytes, ld 9
    C = torch.zeros((10, 8), device="cuda")
    lib = usm.load()
    code = lib.csr_spmm(10, 10, 8, csr.nnz, ro.data_ptr(), ci.data_ptr(), vals.data_ptr(), None, 0,
                        B.data_ptr(), 9, C.data_ptr(), 8, 0, usm._stream())
    assert code == -2
    # the binding pads such operands itself and gets the right answer
    Cb = host(usm.spmm(ro, ci, vals, B, K=10))
    assert np.array_equal(Cb, np.zeros((10, 8), np.float32))


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_scheduler_does_not_change_bits(usm, dtype):
    """Block-diagonal matrix with skewed (lognormal) rows: the results are
    bit-identical with no swizzle, a global swizzle, and per-block swizzle
    and schedule (each output is computed by one unit in a fixed order)."""
    blocks, seq, D = 5, 700, 96
    rng = np.random.default_rng(130)
    lens = W.lengths_lognormal(rng, blocks * seq, seq, 60.0, 0.8)
    base = (np.arange(blocks * seq) // seq) * seq
    ro, ci = W.csr_from_lengths(rng, lens, seq, col_base=base)
    vals = W.values_for(rng, int(ro[-1]), 1.0, dtype)
    csr = W.CSR(blocks * seq, blocks * seq, ro, ci, vals, dtype, seg_rows=seq)
    B = W.dense(rng, csr.K, D, 1.0, dtype)
    X = W.dense(rng, csr.M, D, 1.0, dtype)
    rod, cid, vd = csr_dev(csr)
    Bd, Xd = dev(B, dtype), dev(X, dtype)
    variants = [(None, 0), (usm.row_swizzle(rod, csr.K), 0), (usm.row_swizzle(rod, csr.K, seq), seq),
                (usm.row_swizzle(rod, csr.K, seq), 0)]
    Cs = [host(usm.spmm(rod, cid, vd, Bd, K=csr.K, row_swizzle=p, seg_rows=s)) for p, s in variants]
    Ss = [host(usm.sddmm(rod, cid, Xd, Bd, row_swizzle=p, seg_rows=s)) for p, s in variants]
    for c in Cs[1:]:
        assert np.array_equal(c, Cs[0])
    for o in Ss[1:]:
        assert np.array_equal(o, Ss[0])
    ref, S = oracle_spmm(csr, B, dtype)
    assert_within(Cs[0], ref, S, TOL[dtype], "block-diagonal spmm")
    ref, S, _ = oracle_sddmm(csr, X, B, dtype)
    assert_within(Ss[0], ref, S, TOL[dtype], "block-diagonal sddmm")


@pytest.fixture
def schedule(usm):
    """Sets the launch-shape override for a test and always clears it."""
    yield usm.set_schedule_override
    usm.set_schedule_override(0, 0, 0)


# (rows per warp, tiles per block, K splits); 0 keeps the library's choice.
# Tile counts above the fewest that hold a block give tiles of fewer rows
# (the launch model's wave-filling choice); (0, t, s) forces tiles and splits
# under the model's own rows per warp.
SDDMM_SCHEDULES = [(0, 0, 0), (1, 0, 1), (2, 0, 5), (8, 0, 3), (32, 0, 1), (4, 40, 2), (16, 0, 11), (1, 0, 16),
                   (2, 44, 1), (16, 3, 0), (0, 25, 0), (0, 11, 3)]


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("seg", [0, 350])
def test_sddmm_schedules_do_not_change_bits(usm, schedule, dtype, seg):
    """Rows per warp, tiles per block and K splits change which CTA computes
    a nonzero, never the order of its terms: the outputs are bit-identical
    (D = 300 spans three strips; seg = 350 makes a block-diagonal schedule)."""
    M, K, D = 700, 3000, 300
    csr = W.random_csr([M, K, 140], M, K, 0.1, dtype=dtype)
    rng = np.random.default_rng(141)
    X, Y = W.dense(rng, M, D, 1.0, dtype), W.dense(rng, K, D, 1.0, dtype)
    rod, cid = dev(csr.row_offsets), dev(csr.col_indices)
    Xd, Yd = dev(X, dtype), dev(Y, dtype)
    perm = usm.row_swizzle(rod, K, seg)
    outs = []
    for r, t, s in SDDMM_SCHEDULES:
        schedule(r, t, s)
        outs.append(host(usm.sddmm(rod, cid, Xd, Yd, row_swizzle=perm, seg_rows=seg)))
    for (r, t, s), o in zip(SDDMM_SCHEDULES[1:], outs[1:]):
        assert np.array_equal(o, outs[0]), (r, t, s)
    ref, S, _ = oracle_sddmm(csr, X, Y, dtype)
    assert_within(outs[0], ref, S, TOL[dtype], "sddmm under forced schedules")


SPMM_SCHEDULES = [(0, 0, 0), (2, 0, 0), (4, 0, 0), (2, 50, 0), (4, 7, 0), (0, 44, 1), (0, 9, 0), (0, 30, 0)]


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("N", [64, 300])
@pytest.mark.parametrize("seg", [0, 350])
def test_spmm_schedules_do_not_change_bits(usm, schedule, dtype, N, seg):
    """Rows per warp and tiles per block move rows between CTAs and warps,
    not the order of a row's terms: the outputs are bit-identical."""
    M, K = 700, 3000
    csr = W.random_csr([M, K, N, 142], M, K, 0.1, dtype=dtype)
    B = W.dense(np.random.default_rng(143), K, N, 1.0, dtype)
    rod, cid, vd = csr_dev(csr)
    Bd = dev(B, dtype)
    perm = usm.row_swizzle(rod, K, seg)
    outs = []
    for r, t, s in SPMM_SCHEDULES:
        schedule(r, t, s)
        outs.append(host(usm.spmm(rod, cid, vd, Bd, K=K, row_swizzle=perm, seg_rows=seg)))
    for (r, t, s), c in zip(SPMM_SCHEDULES[1:], outs[1:]):
        assert np.array_equal(c, outs[0]), (r, t, s)
    ref, S = oracle_spmm(csr, B, dtype)
    assert_within(outs[0], ref, S, TOL[dtype], "spmm under forced schedules")


@pytest.mark.parametrize("N", [100, 300])
def test_spmm_sparse_mask_schedules_do_not_change_bits(usm, schedule, N):
    """fp32 masks under 7% set (and, for N <= 128, at least 3%: sparser ones
    take the gather kernel) run 128-wide strips with 4 or 8 rows a warp:
    every forced schedule gives the same bits, and the oracle's result."""
    M, K = 900, 3000
    csr = W.random_csr([M, K, N, 146], M, K, 0.05)
    B = W.dense(np.random.default_rng(147), K, N)
    rod, cid, vd = csr_dev(csr)
    Bd = dev(B)
    perm = usm.row_swizzle(rod, K)
    outs = []
    for r, t, s_ in [(0, 0, 0), (4, 0, 0), (8, 0, 0), (8, 20, 0), (4, 9, 0), (0, 30, 0)]:
        schedule(r, t, s_)
        outs.append(host(usm.spmm(rod, cid, vd, Bd, K=K, row_swizzle=perm)))
    for c in outs[1:]:
        assert np.array_equal(c, outs[0])
    schedule(2, 0, 0)  # no kernel with 2 rows a warp for these masks
    with pytest.raises(RuntimeError, match="UNSUPPORTED"):
        usm.spmm(rod, cid, vd, Bd, K=K, row_swizzle=perm)
    ref, S = oracle_spmm(csr, B, "f32")
    assert_within(outs[0], ref, S, TOL["f32"], "sparse-mask spmm")


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("N", [4, 64, 100, 128])
def test_spmm_gather_path(usm, schedule, dtype, N):
    """fp32 masks under 3% set with N <= 128 take the kernel that gathers the rows
    of B without staging: every element against the oracle, every column
    pass edge (N = 4, 100) included, and against the staged kernels (run by
    forcing a schedule) within the same tolerance."""
    M, K = 3000, 4096
    lengths = np.random.default_rng([N, 148]).binomial(K, 0.02, M)
    lengths[:7] = 0
    lengths[7] = 300   # a row longer than a window of 32
    csr = W.random_csr([M, K, N, 149], M, K, 0.0, dtype=dtype, lengths=lengths)
    B = W.dense(np.random.default_rng(150), K, N, 1.0, dtype)
    rod, cid, vd = csr_dev(csr)
    Bd = dev(B, dtype)
    perm = usm.row_swizzle(rod, K)
    C = host(usm.spmm(rod, cid, vd, Bd, K=K, row_swizzle=perm))
    ref, S = oracle_spmm(csr, B, dtype)
    assert_within(C, ref, S, TOL[dtype], f"gather spmm {dtype} N={N}")
    schedule(4, 0, 0)
    staged = host(usm.spmm(rod, cid, vd, Bd, K=K, row_swizzle=perm))
    assert_within(staged, ref, S, TOL[dtype], f"staged spmm {dtype} N={N}")
    schedule(0, 0, 0)
    again = host(usm.spmm(rod, cid, vd, Bd, K=K))  # no swizzle: same bits (one row a warp)
    assert np.array_equal(again, C)


def test_spmm_rejects_schedules_it_has_no_kernel_for(usm, schedule):
    csr = W.random_csr(144, 100, 200, 0.1)
    rod, cid, vd = csr_dev(csr)
    Bd = dev(W.dense(np.random.default_rng(145), 200, 64))
    for r, t, s in [(8, 0, 0), (1, 0, 0), (0, 0, 3)]:
        schedule(r, t, s)
        with pytest.raises(RuntimeError, match="UNSUPPORTED"):
            usm.spmm(rod, cid, vd, Bd, K=200)
