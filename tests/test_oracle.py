"""Pins for the CPU oracle: each check ties it to something other than itself
(hand-worked examples, numpy's dense matmul and sort, closed forms,
invariants), chosen so a dropped term, a wrong index, a transposed operand or
a reversed tie-break fails at least one of them."""
import json
import os

import numpy as np
import pytest

import oracle
import workloads as W


def _load(golden_dir, name):
    with open(os.path.join(golden_dir, name)) as f:
        return json.load(f)


def densify(M, K, ro, ci, vals):
    A = np.zeros((M, K), dtype=np.float64)
    for r in range(M):
        for p in range(ro[r], ro[r + 1]):
            A[r, ci[p]] = vals[p]
    return A


def mask_of(M, K, ro, ci):
    return densify(M, K, ro, ci, np.ones(len(ci)))


# ---------------------------------------------------------------------------
# Hand-worked examples (tests/golden)
# ---------------------------------------------------------------------------
def test_golden_spmm(golden_dir):
    g = _load(golden_dir, "spmm_worked_example.json")
    C = oracle.spmm(g["M"], g["K"], g["row_offsets"], g["col_indices"], g["values"], np.array(g["B"], float))
    assert np.array_equal(C, np.array(g["C"]))


def test_golden_sddmm(golden_dir):
    g = _load(golden_dir, "sddmm_worked_example.json")
    X, Y = np.array(g["X"], float), np.array(g["Y"], float)
    out = oracle.sddmm(g["M"], g["K"], g["row_offsets"], g["col_indices"], X, Y)
    assert np.array_equal(out, np.array(g["out"]))
    gen = oracle.sddmm_general(g["M"], g["K"], g["row_offsets"], g["col_indices"], g["values"], True, X, Y, True)
    assert np.array_equal(gen, np.array(g["out_scaled_by_values"]))
    # Non-transposed form: pass Yᵀ (D×K) and say so.
    gen_nt = oracle.sddmm_general(g["M"], g["K"], g["row_offsets"], g["col_indices"], None, False,
                                  X, np.ascontiguousarray(Y.T), False)
    assert np.array_equal(gen_nt, np.array(g["out"]))


def test_golden_swizzle(golden_dir):
    g = _load(golden_dir, "row_swizzle_worked_example.json")
    for case in g["cases"]:
        perm = oracle.row_swizzle(case["row_offsets"], case["seg_rows"])
        assert perm.tolist() == case["perm"], case


def test_golden_transpose(golden_dir):
    g = _load(golden_dir, "csr_transpose_worked_example.json")
    ro_t, ci_t, a_t = oracle.csr_transpose(g["M"], g["K"], g["row_offsets"], g["col_indices"], g["values"])
    assert ro_t.tolist() == g["t_row_offsets"]
    assert ci_t.tolist() == g["t_col_indices"]
    assert a_t.tolist() == g["t_values"]


def test_golden_bf16_rounding(golden_dir):
    g = _load(golden_dir, "bf16_rounding_examples.json")
    xs = np.array([c[0] for c in g["cases"]], dtype=np.float64)
    want = [int(c[1], 16) for c in g["cases"]]
    assert oracle.round_to_bf16(xs).tolist() == want


def test_golden_softmax(golden_dir):
    g = _load(golden_dir, "csr_softmax_worked_example.json")
    got = oracle.csr_softmax(g["row_offsets"], g["scores"])
    np.testing.assert_allclose(got, g["probs"], rtol=1e-15, atol=0)


# ---------------------------------------------------------------------------
# Dense brute force (numpy's matmul is the independent routine)
# ---------------------------------------------------------------------------
SHAPES = [(1, 1, 1), (7, 5, 3), (33, 17, 9), (64, 64, 64), (40, 3, 70), (5, 64, 1)]
DENSITIES = [0.0, 0.05, 0.3, 1.0]


@pytest.mark.parametrize("M,K,N", SHAPES)
@pytest.mark.parametrize("density", DENSITIES)
def test_spmm_vs_dense(M, K, N, density):
    csr = W.random_csr([M, K, N, int(density * 100)], M, K, density)
    rng = np.random.default_rng([M, K, N, 7])
    B = rng.standard_normal((K, N))
    A = densify(M, K, csr.row_offsets, csr.col_indices, csr.values.astype(np.float64))
    C = oracle.spmm(M, K, csr.row_offsets, csr.col_indices, csr.values.astype(np.float64), B)
    np.testing.assert_allclose(C, A @ B, rtol=1e-12, atol=1e-12)


@pytest.mark.parametrize("M,K,D", SHAPES)
@pytest.mark.parametrize("density", DENSITIES)
def test_sddmm_vs_dense_masked(M, K, D, density):
    csr = W.random_csr([M, K, D, int(density * 100), 1], M, K, density)
    rng = np.random.default_rng([M, K, D, 8])
    X, Y = rng.standard_normal((M, D)), rng.standard_normal((K, D))
    out = oracle.sddmm(M, K, csr.row_offsets, csr.col_indices, X, Y)
    full = X @ Y.T
    rows = np.repeat(np.arange(M), np.diff(csr.row_offsets))
    np.testing.assert_allclose(out, full[rows, csr.col_indices], rtol=1e-12, atol=1e-12)
    # mask ⊙ (X·Yᵀ) densified equals the densified SDDMM output
    dense_out = densify(M, K, csr.row_offsets, csr.col_indices, out)
    np.testing.assert_allclose(dense_out, mask_of(M, K, csr.row_offsets, csr.col_indices) * full,
                               rtol=1e-12, atol=1e-12)


@pytest.mark.parametrize("scale,ytr", [(False, True), (True, True), (True, False), (False, False)])
def test_sddmm_general_vs_dense(scale, ytr):
    M, K, D = 19, 23, 11
    csr = W.random_csr([5, 5], M, K, 0.4)
    rng = np.random.default_rng(99)
    X, Y = rng.standard_normal((M, D)), rng.standard_normal((K, D))
    vals = csr.values.astype(np.float64)
    Yarg = Y if ytr else np.ascontiguousarray(Y.T)
    out = oracle.sddmm_general(M, K, csr.row_offsets, csr.col_indices, vals, scale, X, Yarg, ytr)
    rows = np.repeat(np.arange(M), np.diff(csr.row_offsets))
    want = (X @ Y.T)[rows, csr.col_indices] * (vals if scale else 1.0)
    np.testing.assert_allclose(out, want, rtol=1e-12, atol=1e-12)


# ---------------------------------------------------------------------------
# Special matrices (bit-exact)
# ---------------------------------------------------------------------------
def test_identity_bit_exact():
    n, N = 50, 13
    B = np.random.default_rng(1).standard_normal((n, N))
    ro = np.arange(n + 1, dtype=np.int32)
    ci = np.arange(n, dtype=np.int32)
    C = oracle.spmm(n, n, ro, ci, np.ones(n), B)
    assert np.array_equal(C, B)
    X = np.random.default_rng(2).standard_normal((n, N))
    out = oracle.sddmm(n, n, ro, ci, X, B)
    np.testing.assert_allclose(out, np.einsum("ij,ij->i", X, B), rtol=1e-13)


def test_permutation_bit_exact():
    n, N = 64, 9
    perm = np.random.default_rng(3).permutation(n).astype(np.int32)
    B = np.random.default_rng(4).standard_normal((n, N))
    ro = np.arange(n + 1, dtype=np.int32)
    C = oracle.spmm(n, n, ro, perm, np.ones(n), B)
    assert np.array_equal(C, B[perm])


# ---------------------------------------------------------------------------
# Adjoint identity: sum(SpMM(S,B) ⊙ C) = sum(vals(S) ⊙ SDDMM_S(C, B))
# (with Y = B, K×D, the SDDMM uses it transposed)
# ---------------------------------------------------------------------------
@pytest.mark.parametrize("M,K,N,density", [(30, 40, 7, 0.2), (64, 16, 33, 0.7), (9, 128, 5, 0.05)])
def test_adjoint_identity(M, K, N, density):
    csr = W.random_csr([M, K, 11], M, K, density)
    rng = np.random.default_rng([M, K, 12])
    B, Cm = rng.standard_normal((K, N)), rng.standard_normal((M, N))
    vals = csr.values.astype(np.float64)
    lhs = np.sum(oracle.spmm(M, K, csr.row_offsets, csr.col_indices, vals, B) * Cm)
    rhs = np.sum(vals * oracle.sddmm(M, K, csr.row_offsets, csr.col_indices, Cm, B))
    scale = np.sum(np.abs(oracle.spmm(M, K, csr.row_offsets, csr.col_indices, np.abs(vals), np.abs(B))) * np.abs(Cm))
    assert abs(lhs - rhs) <= 1e-12 * max(scale, 1.0)


# ---------------------------------------------------------------------------
# Integer-valued inputs: every sum is an exact integer in fp64
# ---------------------------------------------------------------------------
def test_integer_exactness():
    M, K, N = 37, 53, 21
    csr = W.random_csr([13], M, K, 0.3, int_valued=True)
    rng = np.random.default_rng(14)
    B = rng.integers(-4, 5, size=(K, N)).astype(np.float64)
    X = rng.integers(-4, 5, size=(M, N)).astype(np.float64)
    A = densify(M, K, csr.row_offsets, csr.col_indices, csr.values.astype(np.float64))
    C = oracle.spmm(M, K, csr.row_offsets, csr.col_indices, csr.values.astype(np.float64), B)
    assert np.array_equal(C, (A.astype(np.int64) @ B.astype(np.int64)).astype(np.float64))
    out = oracle.sddmm(M, K, csr.row_offsets, csr.col_indices, X, B)
    rows = np.repeat(np.arange(M), np.diff(csr.row_offsets))
    full = X.astype(np.int64) @ B.astype(np.int64).T
    assert np.array_equal(out, full[rows, csr.col_indices].astype(np.float64))


def test_linearity():
    M, K, N = 25, 31, 6
    csr = W.random_csr([15], M, K, 0.25)
    rng = np.random.default_rng(16)
    B1, B2 = rng.standard_normal((K, N)), rng.standard_normal((K, N))
    v = csr.values.astype(np.float64)
    f = lambda B: oracle.spmm(M, K, csr.row_offsets, csr.col_indices, v, B)
    np.testing.assert_allclose(f(B1 + B2), f(B1) + f(B2), rtol=1e-12, atol=1e-12)


def test_error_scale_is_abs_spmm():
    M, K, N = 12, 9, 4
    csr = W.random_csr([17], M, K, 0.5)
    B = np.random.default_rng(18).standard_normal((K, N))
    v = csr.values.astype(np.float64)
    S = oracle.spmm_error_scale(M, K, csr.row_offsets, csr.col_indices, v, B)
    A = densify(M, K, csr.row_offsets, csr.col_indices, v)
    np.testing.assert_allclose(S, np.abs(A) @ np.abs(B), rtol=1e-13)
    assert np.all(S >= np.abs(A @ B) - 1e-12)


# ---------------------------------------------------------------------------
# Row swizzle
# ---------------------------------------------------------------------------
@pytest.mark.parametrize("M,K,seg", [(1, 4, 0), (100, 50, 0), (1000, 300, 0), (999, 64, 100), (512, 8, 512), (77, 10, 1)])
def test_swizzle_vs_lexsort(M, K, seg):
    csr = W.random_csr([M, K, 19], M, K, 0.15)
    lens = np.diff(csr.row_offsets)
    perm = oracle.row_swizzle(csr.row_offsets, seg)
    s = seg if 0 < seg <= M else M
    want = []
    for b in range(0, M, s):
        idx = np.arange(b, min(M, b + s))
        want.extend(idx[np.lexsort((idx, -lens[idx]))].tolist())
    assert perm.tolist() == want
    # invariants: a bijection, non-increasing lengths inside each block,
    # ascending row ids among equal lengths
    assert sorted(perm.tolist()) == list(range(M))
    for b in range(0, M, s):
        blk = perm[b:b + s]
        L = lens[blk]
        assert np.all(np.diff(L) <= 0)
        ties = (np.diff(L) == 0)
        assert np.all(np.diff(blk)[ties] > 0)


def test_swizzle_all_equal_is_identity():
    ro = np.arange(0, 3 * 41, 3, dtype=np.int32)
    assert oracle.row_swizzle(ro).tolist() == list(range(40))


# ---------------------------------------------------------------------------
# CSR transpose
# ---------------------------------------------------------------------------
@pytest.mark.parametrize("M,K,density", [(20, 30, 0.2), (64, 1, 0.5), (1, 64, 0.5), (50, 50, 0.0), (33, 47, 1.0)])
def test_transpose_vs_dense(M, K, density):
    csr = W.random_csr([M, K, 20], M, K, density)
    v = csr.values.astype(np.float64)
    ro_t, ci_t, a_t = oracle.csr_transpose(M, K, csr.row_offsets, csr.col_indices, v)
    assert oracle.csr_check(K, M, ro_t, ci_t) == 0
    A = densify(M, K, csr.row_offsets, csr.col_indices, v)
    assert np.array_equal(densify(K, M, ro_t, ci_t, a_t), A.T)
    ro2, ci2, a2 = oracle.csr_transpose(K, M, ro_t, ci_t, a_t)
    assert np.array_equal(ro2, csr.row_offsets) and np.array_equal(ci2, csr.col_indices)
    assert np.array_equal(a2, v)


# ---------------------------------------------------------------------------
# Softmax against scipy on each row
# ---------------------------------------------------------------------------
def test_softmax_vs_scipy():
    scipy_special = pytest.importorskip("scipy.special")
    csr = W.random_csr([21], 40, 60, 0.2)
    s = np.random.default_rng(22).standard_normal(csr.nnz) * 5
    got = oracle.csr_softmax(csr.row_offsets, s)
    for r in range(40):
        b, e = csr.row_offsets[r], csr.row_offsets[r + 1]
        if b < e:
            np.testing.assert_allclose(got[b:e], scipy_special.softmax(s[b:e]), rtol=1e-13)


# ---------------------------------------------------------------------------
# bf16 rounding against torch's conversion (an independent library routine)
# ---------------------------------------------------------------------------
def test_bf16_rounding_vs_torch():
    torch = pytest.importorskip("torch")
    x = np.random.default_rng(23).standard_normal(20000).astype(np.float32).astype(np.float64)
    x[:10] = [1.00390625, 1.01171875, -1.00390625, 0.0, -0.0, 2.0 ** -20, 3.0, -7.0, 1e4, -1e-4]
    got = oracle.round_to_bf16(x)
    want = torch.from_numpy(x.astype(np.float32)).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(got, want)


def test_widen_bf16_exact():
    bits = np.array([0x3F80, 0xC020, 0x3DCD, 0x0000, 0x8000], dtype=np.uint16)
    assert oracle.widen(bits, "bf16").tolist() == [1.0, -2.5, 0.10009765625, 0.0, -0.0]


# ---------------------------------------------------------------------------
# CSR contract checker (host-side fault injection: corrupted CSRs)
# ---------------------------------------------------------------------------
def test_csr_check_rejects_corruption():
    g = dict(M=3, K=4, ro=[0, 2, 2, 5], ci=[0, 3, 1, 2, 3])
    assert oracle.csr_check(g["M"], g["K"], g["ro"], g["ci"]) == 0
    assert oracle.csr_check(3, 4, [1, 2, 2, 5], g["ci"]) == -2          # ro[0] != 0
    assert oracle.csr_check(3, 4, [0, 2, 1, 5], g["ci"]) == -3          # decreasing
    assert oracle.csr_check(3, 4, [0, 2, 2, 4], g["ci"][:4]) == 0       # consistent shorter
    assert oracle.csr_check(3, 4, [0, 2, 2, 5], [0, 4, 1, 2, 3]) == -5  # col out of range
    assert oracle.csr_check(3, 4, [0, 2, 2, 5], [0, 3, 2, 2, 3]) == -6  # duplicate col
    assert oracle.csr_check(3, 4, [0, 2, 2, 5], [3, 0, 1, 2, 3]) == -6  # unsorted
    assert oracle.csr_check(3, 4, [0, 2, 2, 4], g["ci"]) == -4          # row_offsets[M] != nnz = 5
    assert oracle.csr_check(3, 4, [0, 2, 2, 6], g["ci"]) == -4          # past the arrays: not scanned
    assert oracle.csr_check(3, 4, [1, 0, 2, 4], g["ci"]) == -2          # first rule wins
    assert oracle.csr_check(3, 4, [0, 2, 1, 4], g["ci"]) == -3          # decrease before the last offset
    # entries: the first bad nonzero decides; at one position the range test first
    assert oracle.csr_check(3, 4, [0, 2, 2, 5], [1, 0, 1, 2, 9]) == -6  # order at p=1 before range at p=4
    assert oracle.csr_check(3, 4, [0, 2, 2, 5], [0, 3, 1, 9, 3]) == -5  # range at p=3 before order at p=4
    assert oracle.csr_check(3, 4, [0, 2, 2, 5], [2, -1, 1, 2, 3]) == -5  # p=1 fails both: range
    assert oracle.csr_check(0, 4, [0], []) == 0 and oracle.csr_check(0, 4, [0], [5]) == -4


def test_workload_generators_produce_valid_csr():
    for p in [W.tiny(), W.resnet(with_sddmm=False)]:
        c = p.csr
        assert oracle.csr_check(c.M, c.K, c.row_offsets, c.col_indices) == 0


def test_thread_count_is_per_call():
    """A call pinned to one thread does not shrink later all-cores calls,
    and every thread count gives the same bits (fixed per-row order)."""
    csr = W.random_csr([64, 48, 7], 64, 48, 0.2)
    B = np.random.default_rng(7).standard_normal((48, 16))
    default = oracle.max_threads()
    one = oracle.spmm(64, 48, csr.row_offsets, csr.col_indices, csr.values.astype(np.float64), B, 1)
    assert oracle.max_threads() == default
    allc = oracle.spmm(64, 48, csr.row_offsets, csr.col_indices, csr.values.astype(np.float64), B, 0)
    assert np.array_equal(one, allc)
