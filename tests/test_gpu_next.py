"""The next rows of the path, against the oracle through the C ABI:
CSR transpose and the input-gradient SpMM (bit-exact structure), the
general SDDMM (scaling and operand orientation), the row softmax, the
sparse-attention chain with softmax, and the sparse layer's training step
(forward SpMM, weight-gradient SDDMM, input-gradient SpMM on Aᵀ)."""
import numpy as np
import pytest

import oracle
import workloads as W
from parity_util import TOL, assert_within, dev, host, oracle_sddmm, oracle_spmm

pytestmark = pytest.mark.gpu


def csr_dev(csr):
    return dev(csr.row_offsets), dev(csr.col_indices), dev(csr.values, csr.dtype)


# ---------------------------------------------------------------------------
# f1: CSR transpose (bit-exact) and the input gradient
# ---------------------------------------------------------------------------
TRANSPOSE_CASES = [
    ("ragged", lambda dt: W.random_csr(1, 700, 300, 0.1, dtype=dt)),
    ("empty_rows_and_cols", lambda dt: W.random_csr(2, 500, 5000, 0.0, dtype=dt,
                                                    lengths=np.r_[np.zeros(250, int), np.full(250, 7)])),
    ("one_row", lambda dt: W.random_csr(3, 1, 1000, 0.5, dtype=dt)),
    ("one_col", lambda dt: W.random_csr(4, 1000, 1, 0.5, dtype=dt)),
    ("dense", lambda dt: W.random_csr(5, 64, 64, 1.0, dtype=dt)),
    ("no_nonzeros", lambda dt: W.random_csr(6, 100, 50, 0.0, dtype=dt)),
    ("multi_tile", lambda dt: W.random_csr(7, 3000, 2000, 0.05, dtype=dt)),
]


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("name,make", TRANSPOSE_CASES, ids=[c[0] for c in TRANSPOSE_CASES])
def test_transpose_bit_exact(usm, dtype, name, make):
    csr = make(dtype)
    ro, ci, vals = csr_dev(csr)
    ro_t, ci_t, v_t, perm = usm.csr_transpose(ro, ci, vals, csr.K, with_perm=True)
    w_ro, w_ci, w_v = oracle.csr_transpose(csr.M, csr.K, csr.row_offsets, csr.col_indices,
                                           oracle.widen(csr.values, dtype))
    assert np.array_equal(host(ro_t), w_ro)
    assert np.array_equal(host(ci_t), w_ci)
    assert np.array_equal(oracle.widen(host(v_t), dtype), w_v)
    assert np.array_equal(host(v_t), csr.values[host(perm)])


def test_transpose_full_configs(usm):
    for csr in [W.ffn(4096, 1024, 70, "f32", with_spmm=False, with_sddmm=False).csr, W.lstm(50).csr,
                W.attention().csr]:
        ro, ci, vals = csr_dev(csr)
        ro_t, ci_t, v_t = usm.csr_transpose(ro, ci, vals, csr.K)
        w_ro, w_ci, w_v = oracle.csr_transpose(csr.M, csr.K, csr.row_offsets, csr.col_indices,
                                               oracle.widen(csr.values, csr.dtype))
        assert np.array_equal(host(ro_t), w_ro)
        assert np.array_equal(host(ci_t), w_ci)
        assert np.array_equal(oracle.widen(host(v_t), csr.dtype), w_v)


def test_permute_values_follows_new_weights(usm):
    csr = W.random_csr(8, 900, 600, 0.08)
    ro, ci, vals = csr_dev(csr)
    _, _, _, perm = usm.csr_transpose(ro, ci, vals, csr.K, with_perm=True)
    new_vals = np.random.default_rng(9).standard_normal(csr.nnz).astype(np.float32)
    got = host(usm.csr_permute_values(perm, dev(new_vals)))
    _, _, want = oracle.csr_transpose(csr.M, csr.K, csr.row_offsets, csr.col_indices, new_vals.astype(np.float64))
    assert np.array_equal(got.astype(np.float64), want)


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_input_gradient_spmm_on_transpose(usm, dtype):
    M, K, N = 1500, 700, 136
    csr = W.random_csr(10, M, K, 0.1, dtype=dtype)
    dC = W.dense(np.random.default_rng(11), M, N, 1.0, dtype)
    ro, ci, vals = csr_dev(csr)
    ro_t, ci_t, v_t = usm.csr_transpose(ro, ci, vals, K)
    dB = host(usm.spmm(ro_t, ci_t, v_t, dev(dC, dtype), K=M, row_swizzle=usm.row_swizzle(ro_t, M)))
    t_ro, t_ci, t_v = oracle.csr_transpose(M, K, csr.row_offsets, csr.col_indices, oracle.widen(csr.values, dtype))
    dCw = oracle.widen(dC, dtype)
    ref = oracle.spmm(K, M, t_ro, t_ci, t_v, dCw)
    S = oracle.spmm_error_scale(K, M, t_ro, t_ci, t_v, dCw)
    assert_within(dB, ref, S, TOL[dtype], "input gradient")


# ---------------------------------------------------------------------------
# f2: general SDDMM
# ---------------------------------------------------------------------------
@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("scale", [False, True])
@pytest.mark.parametrize("ytr", [True, False])
@pytest.mark.parametrize("M,K,D", [(300, 200, 64), (257, 333, 300), (40, 1000, 129)])
def test_sddmm_general(usm, dtype, scale, ytr, M, K, D):
    csr = W.random_csr([M, K, D, 12], M, K, 0.15, dtype=dtype)
    rng = np.random.default_rng([M, K, D, 13])
    X = W.dense(rng, M, D, 1.0, dtype)
    Y = W.dense(rng, K, D, 1.0, dtype)
    Yarg = Y if ytr else np.ascontiguousarray(Y.T)
    ro, ci, vals = csr_dev(csr)
    out = host(usm.sddmm_general(ro, ci, dev(X, dtype), dev(Yarg, dtype), values=vals if scale else None,
                                 y_transposed=ytr))
    a = oracle.widen(csr.values, dtype)
    ref = oracle.sddmm_general(M, K, csr.row_offsets, csr.col_indices, a, scale, oracle.widen(X, dtype),
                               oracle.widen(Yarg, dtype), ytr)
    S = oracle.sddmm_error_scale(M, K, csr.row_offsets, csr.col_indices, oracle.widen(X, dtype),
                                 oracle.widen(Y, dtype)) * (np.abs(a) if scale else 1.0)
    assert_within(out, ref, S, TOL[dtype], f"general sddmm scale={scale} ytr={ytr}")


def test_sddmm_general_matches_specialised_form(usm):
    csr = W.random_csr(14, 500, 400, 0.1)
    rng = np.random.default_rng(15)
    X, Y = W.dense(rng, 500, 200), W.dense(rng, 400, 200)
    ro, ci, _ = csr_dev(csr)
    a = host(usm.sddmm(ro, ci, dev(X), dev(Y)))
    b = host(usm.sddmm_general(ro, ci, dev(X), dev(Y)))
    assert np.array_equal(a, b)


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("scale", [False, True])
@pytest.mark.parametrize("nnz_mod4", [0, 3])
def test_sddmm_strip_sum_paths(usm, dtype, scale, nnz_mod4):
    """D = 300 spans several column strips, whose partials a second kernel
    adds: four nonzeros at a time when every array is aligned (strips of
    partials are padded to a multiple of 32; with nnz % 4 = 3 the last group
    is ragged), else one at a time (an output starting one element into its
    buffer forces that).  Both add the same terms in the same order."""
    import torch
    M, K, D = 257, 333, 300
    rng = np.random.default_rng([nnz_mod4, 16])
    lengths = rng.integers(0, 40, M)
    lengths[-1] += (nnz_mod4 - int(lengths.sum())) % 4
    csr = W.random_csr(17, M, K, 0.0, dtype=dtype, lengths=lengths)
    assert csr.nnz % 4 == nnz_mod4
    X, Y = W.dense(rng, M, D, 1.0, dtype), W.dense(rng, K, D, 1.0, dtype)
    ro, ci, vals = csr_dev(csr)
    nnz = csr.nnz
    outs = {}
    for odt in (torch.float32, torch.bfloat16):
        for offset in (0, 1):
            buf = torch.full((nnz + 8,), 7.0, dtype=odt, device="cuda")
            usm.sddmm_general(ro, ci, dev(X, dtype), dev(Y, dtype), values=vals if scale else None,
                              out=buf[offset:offset + nnz])
            assert (buf[:offset] == 7).all() and (buf[offset + nnz:] == 7).all()
            outs[odt, offset] = buf[offset:offset + nnz]
    f32 = outs[torch.float32, 0]
    assert torch.equal(f32, outs[torch.float32, 1])
    for offset in (0, 1):  # bf16 output: the fp32 result rounded to nearest even
        assert torch.equal(outs[torch.bfloat16, offset], f32.to(torch.bfloat16))
    a = oracle.widen(csr.values, dtype)
    ref = oracle.sddmm_general(M, K, csr.row_offsets, csr.col_indices, a, scale, oracle.widen(X, dtype),
                               oracle.widen(Y, dtype), True)
    S = oracle.sddmm_error_scale(M, K, csr.row_offsets, csr.col_indices, oracle.widen(X, dtype),
                                 oracle.widen(Y, dtype)) * (np.abs(a) if scale else 1.0)
    assert_within(host(f32), ref, S, TOL[dtype], f"strip sum scale={scale} nnz%4={nnz_mod4}")


# ---------------------------------------------------------------------------
# f4: row softmax and the attention chain with it
# ---------------------------------------------------------------------------
def test_row_softmax(usm):
    import torch
    # empty, single-entry, short and long rows (up to more than 4096 entries)
    lengths = np.r_[np.zeros(20, int), np.ones(20, int), np.arange(2, 300),
                    [1024, 1025, 2048, 2049, 4096, 4097, 5000, 700]]
    csr = W.random_csr(16, lengths.size, 5000, 0.0, lengths=lengths)
    s = (np.random.default_rng(17).standard_normal(csr.nnz) * 3).astype(np.float32)
    ro = dev(csr.row_offsets)
    p32 = host(usm.row_softmax(ro, dev(s)))
    ref = oracle.csr_softmax(csr.row_offsets, s.astype(np.float64))
    # ≤ n/128 + 9 roundings per output with n ≤ 5000 (≤ 49 u) plus the fast
    # exponential's ≤ 2 + 1.17·|s - m| ulp (|s - m| < 25 here: ≤ 32 u):
    # under 100 u = 6e-6 relative, checked against 2e-5
    assert np.all(np.abs(p32 - ref) <= 2e-5 * ref)
    p16 = host(usm.row_softmax(ro, dev(s), out_dtype=torch.bfloat16))
    want = oracle.round_to_bf16(ref)
    assert np.all(np.abs(p16.astype(np.int64) - want.astype(np.int64)) <= 1)
    assert np.mean(p16 == want) > 0.99


# (N, density, seg_rows); 1% of 1500 columns with N = 64 takes the fp32 gather kernel
FUSED_CASES = [(64, 0.05, 0), (128, 0.1, 0), (300, 0.2, 0), (64, 0.3, 250), (64, 0.01, 0), (1300, 0.6, 0)]


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("N,density,seg", FUSED_CASES)
@pytest.mark.parametrize("swz", [False, True])
def test_spmm_row_softmax_matches_unfused_chain(usm, dtype, N, density, seg, swz):
    """The fused softmax-SpMM gives the bits of csr_row_softmax into a
    buffer of B's type followed by csr_spmm, and the oracle chain's result
    within tolerance (empty, single-entry and long rows included)."""
    import torch
    M, K = 1000, 1500
    rng = np.random.default_rng([N, seg, 21])
    lengths = rng.binomial(K, density, M)
    lengths[:10] = 0
    lengths[10:20] = 1
    lengths[20] = K
    if seg:  # block-diagonal rows: each block of seg rows only touches its own columns
        K = M
        lengths = np.minimum(lengths, seg)
        base = (np.arange(M) // seg) * seg
        ro, ci = W.csr_from_lengths(rng, lengths, seg, col_base=base)
        csr = W.CSR(M, K, ro, ci, W.values_for(rng, int(ro[-1]), 1.0, dtype), dtype, seg_rows=seg)
    else:
        csr = W.random_csr([N, 22], M, K, 0.0, dtype=dtype, lengths=lengths)
    s = (rng.standard_normal(csr.nnz) * 3).astype(np.float32)
    B = W.dense(rng, K, N, 1.0, dtype)
    ro, ci = dev(csr.row_offsets), dev(csr.col_indices)
    perm = usm.row_swizzle(ro, K, seg) if swz else None
    Bd, sd = dev(B, dtype), dev(s)
    fused = host(usm.spmm_row_softmax(ro, ci, sd, Bd, K=K, row_swizzle=perm, seg_rows=seg))
    P = usm.row_softmax(ro, sd, out_dtype=torch.bfloat16 if dtype == "bf16" else torch.float32)
    unfused = host(usm.spmm(ro, ci, P, Bd, K=K, row_swizzle=perm, seg_rows=seg))
    assert np.array_equal(fused, unfused)
    assert usm.poll_status() == 0
    # the oracle chain: fp64 softmax (rounded to bf16 for bf16), fp64 SpMM
    p64 = oracle.csr_softmax(csr.row_offsets, s.astype(np.float64))
    if dtype == "bf16":
        p64 = oracle.widen(oracle.round_to_bf16(p64), "bf16")
    Bw = oracle.widen(B, dtype)
    ref = oracle.spmm(M, K, csr.row_offsets, csr.col_indices, p64, Bw)
    S = oracle.spmm_error_scale(M, K, csr.row_offsets, csr.col_indices, p64, Bw)
    # fp32: the probabilities carry <= n/128 + 9 roundings and the fast
    # exponential's <= 2 + 1.17·|s - m| ulp (under 100 u = 6e-6 relative for
    # n <= 1500, |s - m| < 25) on top of the SpMM's 1e-5; bf16: one bf16 ulp
    # (2^-7 relative) between the GPU's rounding of its fp32 probability and
    # the oracle's rounding of the exact one
    tol = 2e-5 if dtype == "f32" else TOL["bf16"] + 2.0 ** -7
    assert_within(fused, ref, S, tol, f"fused softmax spmm {dtype} N={N}")


@pytest.mark.parametrize("N", [100, 600])
def test_spmm_row_softmax_row_groups(usm, N):
    """fp32 scores on masks 60% set with enough rows for the row-group kernel
    (128-wide strips for N = 100, 256-wide for N = 600): the fused call gives
    the unfused chain's bits and the oracle chain's result."""
    import torch
    M, K = 5000, 700
    csr = W.random_csr([N, 23], M, K, 0.6)
    rng = np.random.default_rng([N, 24])
    s = (rng.standard_normal(csr.nnz) * 3).astype(np.float32)
    B = W.dense(rng, K, N)
    ro, ci = dev(csr.row_offsets), dev(csr.col_indices)
    perm = usm.row_swizzle(ro, K)
    Bd, sd = dev(B), dev(s)
    fused = host(usm.spmm_row_softmax(ro, ci, sd, Bd, K=K, row_swizzle=perm))
    P = usm.row_softmax(ro, sd, out_dtype=torch.float32)
    unfused = host(usm.spmm(ro, ci, P, Bd, K=K, row_swizzle=perm))
    assert np.array_equal(fused, unfused)
    assert usm.poll_status() == 0
    p64 = oracle.csr_softmax(csr.row_offsets, s.astype(np.float64))
    Bw = oracle.widen(B, "f32")
    ref = oracle.spmm(M, K, csr.row_offsets, csr.col_indices, p64, Bw)
    S = oracle.spmm_error_scale(M, K, csr.row_offsets, csr.col_indices, p64, Bw)
    assert_within(fused, ref, S, 2e-5, f"row-group fused softmax spmm N={N}")


@pytest.mark.slow
def test_attention_chain_with_softmax(usm):
    import torch
    p = W.attention()
    csr = p.csr
    ro, ci = dev(csr.row_offsets), dev(csr.col_indices)
    perm = usm.row_swizzle(ro, csr.K, seg_rows=p.meta["seq"])
    seg = p.meta["seq"]
    scores = usm.sddmm(ro, ci, dev(p.X, "bf16"), dev(p.Y, "bf16"), row_swizzle=perm, seg_rows=seg)
    probs = usm.row_softmax(ro, scores, out_dtype=torch.bfloat16)
    O = host(usm.spmm(ro, ci, probs, dev(p.V, "bf16"), K=csr.K, row_swizzle=perm, seg_rows=seg))
    # every nonzero and every output element of the 32768-row stack
    ro_h, ci_h = csr.row_offsets, csr.col_indices
    s64 = oracle.sddmm(csr.M, csr.K, ro_h, ci_h, oracle.widen(p.X, "bf16"), oracle.widen(p.Y, "bf16"))
    p16 = oracle.round_to_bf16(oracle.csr_softmax(ro_h, s64))
    got16 = host(probs)
    # one bf16 ulp at most (the GPU's fp32 scores and softmax against the
    # oracle's fp64 ones, each rounded once to bf16)
    assert np.all(np.abs(got16.astype(np.int64) - p16.astype(np.int64)) <= 1)
    Vw = oracle.widen(p.V, "bf16")
    g64 = oracle.widen(got16, "bf16")
    ref = oracle.spmm(csr.M, csr.K, ro_h, ci_h, g64, Vw)
    S = oracle.spmm_error_scale(csr.M, csr.K, ro_h, ci_h, g64, Vw)
    assert_within(O, ref, S, TOL["bf16"], "attention with softmax")
    # against the oracle's whole chain: probabilities one ulp (2^-7 relative)
    # apart move an output by at most 2^-7 of its error scale
    w64 = oracle.widen(p16, "bf16")
    ref = oracle.spmm(csr.M, csr.K, ro_h, ci_h, w64, Vw)
    S = oracle.spmm_error_scale(csr.M, csr.K, ro_h, ci_h, w64, Vw)
    assert_within(O, ref, S, TOL["bf16"] + 2.0 ** -7, "attention with softmax vs the oracle chain")


@pytest.mark.slow
def test_attention_chain_fused_softmax(usm):
    """The attention chain with the softmax inside the SpMM: SDDMM scores
    (fp32), then csr_spmm_row_softmax with V.  Every output element equals
    the unfused chain's (csr_row_softmax to bf16, then csr_spmm) bit for bit
    and the oracle chain's within tolerance."""
    import torch
    p = W.attention()
    csr = p.csr
    ro, ci = dev(csr.row_offsets), dev(csr.col_indices)
    seg = p.meta["seq"]
    perm = usm.row_swizzle(ro, csr.K, seg_rows=seg)
    V = dev(p.V, "bf16")
    scores = usm.sddmm(ro, ci, dev(p.X, "bf16"), dev(p.Y, "bf16"), row_swizzle=perm, seg_rows=seg)
    O = host(usm.spmm_row_softmax(ro, ci, scores, V, K=csr.K, row_swizzle=perm, seg_rows=seg))
    probs = usm.row_softmax(ro, scores, out_dtype=torch.bfloat16)
    O_unfused = host(usm.spmm(ro, ci, probs, V, K=csr.K, row_swizzle=perm, seg_rows=seg))
    assert np.array_equal(O, O_unfused)
    ro_h, ci_h = csr.row_offsets, csr.col_indices
    s64 = oracle.sddmm(csr.M, csr.K, ro_h, ci_h, oracle.widen(p.X, "bf16"), oracle.widen(p.Y, "bf16"))
    w64 = oracle.widen(oracle.round_to_bf16(oracle.csr_softmax(ro_h, s64)), "bf16")
    Vw = oracle.widen(p.V, "bf16")
    ref = oracle.spmm(csr.M, csr.K, ro_h, ci_h, w64, Vw)
    S = oracle.spmm_error_scale(csr.M, csr.K, ro_h, ci_h, w64, Vw)
    assert_within(O, ref, S, TOL["bf16"] + 2.0 ** -7, "fused attention vs the oracle chain")


# ---------------------------------------------------------------------------
# f3: the sparse layer's training step (forward, weight and input gradients)
# ---------------------------------------------------------------------------
@pytest.mark.slow
@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_training_step_chain(usm, dtype):
    p = W.ffn(4096, 1024, 90, dtype)
    csr = p.csr
    M, K, N = csr.M, csr.K, p.meta["N"]
    dC = W.dense(np.random.default_rng(18), M, N, 1.0, dtype)
    ro, ci, vals = csr_dev(csr)
    perm = usm.row_swizzle(ro, K)
    ro_t, ci_t, v_t, tperm = usm.csr_transpose(ro, ci, vals, K, with_perm=True)
    perm_t = usm.row_swizzle(ro_t, M)
    B, dCd = dev(p.B, dtype), dev(dC, dtype)
    C = usm.spmm(ro, ci, vals, B, K=K, row_swizzle=perm)                  # forward
    dA = usm.sddmm(ro, ci, dCd, B, row_swizzle=perm)                        # weight gradient
    v_t = usm.csr_permute_values(tperm, vals, out=v_t)                      # weights in Aᵀ order
    dB = usm.spmm(ro_t, ci_t, v_t, dCd, K=M, row_swizzle=perm_t)           # input gradient
    # every element of the three products
    ref, S = oracle_spmm(csr, p.B, dtype)
    assert_within(host(C), ref, S, TOL[dtype], "forward")
    ref, S, _ = oracle_sddmm(csr, dC, p.B, dtype)
    assert_within(host(dA), ref, S, TOL[dtype], "weight gradient")
    t_ro, t_ci, t_v = oracle.csr_transpose(M, K, csr.row_offsets, csr.col_indices, oracle.widen(csr.values, dtype))
    dCw = oracle.widen(dC, dtype)
    ref = oracle.spmm(K, M, t_ro, t_ci, t_v, dCw)
    S = oracle.spmm_error_scale(K, M, t_ro, t_ci, t_v, dCw)
    assert_within(host(dB), ref, S, TOL[dtype], "input gradient")
