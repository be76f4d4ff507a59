"""Seeded synthetic inputs shaped like the sparse deep-learning workloads of
"Sparse GPU Kernels for Deep Learning" (Gale, Zaharia, Young, Elsen, SC 2020).

This module only draws inputs: CSR structure, values and dense operands. It
holds none of the SpMM/SDDMM arithmetic, so both the CPU oracle (through the
tests) and the CUDA path consume exactly the same arrays.

The pages characterise deep-learning weight matrices as moderately sparse,
with long rows and low row-length coefficient of variation (CoV), next to the
scientific SuiteSparse collection (summary card, "Key points", matrix
properties bullet). Their 3,012-matrix collection is not available, so the
configurations below stand in for it with seeded synthetic matrices of that
character:

* ``tiny``      256x256 at 90%, Binomial row lengths, N(0,1) values, N=D=64.
* ``resnet``    512x2048 at 80%, Binomial rows (CoV ~0.044), N(0,0.02) values,
                B 2048x3136; SDDMM with X 512x3136, Y 2048x3136.
* ``ffn``       4096x1024 and 1024x4096 at {70,80,90,95}%, row lengths
                round(N(mu, (0.1 mu)^2)) clipped to [1,K], mu = K(1-s),
                N(0,0.02) values, B/X/Y 2048 wide, fp32 or bf16.
* ``lstm``      8192x4096 at {50,...,98}%, Binomial rows, B 4096x128.
* ``attention`` 8 heads x 4096 rows, lognormal row lengths (mean 410, CoV 0.5,
                clipped to [1,4096]), stacked as one block-diagonal
                32768x32768 CSR; Q, K, V 32768x64 N(0,1) in bf16.

Columns are drawn uniformly without replacement per row and sorted, so every
row's column indices are strictly increasing.

Seeds: ``numpy.random.default_rng([config_id, sparsity_pct, operand_id])``
with operand_id 0 = structure, 1 = values, 2 = B / Q, 3 = Y / K, 4 = V,
5 = X (SDDMM left operand, drawn apart from B so the two never coincide).
"""
from __future__ import annotations

from dataclasses import dataclass, field
import math

import numpy as np

CONFIG_IDS = {"tiny": 1, "resnet": 2, "ffn": 3, "lstm": 4, "attention": 5}

FFN_SPARSITIES = (70, 80, 90, 95)
FFN_SHAPES = ((4096, 1024), (1024, 4096))
LSTM_SPARSITIES = (50, 60, 70, 80, 90, 95, 98)


def rng_for(config_id: int, sparsity_pct: int, operand_id: int) -> np.random.Generator:
    return np.random.default_rng([int(config_id), int(sparsity_pct), int(operand_id)])


# ----------------------------------------------------------------------------
# bf16 storage.  Inputs are drawn in fp32 and rounded to bf16 with
# round-to-nearest-even on the bit pattern; the rounded bits are what every
# consumer receives.  No NaN/Inf is ever produced by the draws below.
# ----------------------------------------------------------------------------
def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32).astype(np.uint64)
    rounded = (u + 0x7FFF + ((u >> 16) & 1)) >> 16
    return rounded.astype(np.uint16)


def bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    return (np.ascontiguousarray(b, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)


# ----------------------------------------------------------------------------
# CSR container
# ----------------------------------------------------------------------------
@dataclass
class CSR:
    M: int
    K: int
    row_offsets: np.ndarray          # int32 [M+1]
    col_indices: np.ndarray          # int32 [nnz]
    values: np.ndarray               # float32 [nnz] or uint16 bf16 bits [nnz]
    dtype: str = "f32"               # "f32" or "bf16"
    seg_rows: int = 0                # rows per diagonal block (0 = one block)

    @property
    def nnz(self) -> int:
        return int(self.row_offsets[-1])

    def values_f32(self) -> np.ndarray:
        if self.dtype == "bf16":
            return bf16_bits_to_f32(self.values)
        return self.values

    def row_lengths(self) -> np.ndarray:
        return np.diff(self.row_offsets.astype(np.int64))


def stats(csr: CSR) -> dict:
    """Sparsity, mean row length and row-length CoV (the characterisation
    the pages use to contrast DL matrices with SuiteSparse)."""
    lens = csr.row_lengths().astype(np.float64)
    block_cols = csr.K if not csr.seg_rows else csr.seg_rows
    mean = float(lens.mean()) if lens.size else 0.0
    std = float(lens.std()) if lens.size else 0.0
    return {
        "sparsity": 1.0 - mean / block_cols if block_cols else 1.0,
        "mean_row_length": mean,
        "row_length_cov": std / mean if mean > 0 else 0.0,
        "nnz": csr.nnz,
    }


# ----------------------------------------------------------------------------
# Row-length distributions
# ----------------------------------------------------------------------------
def lengths_binomial(rng, M: int, K: int, density: float) -> np.ndarray:
    return rng.binomial(K, density, size=M).astype(np.int64)


def lengths_normal(rng, M: int, K: int, mean: float, cov: float) -> np.ndarray:
    raw = rng.normal(mean, cov * mean, size=M)
    return np.clip(np.rint(raw), 1, K).astype(np.int64)


def lengths_lognormal(rng, M: int, K: int, mean: float, cov: float) -> np.ndarray:
    sigma = math.sqrt(math.log(1.0 + cov * cov))
    mu = math.log(mean) - 0.5 * sigma * sigma
    raw = rng.lognormal(mu, sigma, size=M)
    return np.clip(np.rint(raw), 1, K).astype(np.int64)


def csr_from_lengths(rng, lengths: np.ndarray, K: int, col_base: np.ndarray | None = None):
    """Sorted, unique, uniformly drawn column indices for each row."""
    M = lengths.size
    row_offsets = np.zeros(M + 1, dtype=np.int64)
    np.cumsum(lengths, out=row_offsets[1:])
    nnz = int(row_offsets[-1])
    if nnz >= 2**31:
        raise ValueError("nnz does not fit int32")
    cols = np.empty(nnz, dtype=np.int32)
    for r in range(M):
        n = int(lengths[r])
        if n == 0:
            continue
        pick = rng.choice(K, size=n, replace=False)
        pick.sort()
        if col_base is not None:
            pick = pick + col_base[r]
        cols[row_offsets[r]:row_offsets[r + 1]] = pick
    return row_offsets.astype(np.int32), cols


def dense(rng, rows: int, cols: int, std: float = 1.0, dtype: str = "f32", int_valued: bool = False):
    if int_valued:
        x = rng.integers(-4, 5, size=(rows, cols)).astype(np.float32)
    else:
        x = (rng.standard_normal(size=(rows, cols)) * std).astype(np.float32)
    return f32_to_bf16_bits(x) if dtype == "bf16" else x


def values_for(rng, nnz: int, std: float, dtype: str, int_valued: bool = False):
    if int_valued:
        v = rng.integers(-4, 5, size=nnz).astype(np.float32)
    else:
        v = (rng.standard_normal(size=nnz) * std).astype(np.float32)
    return f32_to_bf16_bits(v) if dtype == "bf16" else v


# ----------------------------------------------------------------------------
# Generic random CSR (tests: ragged shapes, edge cases)
# ----------------------------------------------------------------------------
def random_csr(seed, M: int, K: int, density: float, dtype: str = "f32", std: float = 1.0,
               int_valued: bool = False, lengths: np.ndarray | None = None) -> CSR:
    rng = np.random.default_rng(seed)
    if lengths is None:
        lengths = lengths_binomial(rng, M, K, density) if K > 0 else np.zeros(M, dtype=np.int64)
    lengths = np.asarray(lengths, dtype=np.int64)
    ro, ci = csr_from_lengths(rng, lengths, K)
    vals = values_for(rng, int(ro[-1]), std, dtype, int_valued)
    return CSR(M, K, ro, ci, vals, dtype)


# ----------------------------------------------------------------------------
# The five workload configurations
# ----------------------------------------------------------------------------
@dataclass
class Problem:
    name: str
    csr: CSR
    B: np.ndarray | None = None       # K x N (SpMM dense operand)
    X: np.ndarray | None = None       # M x D (SDDMM left operand)
    Y: np.ndarray | None = None       # K x D (SDDMM right operand, used transposed)
    V: np.ndarray | None = None       # K x N (attention values)
    dtype: str = "f32"
    meta: dict = field(default_factory=dict)


def tiny(dtype: str = "f32", int_valued: bool = False) -> Problem:
    cid = CONFIG_IDS["tiny"]
    M = K = 256
    rng = rng_for(cid, 90, 0)
    lens = lengths_binomial(rng, M, K, 0.1)
    ro, ci = csr_from_lengths(rng, lens, K)
    vals = values_for(rng_for(cid, 90, 1), int(ro[-1]), 1.0, dtype, int_valued)
    csr = CSR(M, K, ro, ci, vals, dtype)
    return Problem("tiny", csr,
                   B=dense(rng_for(cid, 90, 2), K, 64, 1.0, dtype, int_valued),
                   X=dense(rng_for(cid, 90, 5), M, 64, 1.0, dtype, int_valued),
                   Y=dense(rng_for(cid, 90, 3), K, 64, 1.0, dtype, int_valued),
                   dtype=dtype, meta={"N": 64, "D": 64, "sparsity": 90})


def resnet(dtype: str = "f32", with_sddmm: bool = True) -> Problem:
    cid = CONFIG_IDS["resnet"]
    M, K, N = 512, 2048, 3136
    rng = rng_for(cid, 80, 0)
    lens = lengths_binomial(rng, M, K, 0.2)
    ro, ci = csr_from_lengths(rng, lens, K)
    vals = values_for(rng_for(cid, 80, 1), int(ro[-1]), 0.02, dtype)
    csr = CSR(M, K, ro, ci, vals, dtype)
    p = Problem("resnet", csr, B=dense(rng_for(cid, 80, 2), K, N, 1.0, dtype), dtype=dtype,
                meta={"N": N, "D": N, "sparsity": 80})
    if with_sddmm:
        p.X = dense(rng_for(cid, 80, 5), M, N, 1.0, dtype)
        p.Y = dense(rng_for(cid, 80, 3), K, N, 1.0, dtype)
    return p


def ffn(M: int, K: int, sparsity: int, dtype: str = "f32", N: int = 2048,
        with_spmm: bool = True, with_sddmm: bool = True) -> Problem:
    """Transformer FFN weight at the given sparsity; both shapes share the
    seeds except for the shape tag folded into the config id."""
    cid = CONFIG_IDS["ffn"] * 10 + (0 if M >= K else 1)
    rng = rng_for(cid, sparsity, 0)
    mu = K * (1.0 - sparsity / 100.0)
    lens = lengths_normal(rng, M, K, mu, 0.1)
    ro, ci = csr_from_lengths(rng, lens, K)
    vals = values_for(rng_for(cid, sparsity, 1), int(ro[-1]), 0.02, dtype)
    csr = CSR(M, K, ro, ci, vals, dtype)
    p = Problem(f"ffn_{M}x{K}_s{sparsity}", csr, dtype=dtype,
                meta={"N": N, "D": N, "sparsity": sparsity})
    if with_spmm:
        p.B = dense(rng_for(cid, sparsity, 2), K, N, 1.0, dtype)
    if with_sddmm:
        p.X = dense(rng_for(cid, sparsity, 5), M, N, 1.0, dtype)
        p.Y = dense(rng_for(cid, sparsity, 3), K, N, 1.0, dtype)
    return p


def lstm(sparsity: int, dtype: str = "f32") -> Problem:
    cid = CONFIG_IDS["lstm"]
    M, K, N = 8192, 4096, 128
    rng = rng_for(cid, sparsity, 0)
    lens = lengths_binomial(rng, M, K, 1.0 - sparsity / 100.0)
    ro, ci = csr_from_lengths(rng, lens, K)
    vals = values_for(rng_for(cid, sparsity, 1), int(ro[-1]), 0.02, dtype)
    csr = CSR(M, K, ro, ci, vals, dtype)
    return Problem(f"lstm_s{sparsity}", csr, B=dense(rng_for(cid, sparsity, 2), K, N, 1.0, dtype),
                   dtype=dtype, meta={"N": N, "sparsity": sparsity})


def attention(heads: int = 8, seq: int = 4096, head_dim: int = 64, mean_len: float = 410.0,
              cov: float = 0.5) -> Problem:
    """Block-diagonal stack of per-head masks: row h*seq+i keeps columns in
    [h*seq, (h+1)*seq).  The mask carries no values of its own (the SDDMM
    scores become the SpMM values), so csr.values holds ones."""
    cid = CONFIG_IDS["attention"]
    M = heads * seq
    rng = rng_for(cid, 90, 0)
    lens = lengths_lognormal(rng, M, seq, mean_len, cov)
    col_base = (np.arange(M, dtype=np.int64) // seq) * seq
    ro, ci = csr_from_lengths(rng, lens, seq, col_base=col_base)
    ones = f32_to_bf16_bits(np.ones(int(ro[-1]), dtype=np.float32))
    csr = CSR(M, M, ro, ci, ones, "bf16", seg_rows=seq)
    return Problem("attention", csr,
                   X=dense(rng_for(cid, 90, 2), M, head_dim, 1.0, "bf16"),
                   Y=dense(rng_for(cid, 90, 3), M, head_dim, 1.0, "bf16"),
                   V=dense(rng_for(cid, 90, 4), M, head_dim, 1.0, "bf16"),
                   dtype="bf16", meta={"heads": heads, "seq": seq, "D": head_dim, "N": head_dim})


def ffn_suite(dtype: str, with_spmm: bool = True, with_sddmm: bool = True):
    for (M, K) in FFN_SHAPES:
        for s in FFN_SPARSITIES:
            yield ffn(M, K, s, dtype, with_spmm=with_spmm, with_sddmm=with_sddmm)
