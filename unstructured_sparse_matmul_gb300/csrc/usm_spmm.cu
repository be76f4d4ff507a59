// CSR SpMM: host launch code (tile choice, launch model, kernel launch).
// The kernel and its design are in usm_spmm_kernel.cuh.
#include <cmath>

#include "usm_internal.h"
#include "usm_spmm_kernel.cuh"
#include "usm_spmm_group.cuh"

namespace usm {
namespace {

// 128-entry windows read with 16-byte loads (VL) against 32-entry windows
// read one element a lane: USM_SPMM_VL=1 takes VL wherever the kernel
// allows it (one lane group, no tensor-memory rows, aligned CSR arrays).
#ifndef USM_SPMM_VL
#define USM_SPMM_VL 0
#endif

// UG: the row-group kernel (usm_spmm_group.cuh; fp32 128- or 256-column
// strips, one stage, G = R row slots a warp) instead of the row kernel.
template <bool BF, int L, int VEC, int R, int W, int KC, int NS, int MB, bool LONGK, bool TM, bool SMX, bool VL,
          bool UG = false>
int launch_kernel(SpmmArgs a, int tiles_per_block, const void* B, int ldb, cudaStream_t stream) {
    using C_ = SpmmCfg<BF, L, VEC, R, W, KC, NS, TM, VL>;
    CUtensorMap map;
    if (!encode_tensor_map_2d(&map, B, BF, a.K, a.N, ldb, C_::BOX_COLS, C_::BOX_ROWS)) return USM_ERR_CUDA;
    auto pick = [] {
        if constexpr (UG) {
            static_assert(!BF && L == 32 && (VEC == 4 || VEC == 8) && NS == 1 && MB == 1 && !LONGK && !TM && !VL,
                          "row groups");
            return spmm_group_kernel<KC, W, R, VEC, SMX>;
        } else {
            return spmm_kernel<BF, L, VEC, R, W, KC, NS, MB, LONGK, TM, SMX, VL>;
        }
    };
    auto kern = pick();
    constexpr int SMEM = UG ? GroupCfg<KC, W, R, VEC>::SMEM : C_::SMEM;
    static int configured_mask = 0;  // one bit per device
    int dev = 0;
    cudaGetDevice(&dev);
    if (dev < 31 && !(__atomic_load_n(&configured_mask, __ATOMIC_ACQUIRE) & (1 << dev))) {
        if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM) !=
            cudaSuccess)
            return USM_ERR_CUDA;
        __atomic_fetch_or(&configured_mask, 1 << dev, __ATOMIC_ACQ_REL);
    }
    // Row tiles on x (dispatched first, longest rows first under a swizzle),
    // column strips on y.
    // Every row of a block must have a slot: tiles × R·W ≥ rows per block.
    if (tiles_per_block < 1 || (long long)tiles_per_block * R * W < a.seg_rows) return USM_ERR_INVALID_ARG;
    a.tiles_per_block = tiles_per_block;
    const long long tiles = block_count(a.M, a.seg_rows) * tiles_per_block;
    if (tiles > 0x7fffffffLL) return USM_ERR_UNSUPPORTED;
    const dim3 grid((unsigned)tiles, (a.N + C_::NT - 1) / C_::NT);
    if (grid.y > 65535u) return USM_ERR_UNSUPPORTED;
    kern<<<grid, C_::THREADS, SMEM, stream>>>(map, a);
    return cudaGetLastError() == cudaSuccess ? USM_OK : USM_ERR_CUDA;
}

template <bool BF, int L, int VEC, int R, int W, int KC, int NS, int MB, bool LONGK = false, bool TM = false,
          bool SMX = false, bool UG = false>
int launch_cfg(SpmmArgs a, int tiles_per_block, const void* B, int ldb, cudaStream_t stream) {
    if constexpr (UG) {
        return launch_kernel<BF, L, VEC, R, W, KC, NS, MB, false, false, SMX, false, true>(a, tiles_per_block, B, ldb,
                                                                                         stream);
    } else if constexpr (USM_SPMM_VL && L == 32 && !TM) {
        const bool aligned = (reinterpret_cast<uintptr_t>(a.col_indices) & 15u) == 0 &&
                             (reinterpret_cast<uintptr_t>(a.values) & (BF ? 7u : 15u)) == 0;
        if (aligned) return launch_kernel<BF, L, VEC, R, W, KC, NS, MB, LONGK, TM, SMX, true>(a, tiles_per_block, B, ldb, stream);
    }
    return launch_kernel<BF, L, VEC, R, W, KC, NS, MB, LONGK, TM, SMX, false>(a, tiles_per_block, B, ldb, stream);
}

}  // namespace

int launch_fill_f32(float* C, int M, int N, long long ldc, cudaStream_t stream) {
    if ((long long)M * N == 0) return USM_OK;
    const long long total = (long long)M * N;
    int blocks = (int)((total + 255) / 256);
    if (blocks > 4096) blocks = 4096;
    fill_f32_kernel<<<blocks, 256, 0, stream>>>(C, M, N, ldc);
    return cudaGetLastError() == cudaSuccess ? USM_OK : USM_ERR_CUDA;
}

// Tile choice.  Lanes own 8 elements of a 256-column strip when N > 128
// (fp32: two 16-byte loads per step; bf16: one); 4 elements of a 128- or
// 64-column strip for narrower N.  16 warps per CTA (20 for fp32 128-wide
// strips with 2-4 rows a warp, below).  bf16 steps are
// latency-bound and run two CTAs per SM (≤ 64 registers, 96 KB of stage
// each); fp32 steps are bound by shared-memory bandwidth and run one CTA per
// SM with up to 128 registers and one stage of 192 KB or more (N > 128: KC =
// 192 or 208 rows of 1 KB; N ≤ 128: 384 or 416 rows of 512 B; N ≤ 64: 768 of
// 256 B; the taller where it saves a chunk): taller chunks
// halve the per-(row, chunk) work and more rows per CTA share each staged
// row, and row slots keep their CSR windows across chunks.  Measured against
// two CTAs per SM: FFN fp32 SpMM 3-12% faster, LSTM (N = 128) 5% faster at
// 50% sparsity up to 39% at 98%.  One tall stage (the default) against two
// stages of half the height: the FFN step took 7.69 against 8.90 ms.
#ifndef USM_SPMM_STAGES
#define USM_SPMM_STAGES 1
#endif
// Rows per warp R (RA or RB) and row tiles per diagonal block from a launch
// time model.  For each R two tile counts are tried: the fewest tiles that
// hold the block (R·W rows each), and more tiles of fewer rows that fill the
// last wave of MB·SMs CTA slots (1024x4096 fp32: 19 tiles of ~54 rows x 8
// strips = 152 CTAs instead of 16 x 8 = 128 on 152 SMs).  Time, in units of
// one consumed row, is the larger of
//  * the SMs: whole waves × MB resident CTAs × per-CTA work, where a CTA
//    stages every row of its K span (2 units: a staged row costs about two
//    consumed ones) and consumes its rows' mean-length share of nonzeros;
//  * L2: every CTA's staged rows over the SMs, 5 units a row (aggregate
//    shared-memory bandwidth is about five times what L2 delivers to TMA).
// Measured against the fewest tiles: FFN SpMM 7-14% faster, LSTM 5-13%,
// ResNet 31%, attention 6%.
template <bool BF, int L, int VEC, int W, int KC, int NS, int MB, int RA = 2, int RB = 4, bool TM = false,
          bool SMX = false, bool UG = false>
int launch_pick(const SpmmArgs& a, const void* B, int ldb, cudaStream_t stream) {
    const int sms = sm_count_current_device();
    const long long slots = (long long)sms * MB;
    const int nt = L * VEC;
    const long long strips = (a.N + nt - 1) / nt, blocks = block_count(a.M, a.seg_rows);
    // A block-diagonal schedule (seg_rows < M) is taken to have square blocks.
    const double kspan = (a.seg_rows > 0 && a.seg_rows < a.M) ? (double)min(a.K, a.seg_rows) : (double)a.K;
    const double mean_len = (double)a.nnz / (a.M > 0 ? a.M : 1);
    auto fill = [&](int mt) {  // tiles per block that fill the last wave
        const long long tmin = (a.seg_rows + mt - 1) / mt;
        const long long tmax = max(tmin, (long long)(a.seg_rows + W - 1) / W);  // >= W rows a tile
        const long long per = blocks * strips;
        const long long waves = (per * tmin + slots - 1) / slots;
        return (int)min(tmax, max(tmin, waves * slots / per));
    };
    auto cost = [&](int t) {
        const double n = (double)(blocks * t * strips);
        const double sm = std::ceil(n / slots) * MB * (2.0 * kspan + (double)a.seg_rows / t * mean_len);
        return fmax(sm, n * kspan * 5.0 / sms);
    };
    const ScheduleOverride ov = schedule_override();
    if (ov.k_splits > 1) return USM_ERR_UNSUPPORTED;
    auto tiles = [&](int r) {  // the model's tile count for R = r, or the forced one
        const int t0 = (a.seg_rows + r * W - 1) / (r * W), t1 = fill(r * W);
        if (ov.tiles_per_block > 0) return max(t0, ov.tiles_per_block);
        return cost(t1) < cost(t0) ? t1 : t0;
    };
    const int ta = tiles(RA), tb = tiles(RB);
    // The cheaper tiling; RB's tile count runs on RA's kernel wherever its
    // tiles hold no more rows than RA's slots (measured 3-14% faster than
    // RB at equal tile counts, never slower).
    int R = cost(ta) < cost(tb) ? RA : RB, T = R == RA ? ta : tb;
    if (R == RB && (long long)tb * RA * W >= a.seg_rows) R = RA;
    // Row groups: RB slots a warp share each staged row among more rows.
    if (UG) R = RB, T = tb;
    if (ov.rows_per_warp == RA) R = RA, T = ta;
    else if (ov.rows_per_warp == RB) R = RB, T = tb;
    else if (ov.rows_per_warp != 0) return USM_ERR_UNSUPPORTED;
    // fp32 with more than 128 chunks of K: the kernel with a second-level
    // accumulator keeps the worst-case rounding bound (RA rows a warp only,
    // for the registers it takes).
    if (!UG && !BF && (a.K + KC - 1) / KC > 128) {
        if (ov.rows_per_warp == RB) return USM_ERR_UNSUPPORTED;
        return launch_cfg<BF, L, VEC, RA, W, KC, NS, MB, true, TM, SMX>(a, ta, B, ldb, stream);
    }
    if (R == RA) return launch_cfg<BF, L, VEC, RA, W, KC, NS, MB, false, TM, SMX, UG>(a, T, B, ldb, stream);
    return launch_cfg<BF, L, VEC, RB, W, KC, NS, MB, false, TM, SMX, UG>(a, T, B, ldb, stream);
}

// The six tile shapes by element type and N.  SMX: the values are the rows'
// softmax probabilities of fp32 scores (csr_spmm_row_softmax).
// Direct gather (no staging) for very sparse fp32 masks with narrow rows of
// B: a mask under USM_SPMM_GATHER_PERMILLE per mille set and N <=
// USM_SPMM_GATHER_N, unless a launch shape is forced (the staged kernels'
// schedules are what usm_set_schedule_override controls); with or without
// the fused softmax, so csr_spmm_row_softmax keeps csr_spmm's bits.  Measured on the
// LSTM sweep (8192x4096, N = 128): 98% sparsity 25% faster than staging all
// of K per CTA, 95% 14% slower; FFN 95% (N = 2048) 1.6-4.6x slower.
#ifndef USM_SPMM_GATHER_PERMILLE
#define USM_SPMM_GATHER_PERMILLE 30
#endif
#ifndef USM_SPMM_GATHER_N
#define USM_SPMM_GATHER_N 128
#endif
template <bool SMX>
int launch_gather(const SpmmArgs& a, const void* B, int ldb, cudaStream_t stream) {
    const long long warps_needed = a.M;
    long long blocks = (warps_needed + 7) / 8;
    const long long cap = 8LL * sm_count_current_device();
    if (blocks > cap) blocks = cap;
    spmm_gather_kernel<false, SMX><<<(int)blocks, 256, 0, stream>>>(a, B, ldb);
    return cudaGetLastError() == cudaSuccess ? USM_OK : USM_ERR_CUDA;
}

template <bool SMX>
int launch_shape(const SpmmArgs& a, const void* B, int ldb, bool bf16, cudaStream_t stream) {
    constexpr int W = 16, NS = USM_SPMM_STAGES, F = 2 / NS;  // F: chunk growth with one stage
    // Every kernel choice below depends on the problem (M, N, K, nnz, the
    // element type, the device's SM count), never on the schedule arguments
    // (swizzle, seg_rows), so those never change the result.
    const long long cells = (long long)a.M * a.K;
    {
        const ScheduleOverride ov = schedule_override();
        if (!bf16 && ov.rows_per_warp == 0 && ov.tiles_per_block == 0 && ov.k_splits == 0 &&
            a.N <= USM_SPMM_GATHER_N && 1000LL * a.nnz < (long long)USM_SPMM_GATHER_PERMILLE * cells)
            return launch_gather<SMX>(a, B, ldb, stream);
    }
    if (!bf16) {
#ifndef USM_SPMM_HS_PCT
#define USM_SPMM_HS_PCT 7
#endif
        // Sparse masks (under USM_SPMM_HS_PCT% set): up to 8 rows a warp on
        // 128-wide strips: 128-row tiles halve the staged rows a nonzero costs
        // and 384-row chunks double the nonzeros a (row, chunk) visit covers,
        // at the same registers.  Measured against 256-wide strips with up to 4
        // rows a warp: FFN 95% 6-11% faster, 90% -2..+3%, LSTM even.
        const bool sparse = 100LL * a.nnz < (long long)USM_SPMM_HS_PCT * cells;
        // fp32 masks at least 55% set: row groups (usm_spmm_group.cuh), where
        // a staged row of B serves all of a warp's rows holding its column.
        // Measured against the row kernel with tensor-memory rows (N = 2048,
        // one stream): 60% density 5% (4096x1024) and 9% (1024x4096) faster
        // (80%: 40%, against 16 warps); 50% density 5% slower (4096x1024);
        // 30-40% slower still (the predicated FMAs of the rows without a
        // column cost more than the loads saved), and so are grids whose
        // 64-row tiles cover under half the SMs (2048x2048, N = 512: 26%
        // slower).  64 < N <= 128 takes 128-column strips, where each column
        // carries half the FMAs for the same list work: 8192x4096, N = 128,
        // 50% density even, 60% 9% faster, 70% 23%, 90% 49%; 40% density 9%
        // slower.  K <= 6144 keeps its rounding bound.  The choice depends on
        // M, N, K, nnz only, never on the schedule arguments.
#ifndef USM_SPMM_GROUP
#define USM_SPMM_GROUP 1
#endif
#ifndef USM_GROUP_MIN_PCT
#define USM_GROUP_MIN_PCT 55
#endif
        auto groups = [&](int strip) {
            const long long ctas = (long long)((a.M + 63) / 64) * ((a.N + strip - 1) / strip);
            return USM_SPMM_GROUP && NS == 1 && a.K <= 6144 && 100LL * a.nnz >= USM_GROUP_MIN_PCT * cells &&
                   2 * ctas >= sm_count_current_device();
        };
        if (a.N <= 64) return launch_pick<false, 16, 4, W, 384 * F, NS, 1, 2, 4, false, SMX>(a, B, ldb, stream);
        if (a.N <= 128 && groups(128))
            return launch_pick<false, 32, 4, W, 384, 1, 1, 2, 4, false, SMX, true>(a, B, ldb, stream);
        // Warps a CTA.  128-wide strips with 2-4 rows a warp need 69-87
        // registers, under the 96 that 20 warps leave (five on a subpartition
        // of 16K registers), so 20 warps hide more of the loads' latency: LSTM sweep
        // (N = 128) 3-4% faster at 50-90% sparsity than with 16 (24 warps spill
        // and are slower).  The sparse-mask shape (up to 8 rows a warp) measured
        // mixed at 20 (-4..+2.5%) and slower at 24, so it keeps 16.
#ifndef USM_SPMM_W_N128
#define USM_SPMM_W_N128 20
#endif
#ifndef USM_SPMM_W_HS
#define USM_SPMM_W_HS 16
#endif
        // Chunk rows of the 128-wide shapes: 416 where that saves a chunk
        // against 384 (K = 4096: LSTM at 90-95% sparsity and FFN 1024x4096 at
        // 95% 2-3% faster; with K = 1024, where it saves none, 1-2% slower).
#ifndef USM_SPMM_KC128
#define USM_SPMM_KC128 (208 * F)
#endif
        const bool tall128 = taller_chunk_pays(a.K, 192 * F, USM_SPMM_KC128);
        auto sparse_shape = [&]() {
            if (tall128)
                return launch_pick<false, 32, 4, USM_SPMM_W_HS, USM_SPMM_KC128, NS, 1, 4, 8, false, SMX>(a, B, ldb, stream);
            return launch_pick<false, 32, 4, USM_SPMM_W_HS, 192 * F, NS, 1, 4, 8, false, SMX>(a, B, ldb, stream);
        };
        if (a.N <= 128) {
            if (sparse) return sparse_shape();
            if (tall128)
                return launch_pick<false, 32, 4, USM_SPMM_W_N128, USM_SPMM_KC128, NS, 1, 2, 4, false, SMX>(a, B, ldb,
                                                                                                        stream);
            return launch_pick<false, 32, 4, USM_SPMM_W_N128, 192 * F, NS, 1, 2, 4, false, SMX>(a, B, ldb, stream);
        }
#ifndef USM_SPMM_TMEM
#define USM_SPMM_TMEM 1
#endif
#ifndef USM_TM_MIN_DENSITY_PCT
#define USM_TM_MIN_DENSITY_PCT 15
#endif
#ifndef USM_TM_RB
#define USM_TM_RB 4
#endif
        if (groups(256)) return launch_pick<false, 32, 8, W, 192, 1, 1, 2, 4, false, SMX, true>(a, B, ldb, stream);
        // fp32 256-wide strips of masks at least 15% set (that row groups did
        // not take above): the last 64 rows of every chunk also go to tensor
        // memory.  Measured on the FFN launches: at 70% sparsity 6-8% faster
        // than shared memory alone (both at 16 warps; 18 warps then gained
        // another 3-10%); at 18 warps against the 20-warp shape below, 80%
        // 3-4% faster and 90% 5% slower (the copies and their waits are not
        // paid back), so the threshold sits between the two.  ResNet's
        // 512x2048 at 80% (N = 3136) measured 1% slower.
        // 256-wide strips without tensor-memory rows: 20 warps, the CSR windows
        // fetched a row slot ahead rather than kept (which leaves no spills),
        // against 16 warps with kept windows: FFN 4096x1024 4-7% faster at
        // 80-90% sparsity, 1024x4096 1% slower.  The tensor-memory shape runs
        // 18 warps at 96 registers (five warps on a subpartition, as with 20;
        // the CSR windows fetched a row slot ahead): FFN at 70% sparsity 3%
        // (1024x4096) and 9% (4096x1024) faster than 16 warps at 128 registers,
        // 1024x4096 at 50% 5%; 20 warps ran the same or up to 1% slower; 24
        // (80 registers, spilling) 11% slower than 16 on 1024x4096.
#ifndef USM_TM_W
#define USM_TM_W 18
#endif
#ifndef USM_SPMM_W256
#define USM_SPMM_W256 20
#endif
        // Chunk rows of the 256-wide shapes: 208 (a 208 KB stage, what the
        // shared memory leaves beside the lists) where that saves a chunk
        // against 192: 1-4% faster on the FFN launches at 80-90% sparsity and
        // about 1% with tensor-memory rows at 70-80% (ResNet 2%).
#ifndef USM_SPMM_KC256
#define USM_SPMM_KC256 (104 * F)
#endif
        const bool tall256 = taller_chunk_pays(a.K, 96 * F, USM_SPMM_KC256);
        if (!SMX && USM_SPMM_TMEM && NS == 1 && 100LL * a.nnz >= (long long)USM_TM_MIN_DENSITY_PCT * cells) {
            if (tall256)
                return launch_pick<false, 32, 8, USM_TM_W, USM_SPMM_KC256, NS, 1, 2, USM_TM_RB, NS == 1>(a, B, ldb,
                                                                                                      stream);
            return launch_pick<false, 32, 8, USM_TM_W, 96 * F, NS, 1, 2, USM_TM_RB, NS == 1>(a, B, ldb, stream);
        }
        if (sparse) return sparse_shape();
        if (tall256)
            return launch_pick<false, 32, 8, USM_SPMM_W256, USM_SPMM_KC256, NS, 1, 2, 4, false, SMX>(a, B, ldb, stream);
        return launch_pick<false, 32, 8, USM_SPMM_W256, 96 * F, NS, 1, 2, 4, false, SMX>(a, B, ldb, stream);
    }
    // bf16 warps and CTAs a SM.  256-wide strips: one CTA of 28 warps with one
    // 192 KB stage (twice the rows sharing each staged chunk, windows fetched
    // a row slot ahead rather than kept) against two CTAs of 16 with 96 KB
    // each: measured 2-16% faster on all six FFN launches that take it.
    // 128-wide strips (6% slower that way; 12% with one CTA of 20 warps that
    // keeps its windows) and N <= 64 (attention, 2% and 28% slower) keep two
    // CTAs of 16 warps.
#ifndef USM_SPMM_BF_W
#define USM_SPMM_BF_W 28
#endif
#ifndef USM_SPMM_BF_MB
#define USM_SPMM_BF_MB 1
#endif
#ifndef USM_SPMM_BF128_W
#define USM_SPMM_BF128_W 16
#endif
#ifndef USM_SPMM_BF128_MB
#define USM_SPMM_BF128_MB 2
#endif
#ifndef USM_SPMM_BF64_W
#define USM_SPMM_BF64_W 16
#endif
#ifndef USM_SPMM_BF64_MB
#define USM_SPMM_BF64_MB 2
#endif
    constexpr int BW = USM_SPMM_BF_W, BMB = USM_SPMM_BF_MB, BW1 = USM_SPMM_BF128_W, BMB1 = USM_SPMM_BF128_MB;
    constexpr int BW6 = USM_SPMM_BF64_W, BMB6 = USM_SPMM_BF64_MB;
    // (N <= 64 with 832-row chunks where they save a chunk: the attention
    // SpMM 0.6-1.6% slower, so 768.)
    if (a.N <= 64) return launch_pick<true, 16, 4, BW6, 768 * F / BMB6, NS, BMB6, 2, 4, false, SMX>(a, B, ldb, stream);
    // 128-wide strips (two CTAs of 96 KB): 416-row chunks where they save a
    // chunk against 384 (104 KB each), FFN 1024x4096 at 90-95% 2-3% faster.
#ifndef USM_SPMM_BF128_KC_TALL
#define USM_SPMM_BF128_KC_TALL (416 * F / BMB1)
#endif
#ifndef USM_SPMM_HS_BF_PCT
#define USM_SPMM_HS_BF_PCT 12
#endif
    // bf16 on sparse masks with long rows of B (K > 2048): 128-wide strips
    // (measured: 1024x4096 at 90% 4% faster, at 95% 12%; 4096x1024 1-8% slower).
    if (a.N <= 128 || (a.K > 2048 && 100LL * a.nnz < (long long)USM_SPMM_HS_BF_PCT * cells)) {
        if (taller_chunk_pays(a.K, 384 * F / BMB1, USM_SPMM_BF128_KC_TALL))
            return launch_pick<true, 32, 4, BW1, USM_SPMM_BF128_KC_TALL, NS, BMB1, 2, 4, false, SMX>(a, B, ldb, stream);
        return launch_pick<true, 32, 4, BW1, 384 * F / BMB1, NS, BMB1, 2, 4, false, SMX>(a, B, ldb, stream);
    }
    // 16 bf16 a lane (512-column strips in two TMA boxes, fewer instructions
    // per FMA) measured no faster at 70% and 6-25% slower at 90-95%.
    // bf16 rows in tensor memory (256 columns for each of the two CTAs an SM
    // holds, one tcgen05.ld.x4 a nonzero): measured 8-17% slower at 70%
    // sparsity and even at 80% (two CTAs of 64 registers do not hide the
    // loads' waits), so off by default.
#ifndef USM_SPMM_TMEM_BF
#define USM_SPMM_TMEM_BF 0
#endif
#ifndef USM_TM_RB_BF
#define USM_TM_RB_BF 4
#endif
    if (!SMX && USM_SPMM_TMEM_BF && NS == 1 && 100LL * a.nnz >= (long long)USM_TM_MIN_DENSITY_PCT * cells)
        return launch_pick<true, 32, 8, W, 96 * F, NS, 2, 2, USM_TM_RB_BF, NS == 1>(a, B, ldb, stream);
    // (Chunks of 416 or 432 rows where they save a chunk, as the fp32 shapes
    // and the bf16 SDDMM take: FFN 1024x4096 at 70-95% sparsity 1% faster to
    // 2% slower, so 384.)
    return launch_pick<true, 32, 8, BW, 192 * F / BMB, NS, BMB, 2, 4, false, SMX>(a, B, ldb, stream);
}

int launch_spmm(const SpmmArgs& a, const void* B, int ldb, bool bf16, cudaStream_t stream, bool softmax) {
    return softmax ? launch_shape<true>(a, B, ldb, bf16, stream) : launch_shape<false>(a, B, ldb, bf16, stream);
}

}  // namespace usm
