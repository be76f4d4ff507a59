// CSR SDDMM for sm_103a: out[p] = X[r]·Y[col_p] on the nonzeros of the mask.
//
// "Sparse GPU Kernels for Deep Learning" (Gale et al., SC 2020), summary
// card, "Interesting ideas" I3: the kernel drops the element-wise scaling by
// the mask's values and takes the second operand transposed (Y is K×D and
// the product is X·Yᵀ), the form weight gradients and sparse-attention
// scores need.  GB300 design:
//
// * Tiles.  A CTA owns up to R·W mask rows (dealt from the row-swizzle
//   order by the row scheduler, sched_pos; R, the tiles per block and the K
//   splits chosen at launch), one strip of DT columns of D and one range of
//   K chunks (grid z).  It walks its range in chunks of KC
//   rows; one thread copies Y[k0:k0+KC, d0:d0+DT] into a shared-memory stage
//   with TMA (mbarrier, bounded wait) into one tall stage: the tall chunks
//   halve the per-(row, chunk) work of a double-buffered layout.  One CTA
//   per SM with a stage of 192-216 KB: fp32 with 16 warps and up to 128 registers
//   (24 warps on 128-wide strips), bf16 with 28-32 warps of up to 72
//   registers (latency-bound: the warps cover each other's loads).
// * Per (row, chunk) a warp keeps X[r, d0:d0+DT] in registers (fp32), reads
//   the row's next 32 column indices (coalesced window after its cursor),
//   keeps the prefix inside the chunk and lists their stage offsets.
// * Dot products.  Lanes form G = 32/L groups of L lanes; at step t group g
//   takes list entry t·G+g and each lane multiplies its VV·EPV elements of
//   the staged Y row with its X elements (f32x2 FMA), leaving one partial per
//   step.  After L steps the L partials of each lane are reduced across the L
//   lanes of the group with a transpose-reduction (L-1 shuffles for L
//   results), so lane l of group g ends up with entry l·G+g's strip sum.
// * Strips.  With one strip the result goes straight to `out` (fp32 or bf16
//   rounded to nearest even).  With several, each strip writes fp32 partials
//   to the caller's workspace and a second kernel adds the strips in order:
//   no atomics, results are bit-reproducible.
// * Tensor-memory rows (TM, fp32 256-wide strips).  The last 64 rows of every
//   chunk are also copied into tensor memory (replicated in the four
//   subpartitions; lane t holds Y[k, 4t..4t+3] and Y[k, 128+4t..131+4t]).
//   Lane (g, l) of the 8-lane groups already holds, among its X words, the
//   X values of those columns for t = 8g + l (its words 4g.. and 4(g+4)..),
//   so a nonzero whose column lies in those rows is taken by the whole warp
//   at once: one tcgen05.ld per lane, eight products, an 8-lane
//   transpose-reduction over eight such nonzeros, then the four groups' sums
//   added with two shuffles.
#pragma once

#include <climits>

#include "usm_device.cuh"
#include "usm_args.h"


// SDDMM partials dropped from L2 by the strip sum once read (1), or left to
// be written back (0).  Measured in the FFN step: the SDDMM calls move 10-19%
// fewer DRAM bytes (1024x4096 at 70%: 71.4 -> 60.8 MB, 1.17x algorithmic),
// the SpMM calls after them up to 66% fewer, no change in time.  Storing the
// partials with L2 evict-last priority as well changed nothing more.
#ifndef USM_PARTIAL_DISCARD
#define USM_PARTIAL_DISCARD 1
#endif

namespace usm {
namespace {

template <bool BF, int L, int VV, int W, int KC, int MINB, int NS>
struct SddmmCfg {
    static constexpr int EPV = BF ? 8 : 4;      // elements per 16-byte vector
    static constexpr int DT = L * VV * EPV;     // D columns per CTA
    static constexpr int G = 32 / L;
    static constexpr int PITCH = L * VV * 16;   // bytes per staged Y row
    static constexpr int STAGE = KC * PITCH;
    static constexpr int BOX_ROWS = tma_box_rows(KC);
    static constexpr int THREADS = W * 32;
    static constexpr int SMEM = NS * STAGE + 64 + W * 32 * 4;
    static constexpr int XW = VV * 4;           // 32-bit words of X per lane
    static_assert(G * L == 32, "groups must tile the warp");
    static_assert(L == 8, "the list layout and reduction assume 8-lane groups");
    static_assert(KC % BOX_ROWS == 0 && BOX_ROWS <= 256, "TMA box height");
};

// Scaling by the mask's value at nonzero p (general SDDMM), 1 otherwise.
__device__ __forceinline__ float scale_at(const void* scale, int scale_bf16, long long p) {
    if (!scale) return 1.f;
    if (scale_bf16) return __uint_as_float((uint32_t)__ldg(reinterpret_cast<const unsigned short*>(scale) + p) << 16);
    return __ldg(reinterpret_cast<const float*>(scale) + p);
}

__device__ __forceinline__ int window_col(const SddmmArgs& a, int pos, int end, int lane) {
    const int p = pos + lane;
    return p < end ? __ldg(a.col_indices + p) : INT_MAX;
}

// X[r, d0 + j*L*EPV + l*EPV : +EPV] for j < VV as raw 32-bit words (fp32
// values, or packed bf16 pairs); zero beyond D or for a missing row.
template <bool BF, int L, int VV>
__device__ __forceinline__ void load_x(const SddmmArgs& a, int row, int d0, int l, uint32_t (&xw)[VV * 4]) {
    constexpr int EPV = BF ? 8 : 4;
#pragma unroll
    for (int j = 0; j < VV; ++j) {
        const int c = d0 + j * L * EPV + l * EPV;
        uint4 v = make_uint4(0u, 0u, 0u, 0u);
        if (row >= 0) {
            if (BF) {
                const unsigned short* x =
                    reinterpret_cast<const unsigned short*>(a.X) + (long long)row * a.ldx + c;
                if (c + EPV <= a.D) {
                    v = __ldg(reinterpret_cast<const uint4*>(x));
                } else {
                    uint32_t h[8];
#pragma unroll
                    for (int e = 0; e < 8; ++e) h[e] = (c + e < a.D) ? __ldg(x + e) : 0u;
                    v = make_uint4(h[0] | (h[1] << 16), h[2] | (h[3] << 16), h[4] | (h[5] << 16),
                                   h[6] | (h[7] << 16));
                }
            } else {
                const float* x = reinterpret_cast<const float*>(a.X) + (long long)row * a.ldx + c;
                if (c + EPV <= a.D) {
                    v = __ldg(reinterpret_cast<const uint4*>(x));
                } else {
                    uint32_t h[4];
#pragma unroll
                    for (int e = 0; e < 4; ++e)
                        h[e] = (c + e < a.D) ? __float_as_uint(__ldg(x + e)) : 0u;
                    v = make_uint4(h[0], h[1], h[2], h[3]);
                }
            }
        }
        xw[4 * j + 0] = v.x;
        xw[4 * j + 1] = v.y;
        xw[4 * j + 2] = v.z;
        xw[4 * j + 3] = v.w;
    }
}

// Partial dot product of one lane: its X words with the 16-byte vectors of
// one staged Y row.
template <bool BF, int L, int VV>
__device__ __forceinline__ float lane_dot(const uint32_t (&xw)[VV * 4], uint32_t yrow) {
    if constexpr (BF) {
        float s0 = 0.f, s1 = 0.f;
#pragma unroll
        for (int j = 0; j < VV; ++j) {
            const uint4 y = lds128(yrow + j * L * 16);
            const uint32_t yw[4] = {y.x, y.y, y.z, y.w};
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                s0 = fma_bf16(lo16(xw[4 * j + q]), lo16(yw[q]), s0);
                s1 = fma_bf16(hi16(xw[4 * j + q]), hi16(yw[q]), s1);
            }
        }
        return s0 + s1;
    } else {
        float2 s2 = make_float2(0.f, 0.f);
#pragma unroll
        for (int j = 0; j < VV; ++j) {
            const uint4 y = lds128(yrow + j * L * 16);
            s2 = __ffma2_rn(make_float2(__uint_as_float(xw[4 * j]), __uint_as_float(xw[4 * j + 1])),
                            make_float2(__uint_as_float(y.x), __uint_as_float(y.y)), s2);
            s2 = __ffma2_rn(make_float2(__uint_as_float(xw[4 * j + 2]), __uint_as_float(xw[4 * j + 3])),
                            make_float2(__uint_as_float(y.z), __uint_as_float(y.w)), s2);
        }
        return s2.x + s2.y;
    }
}

template <bool BF, int L, int VV, int W, int KC, int MINB, int NS, bool TM = false>
__global__ void __launch_bounds__(W * 32, MINB)
    sddmm_kernel(const __grid_constant__ CUtensorMap tmY, const SddmmArgs a) {
    using C_ = SddmmCfg<BF, L, VV, W, KC, MINB, NS>;
    constexpr int G = C_::G, PITCH = C_::PITCH, STAGE = C_::STAGE, XW = C_::XW;
    constexpr int TR = TM ? 64 : 0;  // chunk rows also in tensor memory (the last TR)
    constexpr int KL = KC - TR;      // chunk rows read from shared memory only
    static_assert(!TM || (!BF && L == 8 && VV == 8 && NS == 1 && MINB == 1 && KC > TR && TR % W == 0),
                  "tensor-memory rows: fp32 256-wide strips, one stage, one CTA per SM");

    extern __shared__ __align__(1024) unsigned char smem[];
    unsigned char* stages = smem;
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + NS * STAGE);  // [0..1] TMA, [4] TMEM copies
    int* kr = reinterpret_cast<int*>(smem + NS * STAGE + 16);  // [0..1] column range, [2] abort, [3] TMEM base
    uint32_t* lists = reinterpret_cast<uint32_t*>(smem + NS * STAGE + 64);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int g = lane / L, l = lane % L;
    const int R = a.rows_per_warp;  // ≤ 32
    const int tile = blockIdx.x;
    const int strip = blockIdx.y;
    const int d0 = strip * C_::DT;

    // The tile's chunks [c_lo, c_lo + nchunks) are split into gridDim.z
    // contiguous ranges, one per CTA on z: every nonzero falls in exactly one.
    // With one diagonal block the tile's span is all of K, known before any
    // load, so the first copy starts at once and the row look-ups overlap it;
    // block-diagonal schedules first find the tile's column range.
    const bool whole = a.seg_rows >= a.M;
    int c_lo = 0, nchunks = 0;
    auto split = [&](int lo, int hi) {  // columns [lo, hi] of the tile, hi >= lo
        const int per = (hi / KC - lo / KC + 1 + gridDim.z - 1) / gridDim.z;
        const int first = lo / KC + blockIdx.z * per;
        c_lo = first;
        nchunks = max(0, min(hi / KC + 1, first + per) - first);
    };
    if (whole && a.K > 0) split(0, a.K - 1);
    auto issue = [&](int j) {
        const int s = j % NS;
        const uint32_t bar = smem_addr(&bars[s]);
        mbar_arrive_expect_tx(bar, STAGE);
        const uint32_t dst = smem_addr(stages + s * STAGE);
#pragma unroll
        for (int b = 0; b < KC / C_::BOX_ROWS; ++b)
            tma_load_2d(dst + b * C_::BOX_ROWS * PITCH, &tmY, d0, (c_lo + j) * KC + b * C_::BOX_ROWS,
                        bar);
    };

    if constexpr (TM) {
        if (warp == 0) tmem_alloc(smem_addr(&kr[3]), 512);
    }
    if (threadIdx.x == 0) {
        kr[0] = INT_MAX;
        kr[1] = -1;
        kr[2] = 0;
        mbar_init(smem_addr(&bars[0]), 1);
        mbar_init(smem_addr(&bars[1]), 1);
        if (TM) mbar_init(smem_addr(&bars[4]), W);  // one commit per warp and chunk
        fence_barrier_init();
        prefetch_tensor_map(&tmY);
        if (whole) {
            if (nchunks > 0) issue(0);
            if (NS > 1 && nchunks > 1) issue(1);
        }
    }

    int my_row = -1, my_start = 0, my_end = 0;
    if (lane < R) {
        const long long m = sched_pos(tile, sched_slot(lane, warp, W), a.tiles_per_block, a.seg_rows, a.M);
        if (m >= 0) {
            const int r = a.perm ? __ldg(a.perm + m) : (int)m;
            if ((unsigned)r < (unsigned)a.M) {
                int s = __ldg(a.row_offsets + r), e = __ldg(a.row_offsets + r + 1);
                s = min(max(s, 0), a.nnz);
                e = min(max(e, s), a.nnz);
                my_row = r;
                my_start = s;
                my_end = e;
            }
        }
    }
    if (TM) tmem_fence_before_sync();
    if (whole) {
        __syncthreads();  // barrier and flag initialisation visible to every thread
    } else {
        int kmin = INT_MAX, kmax = -1;
        if (my_end > my_start) {
            kmin = __ldg(a.col_indices + my_start);
            kmax = __ldg(a.col_indices + my_end - 1);
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
            kmin = min(kmin, __shfl_xor_sync(kFullMask, kmin, o));
            kmax = max(kmax, __shfl_xor_sync(kFullMask, kmax, o));
        }
        __syncthreads();
        if (lane == 0 && kmax >= 0) {
            atomicMin(&kr[0], kmin);
            atomicMax(&kr[1], kmax);
        }
        __syncthreads();
        const int lo = max(kr[0], 0), hi = min(kr[1], a.K - 1);
        if (kr[1] >= 0 && lo <= hi) split(lo, hi);
        if (threadIdx.x == 0) {
            if (nchunks > 0) issue(0);
            if (NS > 1 && nchunks > 1) issue(1);
        }
    }
    // Later ranges start each row at its first nonzero in range (binary search
    // of the sorted column indices; lanes < R, overlapping the first copy).
    const bool later = blockIdx.z > 0 && nchunks > 0;
    if (later && my_end > my_start) {
        const int k_first = c_lo * KC;
        int lo = my_start, hi = my_end;  // first position with column >= k_first
        while (lo < hi) {
            const int mid = (lo + hi) >> 1;
            if (__ldg(a.col_indices + mid) < k_first) lo = mid + 1;
            else hi = mid;
        }
        my_start = lo;
    }

    int cur = my_start;
    // Prefetched state of the next row to process: its window and X strip.
    int pcol = window_col(a, __shfl_sync(kFullMask, cur, 0), __shfl_sync(kFullMask, my_end, 0), lane);
    uint32_t pxw[XW];
    load_x<BF, L, VV>(a, __shfl_sync(kFullMask, my_row, 0), d0, l, pxw);

    uint32_t* wl = lists + warp * 32;
    // Entry e of a window goes to slot (e % G)·L + e / G, so group g finds
    // its steps 0..L-1 contiguous at g·L and reads four per 128-bit load.
    const int my_slot = (lane % G) * L + lane / G;
    const uint32_t gl = smem_addr(wl + g * L);
    const bool single_strip = gridDim.y == 1;
    uint32_t tlane = 0;  // TM: this warp's tensor-memory lanes, column 0
    if constexpr (TM) {
        tmem_fence_after_sync();
        tlane = (uint32_t)kr[3] + ((uint32_t)(32 * (warp & 3)) << 16);
    }
    // The output (or partial) of nonzero p.
    auto emit = [&](long long p, float v) {
        if (single_strip) {
            const float w = a.scale ? v * scale_at(a.scale, a.scale_bf16, p) : v;
            if (a.out_bf16)
                reinterpret_cast<uint16_t*>(a.out)[p] = f32_to_bf16_rne(w);
            else
                reinterpret_cast<float*>(a.out)[p] = w;
        } else {
            reinterpret_cast<float*>(a.out)[(long long)strip * a.out_stride + p] = v;
        }
    };

    for (int j = 0; j < nchunks; ++j) {
        const int s = j % NS;
        const int k0 = (c_lo + j) * KC;
        // Warp-uniform: the row loop below is full of warp-wide operations.
        const bool ok = __all_sync(kFullMask, mbar_wait_bounded(smem_addr(&bars[s]), (j / NS) & 1, kWaitLimitNs));
        if (!ok) kr[2] = 1;
        const uint32_t stage0 = smem_addr(stages + s * STAGE);
        const uint32_t stage = stage0 + l * 16;
        bool tm_ready = false, tm_failed = false;  // TM: this chunk's tensor-memory rows have landed
        if constexpr (TM) {
            // Each warp copies its TR/W rows of the chunk's tensor-memory part
            // (two 512-byte halves a row) and commits.
            if (ok && lane == 0) {
#pragma unroll
                for (int q = 0; q < TR / W; ++q) {
                    const int rr = warp * (TR / W) + q;
                    tmem_cp_512b_x4((uint32_t)kr[3] + 8 * rr, stage0 + (KL + rr) * PITCH);
                    tmem_cp_512b_x4((uint32_t)kr[3] + 8 * rr + 4, stage0 + (KL + rr) * PITCH + 512);
                }
                tmem_commit(smem_addr(&bars[4]));
            }
        }
        if (ok) {
#pragma unroll 1
            for (int i = 0; i < R; ++i) {
                int rc = __shfl_sync(kFullMask, cur, i);
                const int re = __shfl_sync(kFullMask, my_end, i);
                int col = pcol;
                uint32_t xw[XW];
#pragma unroll
                for (int q = 0; q < XW; ++q) xw[q] = pxw[q];
                // TM: the X words for tensor-memory lane 8g + l (words 4g.. and 4(g+4)..).
                float xs[TM ? 8 : 1];
                if constexpr (TM) {
#pragma unroll
                    for (int q = 0; q < 4; ++q) {
                        uint32_t lo = xw[q], hi = xw[16 + q];
#pragma unroll
                        for (int gg = 1; gg < 4; ++gg) {
                            lo = g == gg ? xw[4 * gg + q] : lo;
                            hi = g == gg ? xw[4 * (gg + 4) + q] : hi;
                        }
                        xs[q] = __uint_as_float(lo);
                        xs[4 + q] = __uint_as_float(hi);
                    }
                }
                // Prefetch the next row slot (slot 0 for the next chunk: its
                // cursor is final once slot 0 has been processed, when R > 1;
                // for R == 1 the reload after the segment covers it).
                {
                    const int ni = (i + 1 < R) ? i + 1 : 0;
                    if (ni != i) {
                        pcol = window_col(a, __shfl_sync(kFullMask, cur, ni),
                                          __shfl_sync(kFullMask, my_end, ni), lane);
                        load_x<BF, L, VV>(a, __shfl_sync(kFullMask, my_row, ni), d0, l, pxw);
                    }
                }
                while (true) {
                    const bool valid = (rc + lane < re) && ((unsigned)(col - k0) < (unsigned)KC);
                    const unsigned bal = __ballot_sync(kFullMask, valid);
                    const int n = (bal == kFullMask) ? 32 : (__ffs(~bal) - 1);
                    if (n == 0) break;
                    // TM: the first n_sm entries lie in the chunk's shared-memory
                    // rows, the rest in its tensor-memory rows.
                    int n_sm = n;
                    if constexpr (TM) {
                        const unsigned smb = __ballot_sync(kFullMask, valid && (unsigned)(col - k0) < (unsigned)KL);
                        n_sm = (smb == kFullMask) ? 32 : (__ffs(~smb) - 1);
                    }
                    // A full window may continue: fetch the next one now so its
                    // latency overlaps this window's work.
                    const int ncol = (n == 32) ? window_col(a, rc + 32, re, lane) : INT_MAX;
                    if (n_sm > 0) {
                        wl[my_slot] = (lane < n_sm) ? (uint32_t)(col - k0) * PITCH : 0u;
                        __syncwarp();
                        float part[L];
#pragma unroll
                        for (int t4 = 0; t4 < L; t4 += 4) {
                            if (t4 * G < n_sm) {
                                const uint4 o4 = lds128(gl + t4 * 4);
                                const uint32_t off[4] = {o4.x, o4.y, o4.z, o4.w};
#pragma unroll
                                for (int u = 0; u < 4; ++u)
                                    part[t4 + u] = ((t4 + u) * G < n_sm) ? lane_dot<BF, L, VV>(xw, stage + off[u]) : 0.f;
                            } else {
#pragma unroll
                                for (int u = 0; u < 4; ++u) part[t4 + u] = 0.f;
                            }
                        }
                        // Transpose-reduce across the L lanes of each group: after it,
                        // lane l holds the group's sum for step l.
#pragma unroll
                        for (int off = L / 2; off >= 1; off >>= 1) {
                            const bool upper = (l & off) != 0;
#pragma unroll
                            for (int q = 0; q < off; ++q) {
                                const float send = upper ? part[q] : part[q + off];
                                const float keep = upper ? part[q + off] : part[q];
                                part[q] = keep + __shfl_xor_sync(kFullMask, send, off);
                            }
                        }
                        const int e = l * G + g;  // window entry whose sum this lane holds
                        if (e < n_sm) emit((long long)rc + e, part[0]);
                        __syncwarp();
                    }
                    if constexpr (TM) {
                        // Entries n_sm..n-1, Y rows from tensor memory, once this
                        // chunk's copies have landed (checked once per chunk).
                        if (n_sm < n && !tm_ready && !tm_failed) {
                            tm_ready = __all_sync(kFullMask, mbar_wait_bounded(smem_addr(&bars[4]), j & 1, kWaitLimitNs));
                            tm_failed = !tm_ready;
                            if (tm_failed) kr[2] = 1;
                            tmem_fence_after_sync();
                        }
                        if (tm_ready) {
#pragma unroll 1
                            for (int t0 = n_sm; t0 < n; t0 += 8) {
                                // Eight nonzeros, each taken by the whole warp: lane
                                // 8g + l multiplies its eight Y values by xs.
                                float tp[8];
#pragma unroll
                                for (int hb = 0; hb < 8; hb += 4) {
                                    uint32_t ad[4];
#pragma unroll
                                    for (int b = 0; b < 4; ++b) {
                                        const int c = __shfl_sync(kFullMask, col, min(t0 + hb + b, n - 1));
                                        ad[b] = tlane + (uint32_t)(c - k0 - KL) * 8u;
                                    }
                                    uint32_t w0[8], w1[8], w2[8], w3[8];
                                    tmem_ld8x4(ad[0], ad[1], ad[2], ad[3], w0, w1, w2, w3);
                                    auto dot8 = [&](const uint32_t (&w)[8]) {
                                        float2 s2 = make_float2(0.f, 0.f);
#pragma unroll
                                        for (int q = 0; q < 8; q += 2)
                                            s2 = __ffma2_rn(make_float2(xs[q], xs[q + 1]),
                                                            make_float2(__uint_as_float(w[q]), __uint_as_float(w[q + 1])), s2);
                                        return s2.x + s2.y;
                                    };
                                    tp[hb] = dot8(w0);
                                    tp[hb + 1] = dot8(w1);
                                    tp[hb + 2] = dot8(w2);
                                    tp[hb + 3] = dot8(w3);
                                }
                                // Transpose-reduce over the 8 lanes of each group (lane l
                                // then holds its group's sum for nonzero t0 + l), then add
                                // the four groups' sums.
#pragma unroll
                                for (int off = 4; off >= 1; off >>= 1) {
                                    const bool upper = (l & off) != 0;
#pragma unroll
                                    for (int q = 0; q < off; ++q) {
                                        const float send = upper ? tp[q] : tp[q + off];
                                        const float keep = upper ? tp[q + off] : tp[q];
                                        tp[q] = keep + __shfl_xor_sync(kFullMask, send, off);
                                    }
                                }
                                float v = tp[0];
                                v += __shfl_xor_sync(kFullMask, v, 8);
                                v += __shfl_xor_sync(kFullMask, v, 16);
                                if (g == 0 && t0 + l < n) emit((long long)rc + t0 + l, v);
                            }
                        }
                    }
                    rc += n;
                    if (n < 32) break;
                    col = ncol;
                }
                if (lane == i) cur = rc;
                if (R == 1) {
                    pcol = window_col(a, __shfl_sync(kFullMask, cur, 0), __shfl_sync(kFullMask, my_end, 0),
                                      lane);
                }
            }
        }
        if constexpr (TM) {
            // Every copy of this chunk has completed before the stage is refilled
            // (and the barrier's phase is consumed by every warp).
            if (ok && !tm_ready && !tm_failed && !mbar_wait_bounded(smem_addr(&bars[4]), j & 1, kWaitLimitNs))
                kr[2] = 1;
            tmem_fence_before_sync();
        }
        __syncthreads();
        if (TM) tmem_fence_after_sync();
        if (kr[2]) break;
        if (threadIdx.x == 0 && j + NS < nchunks) {
            fence_proxy_async_smem();
            issue(j + NS);
        }
    }

    if constexpr (TM) {
        // Every warp is past its last tensor-memory read: free the columns.
        tmem_fence_before_sync();
        __syncthreads();
        tmem_fence_after_sync();
        if (warp == 0) tmem_dealloc((uint32_t)kr[3], 512);
    }

    if (kr[2] && threadIdx.x == 0) {
        record_status(a.status, USM_ERR_TIMEOUT);
        for (int b = 0; b < NS && b < nchunks; ++b) {
            mbar_wait_bounded(smem_addr(&bars[b]), 0, 1000000ull);
            mbar_wait_bounded(smem_addr(&bars[b]), 1, 1000000ull);
        }
    }
}

// Strips are added in increasing order in runs of kStripRun: the strips of
// each run sequentially, then the run totals in order.  Up to kStripRun
// strips this is one sequential sum; beyond, it keeps the additions along an
// output's path to ≤ 63 + nstrips/64 (on top of ≤ 20 inside a strip), so the
// fp32 worst-case rounding bound holds for D up to about 680k columns.
constexpr int kStripRun = 64;

// out[p] = Σ_s partial[s][p] (strip s at part + s·stride), times the mask's
// value when scaling.
__global__ void sddmm_strip_sum_kernel(const float* __restrict__ part, long long nnz, long long stride,
                                       int nstrips, void* out, int out_bf16, const void* scale, int scale_bf16) {
    for (long long p = blockIdx.x * (long long)blockDim.x + threadIdx.x; p < nnz;
         p += (long long)gridDim.x * blockDim.x) {
        float s = 0.f;
        for (int k0 = 0; k0 < nstrips; k0 += kStripRun) {
            float t = part[(long long)k0 * stride + p];
            const int k1 = min(nstrips, k0 + kStripRun);
            for (int k = k0 + 1; k < k1; ++k) t += part[(long long)k * stride + p];
            s = k0 == 0 ? t : s + t;
        }
        if (scale) s *= scale_at(scale, scale_bf16, p);
        if (out_bf16)
            reinterpret_cast<uint16_t*>(out)[p] = f32_to_bf16_rne(s);
        else
            reinterpret_cast<float*>(out)[p] = s;
    }
}

// The same sum four nonzeros at a time with 16-byte loads of every strip's
// partials (stride a multiple of 32; partials, out and scale aligned to the
// vector): several loads in flight per thread instead of one.  The last
// group of four may run past nnz: its partials are in the strip's padding
// and its stores stop at nnz.  discard (partials 128-byte aligned): once a
// warp has added its groups, each 128-byte line of partials it read (eight
// groups, all this warp's, all inside one strip) is dropped from L2 without
// being written back — the partials are dead, and their write-back would
// be DRAM traffic for nothing.  The workspace's contents are undefined
// afterwards.
__global__ void sddmm_strip_sum4_kernel(const float* __restrict__ part, long long nnz, long long stride, int nstrips,
                                        void* out, int out_bf16, const void* scale, int scale_bf16, int discard) {
    const long long n4 = (nnz + 3) / 4, s4 = stride / 4;
    const float4* __restrict__ part4 = reinterpret_cast<const float4*>(part);
    const int lane = threadIdx.x & 31;
    // Warp-uniform trip count (the discard step needs the whole warp).
    for (long long base = blockIdx.x * (long long)blockDim.x + (threadIdx.x & ~31); base < n4;
         base += (long long)gridDim.x * blockDim.x) {
        const long long i = base + lane;
        const unsigned act = __ballot_sync(kFullMask, i < n4);  // the lanes with a group this round
        if (i >= n4) continue;
        float4 s = make_float4(0.f, 0.f, 0.f, 0.f);
        for (int k0 = 0; k0 < nstrips; k0 += kStripRun) {
            float4 t = __ldcs(part4 + (long long)k0 * s4 + i);
            const int k1 = min(nstrips, k0 + kStripRun);
#pragma unroll 4
            for (int k = k0 + 1; k < k1; ++k) {
                const float4 v = __ldcs(part4 + (long long)k * s4 + i);
                t.x += v.x;
                t.y += v.y;
                t.z += v.z;
                t.w += v.w;
            }
            if (k0 == 0) {
                s = t;
            } else {
                s.x += t.x;
                s.y += t.y;
                s.z += t.z;
                s.w += t.w;
            }
        }
        const long long p0 = 4 * i;
        if (p0 + 4 <= nnz) {
            if (scale) {
                if (scale_bf16) {
                    const uint2 b = __ldg(reinterpret_cast<const uint2*>(scale) + i);
                    s.x *= __uint_as_float(b.x << 16);
                    s.y *= __uint_as_float(b.x & 0xffff0000u);
                    s.z *= __uint_as_float(b.y << 16);
                    s.w *= __uint_as_float(b.y & 0xffff0000u);
                } else {
                    const float4 c = __ldg(reinterpret_cast<const float4*>(scale) + i);
                    s.x *= c.x;
                    s.y *= c.y;
                    s.z *= c.z;
                    s.w *= c.w;
                }
            }
            if (out_bf16) {
                const uint32_t lo = (uint32_t)f32_to_bf16_rne(s.x) | ((uint32_t)f32_to_bf16_rne(s.y) << 16);
                const uint32_t hi = (uint32_t)f32_to_bf16_rne(s.z) | ((uint32_t)f32_to_bf16_rne(s.w) << 16);
                reinterpret_cast<uint2*>(out)[i] = make_uint2(lo, hi);
            } else {
                reinterpret_cast<float4*>(out)[i] = s;
            }
        } else {  // the ragged last group: element by element up to nnz
            const float v[4] = {s.x, s.y, s.z, s.w};
            for (int u = 0; u < 4 && p0 + u < nnz; ++u) {
                const float w = scale ? v[u] * scale_at(scale, scale_bf16, p0 + u) : v[u];
                if (out_bf16)
                    reinterpret_cast<uint16_t*>(out)[p0 + u] = f32_to_bf16_rne(w);
                else
                    reinterpret_cast<float*>(out)[p0 + u] = w;
            }
        }
        if (discard) {
            // Every lane of the warp has its sums (the loads are consumed);
            // lanes at a line's first group drop that line in every strip.
            // The line's eight groups [i, i + 8) lie below s4 (a multiple of 8).
            __syncwarp(act);
            if ((i & 7) == 0)
                for (int k = 0; k < nstrips; ++k) l2_discard_line(part4 + (long long)k * s4 + i);
        }
    }
}

__global__ void fill_out_kernel(void* out, long long n, int bf16) {
    for (long long p = blockIdx.x * (long long)blockDim.x + threadIdx.x; p < n;
         p += (long long)gridDim.x * blockDim.x) {
        if (bf16)
            reinterpret_cast<uint16_t*>(out)[p] = 0;
        else
            reinterpret_cast<float*>(out)[p] = 0.f;
    }
}

// 32×32 tiles through shared memory (padded against bank conflicts).
template <typename T>
__global__ void dense_transpose_kernel(const T* __restrict__ src, long long lds, int rows, int cols,
                                       T* __restrict__ dst, long long ldd) {
    __shared__ T tile[32][33];
    const int c0 = blockIdx.x * 32, r0 = blockIdx.y * 32;
    for (int i = threadIdx.y; i < 32; i += blockDim.y) {
        const int r = r0 + i, c = c0 + threadIdx.x;
        if (r < rows && c < cols) tile[i][threadIdx.x] = src[(long long)r * lds + c];
    }
    __syncthreads();
    for (int i = threadIdx.y; i < 32; i += blockDim.y) {
        const int c = c0 + i, r = r0 + threadIdx.x;
        if (r < rows && c < cols) dst[(long long)c * ldd + r] = tile[threadIdx.x][i];
    }
}

}  // namespace
}  // namespace usm
