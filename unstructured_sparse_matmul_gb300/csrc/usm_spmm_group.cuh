// CSR SpMM on row groups (fp32, 256- or 128-column strips), for masks at
// least 55% set.
//
// "Sparse GPU Kernels for Deep Learning" (Gale et al., SC 2020), summary
// card "Summary": SpMM on plain CSR with 1-D row tiles.  The row-at-a-time
// kernel (usm_spmm_kernel.cuh) reads one staged element of B from shared
// memory for every useful FMA, and shared memory delivers a quarter of what
// the FP32 pipes consume.  Here a warp takes G rows together and walks the
// union of their columns: each staged row of B is read once for all the
// group's rows that hold that column (at 50% density with G = 4, 2.1
// nonzeros a load; at 80%, 3.2).
//
// * The CTA, its row slots (G a warp, dealt by the row scheduler), the
//   chunked TMA staging of B and the bounded waits are those of the row
//   kernel with one stage.
// * Per chunk the warp walks slabs of 32 columns.  Each row slot's entries
//   in the slab come from its 32-entry window of the CSR arrays (registers,
//   refilled from the cursor once half used; a window that may stop short of
//   the slab's last entry is reloaded from the cursor first) and become a
//   32-bit column mask (warp OR-reduction).
// * Lane l owns column l of the slab: it forms the column's row-slot mask,
//   and the columns any slot holds are listed in order (ballot and
//   population count), each with a header (staged-row offset | slot mask)
//   and the slots' values.
// * The list is walked in order, the next column's loads in flight while the
//   current one computes: the lane's 8 fp32 of the staged row (two 16-byte
//   loads) times each holding slot's value, into that slot's partial.  The
//   FMAs of slots without the column are predicated off, so no product of a
//   value that is absent is ever formed (infinities and NaNs in B reach
//   exactly the rows whose columns hold them).  Measured at 30% density, a
//   branch per column to code that does only the present slots' FMAs was
//   26% slower, and a branch per nonzero 32%.
// * Accuracy: a row's partial sums its ≤ 64 products of two slabs in column
//   order and is added into the row total after them, so ≤ 64 + ceil(K/64)
//   + 1 additions lie on any output's path: the worst-case rounding bound
//   (about one unit roundoff, 2^-24, per addition) stays below
//   1e-5·Σ|a||b| for K ≤ 6144 (the launch code takes this kernel only
//   there).  A row's additions and their order depend on its own columns
//   only, so results do not depend on which rows share a warp or a tile.
#pragma once

#include <climits>

#include "usm_spmm_kernel.cuh"

namespace usm {
namespace {

template <int KC, int W, int G, int VEC = 8>
struct GroupCfg {
    using Base = SpmmCfg<false, 32, VEC, G, W, KC, 1>;
    // A warp's list for one slab: 33 column headers (the last one empty, so
    // the walk may load one column ahead) and 33 x G values.
    static constexpr int HDR_BYTES = 144;
    static constexpr int LIST_BYTES = HDR_BYTES + 33 * G * 4;
    static constexpr int SMEM = Base::STAGE + 64 + W * LIST_BYTES;
    static constexpr int SLABS = KC / 32;
};

// c += x·w for the VEC fp32 of a lane (packed FMAs).
template <int VEC>
__device__ __forceinline__ void fma_vec(float (&c)[VEC], const uint32_t (&w)[VEC], float x) {
    const float2 a2 = make_float2(x, x);
#pragma unroll
    for (int q = 0; q < VEC; q += 2) {
        float2 c2 = make_float2(c[q], c[q + 1]);
        c2 = __ffma2_rn(a2, make_float2(__uint_as_float(w[q]), __uint_as_float(w[q + 1])), c2);
        c[q] = c2.x;
        c[q + 1] = c2.y;
    }
}

// VEC = 8: 256-column strips (two 16-byte loads a column); VEC = 4:
// 128-column strips (one).
template <int KC, int W, int G, int VEC = 8, bool SMX = false>
__global__ void __launch_bounds__(W * 32, 1)
    spmm_group_kernel(const __grid_constant__ CUtensorMap tmB, const SpmmArgs a) {
    using GC = GroupCfg<KC, W, G, VEC>;
    using C_ = typename GC::Base;
    constexpr int PITCH = C_::PITCH, STAGE = C_::STAGE, NCH = C_::NCH;
    constexpr int FOLD = 2;  // slabs summed in a partial before it joins the row total
    static_assert(KC % 32 == 0 && C_::NBOX == 1 && (VEC == 4 || VEC == 8) && PITCH == 128 * VEC &&
                      (G == 2 || G == 4 || G == 8),
                  "128- or 256-column fp32 strips, slabs of 32 rows, 2, 4 or 8 row slots a warp");

    extern __shared__ __align__(1024) unsigned char smem[];
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + STAGE);  // [0] TMA
    int* kr = reinterpret_cast<int*>(smem + STAGE + 16);        // [0]=min col, [1]=max col, [2]=abort
    unsigned char* wl = smem + STAGE + 64 + (threadIdx.x >> 5) * GC::LIST_BYTES;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int n0 = blockIdx.y * C_::NT;
    const int tile = blockIdx.x;

    // The chunk range: all of K under one diagonal block (the first copy
    // starts at once), else the span of the tile's columns.
    const bool whole = a.seg_rows >= a.M;
    int c_lo = 0, nchunks = whole ? (a.K + KC - 1) / KC : 0;
    auto issue = [&](int j) {
        const uint32_t bar = smem_addr(&bars[0]);
        mbar_arrive_expect_tx(bar, STAGE);
        const uint32_t dst = smem_addr(smem);
#pragma unroll
        for (int b = 0; b < KC / C_::BOX_ROWS; ++b)
            tma_load_2d(dst + b * C_::BOX_ROWS * PITCH, &tmB, n0, (c_lo + j) * KC + b * C_::BOX_ROWS, bar);
    };
    if (threadIdx.x == 0) {
        kr[0] = INT_MAX;
        kr[1] = -1;
        kr[2] = 0;
        mbar_init(smem_addr(&bars[0]), 1);
        fence_barrier_init();
        prefetch_tensor_map(&tmB);
        if (whole && nchunks > 0) issue(0);
    }

    // Row slots of this warp: lane i < G holds slot i's row and CSR range.
    int my_row = -1, my_start = 0, my_end = 0;
    if (lane < G) {
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
    if (whole) {
        __syncthreads();
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
        if (kr[1] >= 0 && lo <= hi) {
            c_lo = lo / KC;
            nchunks = hi / KC - c_lo + 1;
        }
        if (threadIdx.x == 0 && nchunks > 0) issue(0);
    }

    // SMX: each row's softmax statistics while the first copy is in flight;
    // lane i keeps slot i's.
    float my_m = 0.f, my_rz = 0.f;
    if constexpr (SMX) {
#pragma unroll 1
        for (int i = 0; i < G; ++i) {
            float m, rz;
            row_softmax_stats(reinterpret_cast<const float*>(a.values), __shfl_sync(kFullMask, my_start, i),
                              __shfl_sync(kFullMask, my_end, i), lane, m, rz);
            if (lane == i) {
                my_m = m;
                my_rz = rz;
            }
        }
    }

    // Every lane keeps every slot's cursor, end and window base (warp-uniform
    // values), so the per-slab work needs no shuffles for them.
    int rcur[G], rend[G], wb[G];
    int wcol[G];  // slot i's window: lane e holds nonzero wb[i] + e
    uint32_t wval[G];
#pragma unroll
    for (int i = 0; i < G; ++i) {
        rcur[i] = wb[i] = __shfl_sync(kFullMask, my_start, i);
        rend[i] = __shfl_sync(kFullMask, my_end, i);
        load_window<false, SMX>(a, wb[i], rend[i], lane, wcol[i], wval[i]);
    }

    float acc[G][VEC];  // row totals
    float cs[G][VEC];   // partials of the last ≤ FOLD slabs
#pragma unroll
    for (int i = 0; i < G; ++i)
#pragma unroll
        for (int v = 0; v < VEC; ++v) acc[i][v] = cs[i][v] = 0.f;

    const uint32_t hdr_addr = smem_addr(wl);                // column headers
    const uint32_t val_addr = hdr_addr + GC::HDR_BYTES;      // G values a column
    const uint32_t stage = smem_addr(smem) + 16 * lane;      // the lane's first 16-byte piece of a staged row
    const unsigned below = (1u << lane) - 1u;
    int since_fold = 0;  // slabs added into the partials since the last fold

    for (int j = 0; j < nchunks; ++j) {
        const int k0 = (c_lo + j) * KC;
        const bool ok = __all_sync(kFullMask, mbar_wait_bounded(smem_addr(&bars[0]), j & 1, kWaitLimitNs));
        if (!ok) kr[2] = 1;
        if (ok) {
#pragma unroll 1
            for (int sl = 0; sl < GC::SLABS; ++sl) {
                const int slab0 = k0 + 32 * sl;
                unsigned mask[G];  // slot i's columns in the slab (bit l: column slab0 + l)
                int wo[G];         // window lane of slot i's first entry in the slab
#pragma unroll
                for (int i = 0; i < G; ++i) {
                    // The window entries from the cursor whose columns fall in
                    // the slab: a run, as columns are sorted.
                    int w0 = rcur[i] - wb[i];
                    bool in = lane >= w0 && lane < rend[i] - wb[i] && (unsigned)(wcol[i] - slab0) < 32u;
                    unsigned bal = __ballot_sync(kFullMask, in);
                    if ((bal >> 31) && w0 > 0) {
                        // The run reaches the window's end: reload the window
                        // from the cursor so it holds the whole slab (≤ 32 entries).
                        wb[i] = rcur[i];
                        load_window<false, SMX>(a, wb[i], rend[i], lane, wcol[i], wval[i]);
                        w0 = 0;
                        in = lane < rend[i] - wb[i] && (unsigned)(wcol[i] - slab0) < 32u;
                        bal = __ballot_sync(kFullMask, in);
                    }
                    wo[i] = w0;
                    rcur[i] += __popc(bal);
                    mask[i] = __reduce_or_sync(kFullMask, in ? 1u << ((wcol[i] - slab0) & 31) : 0u);
                }
                // Lane l: the row slots holding column slab0 + l.  The slab's
                // columns held by any slot, in order, each with a header
                // (staged-row offset | slot mask) and the slots' values
                // (undefined for slots without the column).
                unsigned cm = 0;
#pragma unroll
                for (int i = 0; i < G; ++i) cm |= ((mask[i] >> lane) & 1u) << i;
                const unsigned present = __ballot_sync(kFullMask, cm != 0u);
                const int ucols = __popc(present);
                const int pos = __popc(present & below);
                uint32_t v[G];
#pragma unroll
                for (int i = 0; i < G; ++i) {
                    // shfl takes the source lane modulo 32
                    v[i] = __shfl_sync(kFullMask, wval[i], wo[i] + __popc(mask[i] & below));
                    if constexpr (SMX)
                        v[i] = value_bits<false, true>(v[i], __shfl_sync(kFullMask, my_m, i),
                                                       __shfl_sync(kFullMask, my_rz, i));
                }
                if (lane == 0) reinterpret_cast<uint32_t*>(wl)[ucols] = 0u;  // the empty header after the last
                if (cm) {
                    reinterpret_cast<uint32_t*>(wl)[pos] = (uint32_t)(32 * sl + lane) * PITCH | cm;
                    uint32_t* vd = reinterpret_cast<uint32_t*>(wl + GC::HDR_BYTES) + pos * G;
                    if constexpr (G == 2) {
                        *reinterpret_cast<uint2*>(vd) = make_uint2(v[0], v[1]);
                    } else {
#pragma unroll
                        for (int i = 0; i < G; i += 4)
                            *reinterpret_cast<uint4*>(vd + i) = make_uint4(v[i], v[i + 1], v[i + 2], v[i + 3]);
                    }
                }
                // A window half used is refilled now, its load landing while
                // the columns below are walked.
#pragma unroll
                for (int i = 0; i < G; ++i) {
                    if (rcur[i] - wb[i] >= 16 && rcur[i] < rend[i]) {
                        wb[i] = rcur[i];
                        load_window<false, SMX>(a, wb[i], rend[i], lane, wcol[i], wval[i]);
                    }
                }
                __syncwarp();

                // One column: the lane's VEC fp32 of its staged row, times each
                // holding slot's value, into that slot's partial (predicated
                // on the slot mask: slots without the column do no FMA).
                auto load_col = [&](int u, uint32_t& h, uint32_t (&w)[VEC], uint32_t (&x)[G]) {
                    h = lds32(hdr_addr + 4 * u);
                    const uint32_t off = h & ~(uint32_t)(PITCH - 1);
#pragma unroll
                    for (int c = 0; c < NCH; ++c) {
                        const uint4 b = lds128(stage + off + C_::piece_off(c));
                        w[4 * c] = b.x; w[4 * c + 1] = b.y; w[4 * c + 2] = b.z; w[4 * c + 3] = b.w;
                    }
                    if constexpr (G == 2) {
                        const uint2 q = lds64(val_addr + u * 8);
                        x[0] = q.x;
                        x[1] = q.y;
                    } else {
#pragma unroll
                        for (int i = 0; i < G; i += 4) {
                            const uint4 q = lds128(val_addr + (u * G + i) * 4);
                            x[i] = q.x; x[i + 1] = q.y; x[i + 2] = q.z; x[i + 3] = q.w;
                        }
                    }
                };
                auto fma_col = [&](uint32_t h, const uint32_t (&w)[VEC], const uint32_t (&x)[G]) {
#pragma unroll
                    for (int i = 0; i < G; ++i)
                        if (h & (1u << i)) fma_vec<VEC>(cs[i], w, __uint_as_float(x[i]));
                };
                // Software-pipelined: column u + 1 (or the empty header past
                // the last, whose mask does nothing) loads while column u's
                // FMAs run.
                uint32_t h0, h1, w0[VEC], w1[VEC], x0[G], x1[G];
                if (ucols > 0) load_col(0, h0, w0, x0);
#pragma unroll 1
                for (int u = 0; u < ucols; u += 2) {
                    load_col(u + 1, h1, w1, x1);
                    fma_col(h0, w0, x0);
                    if (u + 1 == ucols) break;
                    load_col(u + 2, h0, w0, x0);
                    fma_col(h1, w1, x1);
                }
                __syncwarp();
                // Every FOLD slabs (≤ 32·FOLD products) the partials go into
                // the row totals.
                if (++since_fold == FOLD) {
                    since_fold = 0;
#pragma unroll
                    for (int i = 0; i < G; ++i)
#pragma unroll
                        for (int q = 0; q < VEC; q += 2) {
                            const float2 s2 = __fadd2_rn(make_float2(acc[i][q], acc[i][q + 1]),
                                                         make_float2(cs[i][q], cs[i][q + 1]));
                            acc[i][q] = s2.x;
                            acc[i][q + 1] = s2.y;
                            cs[i][q] = cs[i][q + 1] = 0.f;
                        }
                }
            }
        }
        __syncthreads();  // every warp is done with the stage
        if (kr[2]) break;
        if (threadIdx.x == 0 && j + 1 < nchunks) {
            fence_proxy_async_smem();
            issue(j + 1);
        }
    }

    if (kr[2]) {
        // A transfer never completed: record it, wait (bounded) for a copy
        // still in flight so none lands after the CTA exits, and leave.
        if (threadIdx.x == 0) {
            record_status(a.status, USM_ERR_TIMEOUT);
            if (nchunks > 0) {
                mbar_wait_bounded(smem_addr(&bars[0]), 0, 1000000ull);
                mbar_wait_bounded(smem_addr(&bars[0]), 1, 1000000ull);
            }
        }
        return;
    }

#pragma unroll
    for (int i = 0; i < G; ++i)
#pragma unroll
        for (int q = 0; q < VEC; ++q) acc[i][q] += cs[i][q];  // the last partials

#pragma unroll
    for (int i = 0; i < G; ++i) {
        const int row = __shfl_sync(kFullMask, my_row, i);
        if (row < 0) continue;
        float* crow = a.C + (long long)row * a.ldc + n0;
#pragma unroll
        for (int v = 0; v < VEC; v += 4) {
            const int c = lane_col<32, VEC, 4>(lane, v);
            if (n0 + c + 4 <= a.N) {
                *reinterpret_cast<float4*>(crow + c) = make_float4(acc[i][v], acc[i][v + 1], acc[i][v + 2], acc[i][v + 3]);
            } else {
#pragma unroll
                for (int u = 0; u < 4; ++u)
                    if (n0 + c + u < a.N) crow[c + u] = acc[i][v + u];
            }
        }
    }
}

}  // namespace
}  // namespace usm
