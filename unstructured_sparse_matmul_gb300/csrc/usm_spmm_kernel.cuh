// CSR SpMM, C = A·B, for sm_103a.
//
// "Sparse GPU Kernels for Deep Learning" (Gale et al., SC 2020), summary
// card "Summary": SpMM on plain CSR with 1-D tiling, vector memory access on
// misaligned sparse rows and a load-balancing order kept apart from how the
// work is split ("Interesting ideas" I4).  The design below is written for
// GB300, not taken from the V100 kernels:
//
// * 1-D tiles.  A CTA owns one row tile (at most R·W rows of A) and one
//   strip of NT output columns; the row scheduler (sched_pos) deals the
//   row-swizzle order out to tiles and warps boustrophedon-fashion, so every
//   tile and warp gets a similar mix of row lengths even when lengths are
//   skewed (the launch code picks R and the tiles per block).  Each output
//   element is accumulated by exactly one lane group in a fixed order:
//   results do not depend on the swizzle or the tile shape.  bf16 runs two CTAs per SM, so one CTA's barrier waits and
//   prologue overlap the other's arithmetic; fp32, bound by shared-memory
//   bandwidth, runs one CTA per SM with more registers and a taller stage.
// * Dense operand staging.  The CTA walks K in chunks of KC rows.  For each
//   chunk one thread issues TMA tensor copies of B[k0:k0+KC, n0:n0+NT] into a
//   shared-memory stage (completion on an mbarrier, bounded wait; one or two
//   stages).  Under a block-diagonal schedule only the chunks between the
//   smallest and largest column index of the CTA's rows are fetched, so
//   batched matrices stay cheap; with one block the CTA walks all of K and
//   starts its first copy before looking its rows up.
// * Sparse operand.  For each (row, chunk) a warp reads the next 32 column
//   indices and values of the row with coalesced loads (the window after the
//   row's cursor, so a misaligned row start costs nothing), keeps the prefix
//   whose columns fall in the chunk (ballot) and writes (stage offset, value)
//   entries to a per-warp list.  With one CTA per SM each row slot keeps its
//   window in registers across chunks (refilled from the cursor once half
//   used); with two, the next row slot's window is fetched while the current
//   one computes.
// * Inner loop.  G = 32/L lane groups split the list into contiguous blocks.
//   Four steps at a time a group reads its four entries with 128-bit
//   broadcast loads (then 0-3 single steps), each lane reads 8, 16 or 32
//   bytes of the staged B row (a group covers whole rows, conflict-free) and
//   does VEC FMAs: packed f32x2 FMA for fp32, fma.rn.f32.bf16 on the bf16
//   halves for bf16 (one instruction an element: splitting the pairs to fp32
//   for packed FMAs measured 10-25% slower).  The G partial rows are added
//   across groups at the end.
// * Accuracy.  In fp32 each window of ≤ 32 nonzeros is summed into a fresh
//   accumulator, windows are added into a per-(row, chunk) partial and those
//   into the row total: ≤ 32 + KC/32 + 1 + K/KC additions lie along any
//   output's path, which keeps the worst-case rounding bound (about one unit
//   roundoff, 2^-24, per addition) below 1e-5·Σ|a||b| while K/KC ≤ 128.
//   Longer K (LONGK) adds one more level: every 64 chunks the row total is
//   moved into a second accumulator, so the path is ≤ 32 + KC/32 + 1 + 64 +
//   K/(64·KC) additions (the bound holds to K ≈ 786k with KC = 192).
#pragma once

#include <climits>
#include <type_traits>

// Tensor-memory reads in software-pipelined pairs (1) or batches of four
// behind one wait (0, measured faster: the pairs need more registers).
#ifndef USM_TM_PIPE
#define USM_TM_PIPE 0
#endif

#include "usm_device.cuh"
#include "usm_args.h"

namespace usm {
namespace {

template <bool BF, int L, int VEC, int R, int W, int KC, int NS, bool TM = false, bool VL = false>
struct SpmmCfg {
    static constexpr int ES = BF ? 2 : 4;          // element bytes
    static constexpr int NT = L * VEC;             // output columns per CTA (VEC per lane)
    static constexpr int G = 32 / L;               // lane groups (nonzeros per warp step)
    static constexpr int LANE_BYTES = VEC * ES;    // B bytes per lane per step
    static constexpr int NCH = LANE_BYTES / 16;    // 16-byte loads per lane per step (0: one 8-byte load)
    // The stage holds NBOX TMA boxes side by side in memory, each KC rows of
    // BOX_COLS columns (a box is at most 256 elements wide).
    static constexpr int BOX_COLS = NT <= 256 ? NT : 256;
    static constexpr int NBOX = NT / BOX_COLS;
    static constexpr int PITCH = BOX_COLS * ES;    // bytes per staged row of one box
    static constexpr int NW = LANE_BYTES / 4;      // 32-bit words per lane per step
    static constexpr int BOX_BYTES = KC * PITCH;
    static constexpr int STAGE = NBOX * BOX_BYTES;
    static constexpr int BOX_ROWS = tma_box_rows(KC);
    static constexpr int THREADS = W * 32;
    // List entries.  fp32: (stage offset, value bits), 8 bytes.  bf16 with
    // 8-byte lane slices (ADDR): an array of shared-memory row addresses and
    // one of bf16 values, 6 bytes, so a step needs one add for its address.
    // bf16 with 16-byte slices: offset/8 | value << 16 in 4 bytes (the extra
    // value load of the split form cost more than its saved arithmetic there).
    static constexpr bool ADDR = BF && NCH == 0;
    static constexpr int ENTRY = ADDR ? 6 : (BF ? 4 : 8);
    // A warp's list: 32 slots (one window); TM adds 32 for tensor-memory
    // entries; VL windows hold 128 entries.
    static constexpr int LIST_SLOTS = VL ? 128 : (TM ? 64 : 32);
    static constexpr int LIST_BYTES = W * LIST_SLOTS * ENTRY;
    static constexpr int SMEM = NS * STAGE + 64 + LIST_BYTES;
    static_assert(NS == 1 || NS == 2, "one or two stages");
    static_assert(32 % L == 0, "L must divide the warp");
    static_assert(KC % BOX_ROWS == 0 && BOX_ROWS <= 256, "TMA box height");
    static_assert(LANE_BYTES == 8 || LANE_BYTES == 16 || LANE_BYTES == 32, "8, 16 or 32 bytes per lane");
    // Byte offset, from a staged row's start in box 0, of 16-byte piece c of
    // a lane's slice (lane offset excluded): piece c covers bytes
    // [c·L·16, (c+1)·L·16) of the row, which may lie in a later box.
    static constexpr int piece_off(int c) { return (c * L * 16) / PITCH * BOX_BYTES + (c * L * 16) % PITCH; }
    static_assert(NT % BOX_COLS == 0 && (NCH == 0 || PITCH % (L * 16) == 0), "16-byte pieces tile the boxes");
    static_assert(!BF || ADDR || BOX_BYTES / 8 < 65536, "packed bf16 offsets are 16-bit multiples of 8 bytes");
};

// Output column (within the strip) of element v of lane l.  8-byte lanes own
// VEC contiguous columns; wider lanes own one 16-byte chunk per L·16-byte
// slice of the staged row, so every warp-wide load reads contiguous bytes.
template <int L, int VEC, int ES>
__device__ __forceinline__ int lane_col(int l, int v) {
    constexpr int EPC = 16 / ES;
    if constexpr (VEC * ES == 8) return l * VEC + v;
    return (v / EPC) * L * EPC + l * EPC + (v % EPC);
}

// Window of 32 consecutive nonzeros of a row starting at `pos`: lane i gets
// nonzero pos+i (column INT_MAX past the row end).  SMX: val holds the raw
// fp32 score; value_bits turns it into the probability when the entry is
// listed (so the load's latency stays hidden behind other work).
template <bool BF, bool SMX = false>
__device__ __forceinline__ void load_window(const SpmmArgs& a, int pos, int end, int lane, int& col,
                                            uint32_t& val) {
    const int p = pos + lane;
    if (p < end) {
        col = __ldg(a.col_indices + p);
        if constexpr (SMX) {
            val = __ldg(reinterpret_cast<const unsigned int*>(a.values) + p);
        } else if (BF) {
            val = __ldg(reinterpret_cast<const unsigned short*>(a.values) + p);
        } else {
            val = __ldg(reinterpret_cast<const unsigned int*>(a.values) + p);
        }
    } else {
        col = INT_MAX;
        val = 0;
    }
}

// The value bits a list entry carries: the stored value, or (SMX) the row's
// softmax probability of the score (maximum m, reciprocal sum rz) rounded to
// B's element type.
template <bool BF, bool SMX>
__device__ __forceinline__ uint32_t value_bits(uint32_t val, float m, float rz) {
    if constexpr (SMX) {
        const float v = softmax_prob(__uint_as_float(val), m, rz);
        return BF ? (uint32_t)f32_to_bf16_rne(v) : __float_as_uint(v);
    }
    return val;
}

// VL: window of 128 consecutive nonzeros starting at `base` (a multiple of
// 4, at or before the row cursor): lane i gets nonzeros base+4i..base+4i+3
// with one 16-byte load of column indices and one 16-byte (fp32) or 8-byte
// (bf16) load of values, when all four lie before the row end; else the ones
// that do, one by one (column INT_MAX past the row end).  The entries before
// the cursor (the misaligned start's residue) are loaded but never used:
// the caller masks them by position.  Needs col_indices 16-byte aligned and
// values 16-byte (fp32) or 8-byte (bf16) aligned; base >= 0 keeps every
// load inside the arrays.
template <bool BF, bool SMX = false>
__device__ __forceinline__ void load_window_v(const SpmmArgs& a, int base, int end, int lane, int (&col)[4],
                                              uint32_t (&val)[4]) {
    const int p = base + 4 * lane;
    if (!SMX && p + 4 <= end) {
        const int4 c = __ldg(reinterpret_cast<const int4*>(a.col_indices + p));
        col[0] = c.x;
        col[1] = c.y;
        col[2] = c.z;
        col[3] = c.w;
        if constexpr (BF) {
            const uint2 v = __ldg(reinterpret_cast<const uint2*>(reinterpret_cast<const unsigned short*>(a.values) + p));
            val[0] = v.x & 0xffffu;
            val[1] = v.x >> 16;
            val[2] = v.y & 0xffffu;
            val[3] = v.y >> 16;
        } else {
            const uint4 v = __ldg(reinterpret_cast<const uint4*>(reinterpret_cast<const unsigned int*>(a.values) + p));
            val[0] = v.x;
            val[1] = v.y;
            val[2] = v.z;
            val[3] = v.w;
        }
    } else {
#pragma unroll
        for (int u = 0; u < 4; ++u) {
            int c;
            uint32_t v;
            load_window<BF, SMX>(a, p + u - lane, end, lane, c, v);  // nonzero p + u
            col[u] = c;
            val[u] = v;
        }
    }
}

template <bool BF, int L, int VEC, int R, int W, int KC, int NS, int MB, bool LONGK = false, bool TM = false,
          bool SMX = false, bool VL = false>
__global__ void __launch_bounds__(W * 32, MB)
    spmm_kernel(const __grid_constant__ CUtensorMap tmB, const SpmmArgs a) {
    using C_ = SpmmCfg<BF, L, VEC, R, W, KC, NS, TM, VL>;
    constexpr int NCH = C_::NCH, NW = C_::NW;
    constexpr int G = C_::G, PITCH = C_::PITCH, STAGE = C_::STAGE, ENTRY = C_::ENTRY;
    constexpr bool ADDR = C_::ADDR;
    // TM: the last TR rows of every chunk are also copied into tensor memory
    // (replicated in the four subpartitions: lane t of every subpartition
    // holds the lane's 8 fp32 of each row, columns 8·row .. 8·row+7), and
    // nonzeros in those rows read B from there instead of shared memory.
    // fp32: 8 columns a row (two 512-byte halves), all 512 columns of the SM;
    // bf16: 4 columns a row (one 512-byte row), 256 columns for each of the
    // two CTAs an SM holds.
    constexpr int TR = TM ? 64 : 0;
    constexpr int KL = KC - TR;  // chunk rows read from shared memory
    constexpr int TCPR = BF ? 4 : 8;         // tensor-memory columns a row
    constexpr uint32_t TCOLS = BF ? 256 : 512;  // columns allocated
    static_assert(!TM || (L == 32 && VEC == 8 && NS == 1 && MB == (BF ? 2 : 1) && KC > TR && TR >= W &&
                          TR * TCPR == (int)TCOLS),
                  "tensor-memory rows: 32 lanes x 16 or 32 bytes, one stage, 1 (fp32) or 2 (bf16) CTAs per SM");
    static_assert(!VL || (G == 1 && !TM), "vector windows: one lane group, no tensor-memory rows");

    extern __shared__ __align__(1024) unsigned char smem[];
    unsigned char* stages = smem;
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + NS * STAGE);  // [0..1] TMA, [4] TMEM copies
    int* kr = reinterpret_cast<int*>(smem + NS * STAGE + 16);  // [0]=min col, [1]=max col, [2]=abort, [3]=TMEM base
    unsigned char* lists = smem + NS * STAGE + 64;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int g = lane / L, l = lane % L;
    const int n0 = blockIdx.y * C_::NT;
    const int tile = blockIdx.x;

    // With one diagonal block every tile may touch any column: the chunk range
    // is all of K, known before any load, so the first copy starts at once and
    // the row look-ups below overlap it.  Block-diagonal schedules first find
    // the tile's column range (a block touches only its own columns).
    const bool whole = a.seg_rows >= a.M;
    int c_lo = 0, nchunks = whole ? (a.K + KC - 1) / KC : 0;
    auto issue = [&](int j) {
        const int s = j % NS;
        const uint32_t bar = smem_addr(&bars[s]);
        mbar_arrive_expect_tx(bar, STAGE);
        const uint32_t dst = smem_addr(stages + s * STAGE);
#pragma unroll
        for (int x = 0; x < C_::NBOX; ++x)
#pragma unroll
            for (int b = 0; b < KC / C_::BOX_ROWS; ++b)
                tma_load_2d(dst + x * C_::BOX_BYTES + b * C_::BOX_ROWS * PITCH, &tmB, n0 + x * C_::BOX_COLS,
                            (c_lo + j) * KC + b * C_::BOX_ROWS, bar);
    };

    if constexpr (TM) {
        if (warp == 0) tmem_alloc(smem_addr(&kr[3]), TCOLS);
    }
    if (threadIdx.x == 0) {
        kr[0] = INT_MAX;
        kr[1] = -1;
        kr[2] = 0;
        mbar_init(smem_addr(&bars[0]), 1);
        mbar_init(smem_addr(&bars[1]), 1);
        if (TM) mbar_init(smem_addr(&bars[4]), W);  // one commit per warp and chunk
        fence_barrier_init();
        prefetch_tensor_map(&tmB);
        if (whole) {
            if (nchunks > 0) issue(0);
            if (NS > 1 && nchunks > 1) issue(1);
        }
    }

    // Row slots of this warp: slot i is row perm[tile*MT + i*W + warp].
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
        if (kr[1] >= 0 && lo <= hi) {
            c_lo = lo / KC;
            nchunks = hi / KC - c_lo + 1;
        }
        if (threadIdx.x == 0) {
            if (nchunks > 0) issue(0);
            if (NS > 1 && nchunks > 1) issue(1);
        }
    }

    // SMX: each row's softmax statistics (warp-cooperative, while the first
    // chunk's copy is in flight); lane i keeps row slot i's.
    float my_m = 0.f, my_rz = 0.f;
    if constexpr (SMX) {
#pragma unroll 1
        for (int i = 0; i < R; ++i) {
            float m, rz;
            row_softmax_stats(reinterpret_cast<const float*>(a.values), __shfl_sync(kFullMask, my_start, i),
                              __shfl_sync(kFullMask, my_end, i), lane, m, rz);
            if (lane == i) {
                my_m = m;
                my_rz = rz;
            }
        }
    }
    // The window of row slot `slot` from position pos (warp-wide call).
    auto window = [&](int, int pos, int end, int& col, uint32_t& val) { load_window<BF, SMX>(a, pos, end, lane, col, val); };

    float acc[R][VEC];
    float acc_hi[LONGK ? R : 1][LONGK ? VEC : 1];  // LONGK: totals of whole 64-chunk runs
#pragma unroll
    for (int i = 0; i < R; ++i)
#pragma unroll
        for (int v = 0; v < VEC; ++v) acc[i][v] = 0.f;
    if constexpr (LONGK) {
#pragma unroll
        for (int i = 0; i < R; ++i)
#pragma unroll
            for (int v = 0; v < VEC; ++v) acc_hi[i][v] = 0.f;
    }

    int cur = my_start;  // lane i: cursor of row slot i
    // PERSIST (one CTA per SM with registers to spare: up to 20 warps with 4
    // elements a lane, 16 with 8): each row slot keeps a 32-entry window of
    // its CSR arrays in registers across chunks (lane e holds entry wb[i] +
    // e), so at high sparsity one window serves several chunks.  Otherwise
    // (two CTAs per SM, or larger CTAs, where the kept windows would spill)
    // the window of the next row slot is fetched while the current one
    // computes.
    constexpr bool PERSIST = MB == 1 && W * 32 <= (VEC <= 4 ? 640 : 512);
    constexpr int RW = PERSIST ? R : 1;
    int wcol[RW];
    uint32_t wval[RW];
    int wb[RW];
    // VL: 128-entry windows (4 entries a lane), from the 16-byte-aligned floor
    // of the cursor.  (Each form's arrays are dead in the other and compiled away.)
    int wcv[RW][4];
    uint32_t wvv[RW][4];
    int wbv[RW];
    auto window_v = [&](int, int pos, int end, int (&col)[4], uint32_t (&val)[4]) {
        load_window_v<BF, SMX>(a, pos, end, lane, col, val);
    };
    if constexpr (VL) {
#pragma unroll
        for (int i = 0; i < RW; ++i) {
            wbv[i] = __shfl_sync(kFullMask, cur, i) & ~3;
            window_v(i, wbv[i], __shfl_sync(kFullMask, my_end, i), wcv[i], wvv[i]);
        }
    } else {
#pragma unroll
        for (int i = 0; i < RW; ++i) {
            wb[i] = __shfl_sync(kFullMask, cur, i);
            window(i, wb[i], __shfl_sync(kFullMask, my_end, i), wcol[i], wval[i]);
        }
    }

    unsigned char* wl = lists + warp * C_::LIST_SLOTS * ENTRY;
    const uint32_t wl_addr = smem_addr(wl);
    uint32_t tlane = 0;  // TM: this warp's TMEM lanes, column 0
    if constexpr (TM) {
        tmem_fence_after_sync();
        tlane = (uint32_t)kr[3] + ((uint32_t)(32 * (warp & 3)) << 16);
    }

    for (int j = 0; j < nchunks; ++j) {
        const int s = j % NS;
        const int k0 = (c_lo + j) * KC;
        // Warp-uniform: the row loop below is full of warp-wide operations.
        bool ok = __all_sync(kFullMask, mbar_wait_bounded(smem_addr(&bars[s]), (j / NS) & 1, kWaitLimitNs));
        if (!ok) kr[2] = 1;
        const uint32_t stage0 = smem_addr(stages + s * STAGE);
        const uint32_t lane_off = l * (NCH ? 16 : 8);
        const uint32_t stage = stage0 + lane_off;
        bool tm_ready = false, tm_failed = false;  // TM: this chunk's tensor-memory rows have landed
        if constexpr (TM) {
            // The chunk is in shared memory: warp w copies rows w, w + W, ... of
            // the tensor-memory part (two 512-byte halves a row) and commits.
            if (ok && lane == 0) {
#pragma unroll
                for (int q = 0; q < (TR + W - 1) / W; ++q) {
                    const int rr = warp + q * W;
                    if (rr >= TR) break;
                    tmem_cp_512b_x4((uint32_t)kr[3] + TCPR * rr, stage0 + (KL + rr) * PITCH);
                    if (!BF) tmem_cp_512b_x4((uint32_t)kr[3] + TCPR * rr + 4, stage0 + (KL + rr) * PITCH + 512);
                }
                tmem_commit(smem_addr(&bars[4]));
            }
        }
        if (ok) {
#pragma unroll
            for (int i = 0; i < R; ++i) {
                // SMX: this row's softmax statistics, for the list entries.
                const float row_m = SMX ? __shfl_sync(kFullMask, my_m, i) : 0.f;
                const float row_rz = SMX ? __shfl_sync(kFullMask, my_rz, i) : 0.f;
                if constexpr (VL) {
                    // The row's entries in this chunk, 128-entry windows at a time.
                    int rc = __shfl_sync(kFullMask, cur, i);
                    const int re = __shfl_sync(kFullMask, my_end, i);
                    int vc[4];
                    uint32_t vv[4];
                    int base = wbv[PERSIST ? i : 0];
#pragma unroll
                    for (int u = 0; u < 4; ++u) {
                        vc[u] = wcv[PERSIST ? i : 0][u];
                        vv[u] = wvv[PERSIST ? i : 0][u];
                    }
                    if constexpr (!PERSIST) {
                        if (i + 1 < R) {  // the next row slot's window, fetched while this one computes
                            wbv[0] = __shfl_sync(kFullMask, cur, i + 1) & ~3;
                            window_v(i + 1, wbv[0], __shfl_sync(kFullMask, my_end, i + 1), wcv[0], wvv[0]);
                        }
                    }
                    float c4[BF ? 1 : VEC], cc[BF ? 1 : VEC];
#pragma unroll
                    for (int v = 0; v < (BF ? 1 : VEC); ++v) c4[v] = cc[v] = 0.f;
                    while (true) {
                        // Entry e = 4·lane + u of the window is valid from the
                        // cursor (e >= wo: the aligned floor's residue is masked)
                        // to the row end, inside the chunk: a contiguous run.
                        const int wo = rc - base;  // 0 <= wo < 128
                        unsigned bal[4];
                        int n = 0;
#pragma unroll
                        for (int u = 0; u < 4; ++u) {
                            const int e = 4 * lane + u;
                            bal[u] = __ballot_sync(kFullMask, e >= wo && base + e < re &&
                                                                  (unsigned)(vc[u] - k0) < (unsigned)KC);
                            n += __popc(bal[u]);
                        }
                        if (n == 0) break;
                        const bool more = wo + n == 128;  // the run reaches the window's end
                        int nc[4];
                        uint32_t nv[4];
                        if (more) window_v(i, base + 128, re, nc, nv);
#pragma unroll
                        for (int u = 0; u < 4; ++u) {
                            if ((bal[u] >> lane) & 1u) {
                                const int slot = 4 * lane + u - wo;
                                const uint32_t off = (uint32_t)(vc[u] - k0) * PITCH;
                                const uint32_t vb = value_bits<BF, SMX>(vv[u], row_m, row_rz);
                                if constexpr (ADDR) {
                                    reinterpret_cast<uint32_t*>(wl)[slot] = stage0 + off;
                                    reinterpret_cast<uint16_t*>(wl + 4 * C_::LIST_SLOTS)[slot] = (uint16_t)vb;
                                } else if constexpr (BF) {
                                    reinterpret_cast<uint32_t*>(wl)[slot] = (off >> 3) | (vb << 16);
                                } else {
                                    reinterpret_cast<uint2*>(wl)[slot] = make_uint2(off, vb);
                                }
                            }
                        }
                        __syncwarp();
                        auto load_b = [&](uint32_t p, uint32_t (&w)[NW]) {
                            if constexpr (NCH == 0) {
                                const uint2 b = lds64(p);
                                w[0] = b.x;
                                w[1] = b.y;
                            } else {
#pragma unroll
                                for (int c = 0; c < NCH; ++c) {
                                    const uint4 b = lds128(p + C_::piece_off(c));
                                    w[4 * c] = b.x;
                                    w[4 * c + 1] = b.y;
                                    w[4 * c + 2] = b.z;
                                    w[4 * c + 3] = b.w;
                                }
                            }
                        };
                        auto step_bf16 = [&](uint32_t ad, uint16_t av) {
                            uint32_t w[NW];
                            load_b(ad + lane_off, w);
#pragma unroll
                            for (int q = 0; q < NW; ++q) {
                                acc[i][2 * q] = fma_bf16(av, lo16(w[q]), acc[i][2 * q]);
                                acc[i][2 * q + 1] = fma_bf16(av, hi16(w[q]), acc[i][2 * q + 1]);
                            }
                        };
                        auto step_f32 = [&](uint32_t off, uint32_t av) {
                            uint32_t w[NW];
                            load_b(stage + off, w);
                            const float x = __uint_as_float(av);
                            const float2 a2 = make_float2(x, x);
#pragma unroll
                            for (int q = 0; q < NW; q += 2) {
                                float2 c2 = make_float2(c4[q], c4[q + 1]);
                                c2 = __ffma2_rn(a2, make_float2(__uint_as_float(w[q]), __uint_as_float(w[q + 1])), c2);
                                c4[q] = c2.x;
                                c4[q + 1] = c2.y;
                            }
                        };
                        // Runs of at most 32 entries, each into a fresh fp32
                        // window partial (the same rounding path as 32-entry windows).
#pragma unroll 1
                        for (int s0 = 0; s0 < n; s0 += 32) {
                            const int s1 = min(n, s0 + 32), s4 = s0 + ((s1 - s0) & ~3);
#pragma unroll 1
                            for (int t = s0; t < s4; t += 4) {
                                if constexpr (ADDR) {
                                    const uint4 ad = lds128(wl_addr + t * 4);
                                    const uint2 av = lds64(wl_addr + 4 * C_::LIST_SLOTS + t * 2);
                                    step_bf16(ad.x, lo16(av.x));
                                    step_bf16(ad.y, hi16(av.x));
                                    step_bf16(ad.z, lo16(av.y));
                                    step_bf16(ad.w, hi16(av.y));
                                } else if constexpr (BF) {
                                    const uint4 e = lds128(wl_addr + t * 4);
                                    step_bf16(stage0 + ((e.x & 0xffffu) << 3), hi16(e.x));
                                    step_bf16(stage0 + ((e.y & 0xffffu) << 3), hi16(e.y));
                                    step_bf16(stage0 + ((e.z & 0xffffu) << 3), hi16(e.z));
                                    step_bf16(stage0 + ((e.w & 0xffffu) << 3), hi16(e.w));
                                } else {
                                    const uint4 e01 = lds128(wl_addr + t * 8);
                                    const uint4 e23 = lds128(wl_addr + t * 8 + 16);
                                    step_f32(e01.x, e01.y);
                                    step_f32(e01.z, e01.w);
                                    step_f32(e23.x, e23.y);
                                    step_f32(e23.z, e23.w);
                                }
                            }
#pragma unroll 1
                            for (int t = s4; t < s1; ++t) {
                                if constexpr (ADDR) {
                                    step_bf16(lds32(wl_addr + t * 4), lds16(wl_addr + 4 * C_::LIST_SLOTS + t * 2));
                                } else if constexpr (BF) {
                                    const uint32_t e = lds32(wl_addr + t * 4);
                                    step_bf16(stage0 + ((e & 0xffffu) << 3), hi16(e));
                                } else {
                                    const uint2 e = lds64(wl_addr + t * 8);
                                    step_f32(e.x, e.y);
                                }
                            }
                            if constexpr (!BF) {
#pragma unroll
                                for (int v = 0; v < VEC; ++v) {
                                    cc[v] += c4[v];
                                    c4[v] = 0.f;
                                }
                            }
                        }
                        __syncwarp();
                        rc += n;
                        if (!more) break;
#pragma unroll
                        for (int u = 0; u < 4; ++u) {
                            vc[u] = nc[u];
                            vv[u] = nv[u];
                        }
                        base += 128;
                    }
                    if constexpr (!BF) {
#pragma unroll
                        for (int v = 0; v < VEC; ++v) acc[i][v] += cc[v];
                    }
                    if constexpr (PERSIST) {
                        // Half the window used: refill it from the cursor's aligned floor.
                        if (rc - base >= 64 && rc < re) {
                            base = rc & ~3;
                            window_v(i, base, re, vc, vv);
                        }
#pragma unroll
                        for (int u = 0; u < 4; ++u) {
                            wcv[i][u] = vc[u];
                            wvv[i][u] = vv[u];
                        }
                        wbv[i] = base;
                    }
                    if (lane == i) cur = rc;
                    if constexpr (!PERSIST) {
                        if (i + 1 == R) {
                            wbv[0] = __shfl_sync(kFullMask, cur, 0) & ~3;
                            window_v(0, wbv[0], __shfl_sync(kFullMask, my_end, 0), wcv[0], wvv[0]);
                        }
                    }
                    continue;
                }
                int rc = __shfl_sync(kFullMask, cur, i);
                const int re = __shfl_sync(kFullMask, my_end, i);
                int col = wcol[PERSIST ? i : 0];
                uint32_t val = wval[PERSIST ? i : 0];
                int base = PERSIST ? wb[i] : rc;  // position of the window's lane 0 (rc - base < 32)
                if constexpr (!PERSIST) {
                    if (i + 1 < R) {
                        wb[0] = __shfl_sync(kFullMask, cur, i + 1);
                        window(i + 1, wb[0], __shfl_sync(kFullMask, my_end, i + 1), wcol[0], wval[0]);
                    }
                }
                float c4[BF ? 1 : VEC];  // fp32: this window's partial sums (≤ 32 terms)
                float cc[BF ? 1 : VEC];  // fp32: this chunk segment's windows
#pragma unroll
                for (int v = 0; v < (BF ? 1 : VEC); ++v) c4[v] = cc[v] = 0.f;
                while (true) {
                    // The chunk's entries of this row: a run of the window from
                    // lane rc - base (columns are sorted).
                    const int wo = PERSIST ? rc - base : 0;  // without PERSIST the window starts at rc
                    const bool valid = lane >= wo && (base + lane < re) && ((unsigned)(col - k0) < (unsigned)KC);
                    const unsigned run = __ballot_sync(kFullMask, valid) >> wo;
                    const int n = (run == kFullMask) ? 32 : (__ffs(~run) - 1);
                    if (n == 0) break;
                    // TM: the run's first n_sm entries lie in the shared-memory
                    // rows of the chunk, the rest in its tensor-memory rows.
                    int n_sm = n;
                    if constexpr (TM) {
                        const unsigned sm_run =
                            __ballot_sync(kFullMask, valid && (unsigned)(col - k0) < (unsigned)KL) >> wo;
                        n_sm = (sm_run == kFullMask) ? 32 : (__ffs(~sm_run) - 1);
                    }
                    // The window runs out inside this chunk: fetch the next one
                    // now so its latency overlaps this window's work.
                    const bool more = wo + n == 32;
                    int ncol = INT_MAX;
                    uint32_t nval = 0;
                    if (more) window(i, base + 32, re, ncol, nval);
                    // G == 1: exact count (0-3 single steps at the end).  G > 1: each
                    // group's block must start 16-byte aligned for the 128-bit
                    // entry loads, so pad to a multiple of 4·G.  Lane e writes
                    // list slot (e - wo) mod 32: every slot below npad is written.
                    const int npad = (G == 1) ? n : (n + 4 * G - 1) / (4 * G) * (4 * G);
                    const int slot = (lane - wo) & 31;
                    const uint32_t vb = value_bits<BF, SMX>(val, row_m, row_rz);
                    if (TM && slot >= n_sm && slot < n) {
                        // Tensor-memory rows: (TMEM address, value) in the second
                        // region, from its first slot, so it reads 16 bytes at a time.
                        if constexpr (BF)  // column | bf16 value << 16 (the warp's lanes added at use)
                            reinterpret_cast<uint32_t*>(wl)[32 + slot - n_sm] = (uint32_t)(col - k0 - KL) * TCPR | (vb << 16);
                        else
                            reinterpret_cast<uint2*>(wl)[32 + slot - n_sm] =
                                make_uint2(tlane + (uint32_t)(col - k0 - KL) * TCPR, vb);
                    } else if (slot < npad) {
                        const bool live = slot < n;
                        const uint32_t off = live ? (uint32_t)(col - k0) * PITCH : 0u;
                        if constexpr (ADDR) {
                            reinterpret_cast<uint32_t*>(wl)[slot] = stage0 + off;
                            reinterpret_cast<uint16_t*>(wl + 128)[slot] = live ? (uint16_t)vb : (uint16_t)0;
                        } else if constexpr (BF) {
                            reinterpret_cast<uint32_t*>(wl)[slot] = live ? ((off >> 3) | (vb << 16)) : 0u;
                        } else {
                            reinterpret_cast<uint2*>(wl)[slot] = live ? make_uint2(off, vb) : make_uint2(0u, 0u);
                        }
                    }
                    __syncwarp();
                    const int q = (TM ? n_sm : npad) / G;  // steps of each group (TM: shared-memory part)
                    const int q4 = q & ~3;
                    const uint32_t gl = wl_addr + g * q * (ADDR ? 4 : ENTRY);  // ADDR: addresses
                    const uint32_t gv = wl_addr + 128 + g * q * 2;             // ADDR: values
                    // The lane's words of the staged B row whose lane slice starts at p.
                    auto load_b = [&](uint32_t p, uint32_t (&w)[NW]) {
                        if constexpr (NCH == 0) {
                            const uint2 b = lds64(p);
                            w[0] = b.x;
                            w[1] = b.y;
                        } else {
#pragma unroll
                            for (int c = 0; c < NCH; ++c) {
                                const uint4 b = lds128(p + C_::piece_off(c));
                                w[4 * c] = b.x;
                                w[4 * c + 1] = b.y;
                                w[4 * c + 2] = b.z;
                                w[4 * c + 3] = b.w;
                            }
                        }
                    };
                    // One bf16 step: staged row at shared address ad, value av.
                    auto step_bf16 = [&](uint32_t ad, uint16_t av) {
                        uint32_t w[NW];
                        load_b(ad + lane_off, w);
#pragma unroll
                        for (int q = 0; q < NW; ++q) {
                            acc[i][2 * q] = fma_bf16(av, lo16(w[q]), acc[i][2 * q]);
                            acc[i][2 * q + 1] = fma_bf16(av, hi16(w[q]), acc[i][2 * q + 1]);
                        }
                    };
                    // fp32 FMAs of one step: the lane's words w of the B row, value bits av.
                    auto fma_f32 = [&](const uint32_t (&w)[NW], uint32_t av) {
                        const float x = __uint_as_float(av);
                        const float2 a2 = make_float2(x, x);
#pragma unroll
                        for (int q = 0; q < NW; q += 2) {
                            float2 c2 = make_float2(c4[q], c4[q + 1]);
                            c2 = __ffma2_rn(a2, make_float2(__uint_as_float(w[q]), __uint_as_float(w[q + 1])), c2);
                            c4[q] = c2.x;
                            c4[q + 1] = c2.y;
                        }
                    };
                    // One fp32 step: staged row at byte offset off, value bits av.
                    auto step_f32 = [&](uint32_t off, uint32_t av) {
                        uint32_t w[NW];
                        load_b(stage + off, w);
                        fma_f32(w, av);
                    };
#pragma unroll 1
#pragma unroll 1
                    for (int t = 0; t < q4; t += 4) {
                        if constexpr (ADDR) {
                            const uint4 ad = lds128(gl + t * 4);
                            const uint2 av = lds64(gv + t * 2);
                            step_bf16(ad.x, lo16(av.x));
                            step_bf16(ad.y, hi16(av.x));
                            step_bf16(ad.z, lo16(av.y));
                            step_bf16(ad.w, hi16(av.y));
                        } else if constexpr (BF) {
                            const uint4 e = lds128(gl + t * 4);
                            step_bf16(stage0 + ((e.x & 0xffffu) << 3), hi16(e.x));
                            step_bf16(stage0 + ((e.y & 0xffffu) << 3), hi16(e.y));
                            step_bf16(stage0 + ((e.z & 0xffffu) << 3), hi16(e.z));
                            step_bf16(stage0 + ((e.w & 0xffffu) << 3), hi16(e.w));
                        } else {
                            const uint4 e01 = lds128(gl + t * 8);
                            const uint4 e23 = lds128(gl + t * 8 + 16);
                            step_f32(e01.x, e01.y);
                            step_f32(e01.z, e01.w);
                            step_f32(e23.x, e23.y);
                            step_f32(e23.z, e23.w);
                        }
                    }
#pragma unroll 1
                    for (int t = q4; t < q; ++t) {  // 0-3 remaining steps (G == 1 only)
                        if constexpr (ADDR) {
                            step_bf16(lds32(gl + t * 4), lds16(gv + t * 2));
                        } else if constexpr (BF) {
                            const uint32_t e = lds32(gl + t * 4);
                            step_bf16(stage0 + ((e & 0xffffu) << 3), hi16(e));
                        } else {
                            const uint2 e = lds64(gl + t * 8);
                            step_f32(e.x, e.y);
                        }
                    }
                    if constexpr (TM) {
                        // Entries n_sm..n-1: B rows from tensor memory, once this
                        // chunk's copies have landed (checked once per chunk).
                        if (n_sm < n && !tm_ready && !tm_failed) {
                            tm_ready = __all_sync(kFullMask, mbar_wait_bounded(smem_addr(&bars[4]), j & 1, kWaitLimitNs));
                            tm_failed = !tm_ready;
                            if (tm_failed) kr[2] = 1;
                            tmem_fence_after_sync();
                        }
                        if constexpr (!BF && USM_TM_PIPE != 0) {
                        if (tm_ready) {
                            // Pairs of entries, software-pipelined: the next pair's
                            // loads are in flight while the current pair's FMAs run
                            // (the wait covers every outstanding load, so the loads
                            // of one pair and the FMAs of the previous alternate).
                            int t = 0, cnt = n - n_sm;
                            auto ent = [&](int k) { return lds64(wl_addr + (32 + k) * 8); };
                            if (cnt >= 2) {
                                uint32_t wa0[NW], wa1[NW], wb0[NW], wb1[NW];
                                uint2 ea0 = ent(t), ea1 = ent(t + 1);
                                tmem_ld8x2_nowait(ea0.x, ea1.x, wa0, wa1, c4);
                                tmem_wait_tied(wa0, wa1, c4);
                                t += 2;
                                cnt -= 2;
#pragma unroll 1
                                for (; cnt >= 4; cnt -= 4, t += 4) {
                                    const uint2 eb0 = ent(t), eb1 = ent(t + 1);
                                    tmem_ld8x2_nowait(eb0.x, eb1.x, wb0, wb1, c4);
                                    fma_f32(wa0, ea0.y);
                                    fma_f32(wa1, ea1.y);
                                    tmem_wait_tied(wb0, wb1, c4);
                                    ea0 = ent(t + 2);
                                    ea1 = ent(t + 3);
                                    tmem_ld8x2_nowait(ea0.x, ea1.x, wa0, wa1, c4);
                                    fma_f32(wb0, eb0.y);
                                    fma_f32(wb1, eb1.y);
                                    tmem_wait_tied(wa0, wa1, c4);
                                }
                                if (cnt >= 2) {
                                    const uint2 eb0 = ent(t), eb1 = ent(t + 1);
                                    tmem_ld8x2_nowait(eb0.x, eb1.x, wb0, wb1, c4);
                                    fma_f32(wa0, ea0.y);
                                    fma_f32(wa1, ea1.y);
                                    tmem_wait_tied(wb0, wb1, c4);
                                    fma_f32(wb0, eb0.y);
                                    fma_f32(wb1, eb1.y);
                                    t += 2;
                                    cnt -= 2;
                                } else {
                                    fma_f32(wa0, ea0.y);
                                    fma_f32(wa1, ea1.y);
                                }
                            }
                            if (cnt == 1) {
                                const uint2 e = ent(t);
                                uint32_t w[NW];
                                tmem_ld8(e.x, w);
                                fma_f32(w, e.y);
                            }
                        }
                        }
                        if constexpr (BF) {
                          if (tm_ready) {
                            // bf16: four entries (column | value << 16) a 128-bit load.
                            const uint32_t tl = wl_addr + 32 * ENTRY;
                            const int m = n - n_sm;
                            auto fma_w = [&](uint4 w, uint32_t e) {
                                const uint16_t av = hi16(e);
                                const uint32_t ww[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
                                for (int q = 0; q < 4; ++q) {
                                    acc[i][2 * q] = fma_bf16(av, lo16(ww[q]), acc[i][2 * q]);
                                    acc[i][2 * q + 1] = fma_bf16(av, hi16(ww[q]), acc[i][2 * q + 1]);
                                }
                            };
                            int t = 0;
#pragma unroll 1
                            for (; t + 4 <= m; t += 4) {
                                const uint4 e = lds128(tl + t * 4);
                                uint4 w0, w1, w2, w3;
                                tmem_ld4x4(tlane + (e.x & 0xffffu), tlane + (e.y & 0xffffu), tlane + (e.z & 0xffffu),
                                           tlane + (e.w & 0xffffu), w0, w1, w2, w3);
                                fma_w(w0, e.x);
                                fma_w(w1, e.y);
                                fma_w(w2, e.z);
                                fma_w(w3, e.w);
                            }
#pragma unroll 1
                            for (; t < m; ++t) {
                                const uint32_t e = lds32(tl + t * 4);
                                fma_w(tmem_ld4(tlane + (e & 0xffffu)), e);
                            }
                          }
                        } else {
                        if (tm_ready && !USM_TM_PIPE) {
                            const uint32_t tl = wl_addr + 32 * 8;  // tensor-memory entries
                            const int m = n - n_sm;
                            int t = 0;
#pragma unroll 1
                            for (; t + 4 <= m; t += 4) {
                                const uint4 e01 = lds128(tl + t * 8), e23 = lds128(tl + t * 8 + 16);
                                uint32_t w0[NW], w1[NW], w2[NW], w3[NW];
                                tmem_ld8x4(e01.x, e01.z, e23.x, e23.z, w0, w1, w2, w3);
                                fma_f32(w0, e01.y);
                                fma_f32(w1, e01.w);
                                fma_f32(w2, e23.y);
                                fma_f32(w3, e23.w);
                            }
#pragma unroll 1
                            for (; t < m; ++t) {
                                const uint2 e = lds64(tl + t * 8);
                                uint32_t w[NW];
                                tmem_ld8(e.x, w);
                                fma_f32(w, e.y);
                            }
                        }
                        }
                    }
                    __syncwarp();
                    if constexpr (!BF) {
#pragma unroll
                        for (int v = 0; v < VEC; ++v) {
                            cc[v] += c4[v];
                            c4[v] = 0.f;
                        }
                    }
                    rc += n;
                    if (!more) break;
                    col = ncol;
                    val = nval;
                    base += 32;
                }
                if constexpr (!BF) {
#pragma unroll
                    for (int v = 0; v < VEC; ++v) acc[i][v] += cc[v];
                }
                if constexpr (PERSIST) {
                    // Half the window used: refill it from the cursor now; the
                    // load lands while the other rows and the next chunk's wait
                    // go by.
                    if (rc - base >= 16 && rc < re) {
                        base = rc;
                        window(i, rc, re, col, val);
                    }
                    wcol[i] = col;
                    wval[i] = val;
                    wb[i] = base;
                }
                if (lane == i) cur = rc;
                if constexpr (!PERSIST) {
                    if (i + 1 == R)
                        window(0, __shfl_sync(kFullMask, cur, 0), __shfl_sync(kFullMask, my_end, 0), wcol[0],
                               wval[0]);
                }
            }
        }
        if constexpr (LONGK) {
            if ((j & 63) == 63) {
#pragma unroll
                for (int i = 0; i < R; ++i)
#pragma unroll
                    for (int v = 0; v < VEC; ++v) {
                        acc_hi[i][v] += acc[i][v];
                        acc[i][v] = 0.f;
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
        __syncthreads();  // every warp is done with stage s
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
        if (warp == 0) tmem_dealloc((uint32_t)kr[3], TCOLS);
    }

    if (kr[2]) {
        // A transfer never completed: record it, wait (bounded) for the copies
        // still in flight so none lands after the CTA exits, and leave.
        if (threadIdx.x == 0) {
            record_status(a.status, USM_ERR_TIMEOUT);
            for (int b = 0; b < nchunks && b < NS; ++b) {
                // Waiting on both parities waits for the barrier's current phase
                // (the other parity reports complete at once); each wait is bounded.
                mbar_wait_bounded(smem_addr(&bars[b]), 0, 1000000ull);
                mbar_wait_bounded(smem_addr(&bars[b]), 1, 1000000ull);
            }
        }
        return;
    }

    // Add the G partial rows held by the lane groups.
#pragma unroll
    for (int i = 0; i < R; ++i)
#pragma unroll
        for (int v = 0; v < VEC; ++v) {
            float x = LONGK ? acc_hi[i][v] + acc[i][v] : acc[i][v];
            if (G >= 2) x += __shfl_xor_sync(kFullMask, x, L);
            if (G >= 4) x += __shfl_xor_sync(kFullMask, x, 2 * L);
            if (G >= 8) x += __shfl_xor_sync(kFullMask, x, 4 * L);
            acc[i][v] = x;
        }

#pragma unroll
    for (int i = 0; i < R; ++i) {
        const int row = __shfl_sync(kFullMask, my_row, i);
        if (row < 0 || g != 0) continue;
        float* crow = a.C + (long long)row * a.ldc + n0;
#pragma unroll
        for (int v = 0; v < VEC; v += 4) {  // 4 contiguous columns at a time
            const int c = lane_col<L, VEC, C_::ES>(l, v);
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

// Direct-gather SpMM, for masks so sparse that staging every row of B in
// each CTA costs more than the nonzeros use (LSTM-like shapes at 98%): no
// shared memory.  SMX: the values are the rows' softmax probabilities of
// fp32 scores, formed as in the staged kernel.  Each warp takes rows of the swizzled order (grid-stride),
// and for every nonzero reads the lane's 16 bytes of the B row (4 fp32 or 8
// bf16 of a 32·VEC-column pass) straight from global memory, eight
// nonzeros' loads in flight.  fp32 sums: ≤ 32 terms (one window) into a
// fresh partial, partials into the row total.  Column indices outside
// [0, K) read row 0 (undefined result, in-bounds access).
#ifndef USM_GATHER_MINB
#define USM_GATHER_MINB 4
#endif
template <bool BF, bool SMX = false>
__global__ void __launch_bounds__(256, USM_GATHER_MINB) spmm_gather_kernel(const SpmmArgs a, const void* __restrict__ Bv, long long ldb) {
    constexpr int VEC = BF ? 8 : 4;
    constexpr int ES = BF ? 2 : 4;
    const int lane = threadIdx.x & 31;
    const long long warps = (long long)gridDim.x * (blockDim.x >> 5);
    const unsigned char* B = static_cast<const unsigned char*>(Bv);
    for (long long m = (blockIdx.x * (long long)blockDim.x + threadIdx.x) >> 5; m < a.M; m += warps) {
        const int r = a.perm ? __ldg(a.perm + m) : (int)m;
        if ((unsigned)r >= (unsigned)a.M) continue;  // warp-uniform
        int s = __ldg(a.row_offsets + r), e = __ldg(a.row_offsets + r + 1);
        s = min(max(s, 0), a.nnz);
        e = min(max(e, s), a.nnz);
        float row_m = 0.f, row_rz = 0.f;  // SMX: the row's softmax statistics
        if constexpr (SMX) row_softmax_stats(reinterpret_cast<const float*>(a.values), s, e, lane, row_m, row_rz);
        for (int n0 = 0; n0 < a.N; n0 += 32 * VEC) {
            const int c0 = n0 + lane * VEC;          // the lane's first column
            const bool full = c0 + VEC <= a.N;       // a whole 16-byte piece
            const bool any = c0 < a.N;
            float acc[VEC];
#pragma unroll
            for (int v = 0; v < VEC; ++v) acc[v] = 0.f;
            // The lane's 16 bytes of B row k (zeros past N).
            auto load_b = [&](int k) {
                uint4 w = make_uint4(0u, 0u, 0u, 0u);
                const unsigned char* row = B + ((long long)k * ldb + c0) * ES;
                if (full) {
                    w = __ldg(reinterpret_cast<const uint4*>(row));
                } else if (any) {
                    uint32_t h[VEC];
#pragma unroll
                    for (int v = 0; v < VEC; ++v)
                        h[v] = c0 + v < a.N ? (BF ? (uint32_t)__ldg(reinterpret_cast<const unsigned short*>(row) + v)
                                                  : __ldg(reinterpret_cast<const unsigned int*>(row) + v))
                                            : 0u;
                    if constexpr (BF)
                        w = make_uint4(h[0] | (h[1] << 16), h[2] | (h[3] << 16), h[4] | (h[5] << 16), h[6] | (h[7] << 16));
                    else
                        w = make_uint4(h[0], h[1], h[2], h[3]);
                }
                return w;
            };
            auto fma_b = [&](float (&c)[VEC], uint32_t av, uint4 w) {
                const uint32_t ww[4] = {w.x, w.y, w.z, w.w};
                if constexpr (BF) {
#pragma unroll
                    for (int q = 0; q < 4; ++q) {
                        c[2 * q] = fma_bf16((uint16_t)av, lo16(ww[q]), c[2 * q]);
                        c[2 * q + 1] = fma_bf16((uint16_t)av, hi16(ww[q]), c[2 * q + 1]);
                    }
                } else {
                    const float x = __uint_as_float(av);
                    const float2 a2 = make_float2(x, x);
#pragma unroll
                    for (int q = 0; q < 4; q += 2) {
                        float2 c2 = make_float2(c[q], c[q + 1]);
                        c2 = __ffma2_rn(a2, make_float2(__uint_as_float(ww[q]), __uint_as_float(ww[q + 1])), c2);
                        c[q] = c2.x;
                        c[q + 1] = c2.y;
                    }
                }
            };
            for (int base = s; base < e; base += 32) {
                int col;
                uint32_t val;
                load_window<BF, SMX>(a, base, e, lane, col, val);
                col = (unsigned)col < (unsigned)a.K ? col : 0;
                val = value_bits<BF, SMX>(val, row_m, row_rz);
                const int n = min(32, e - base);
                float part[VEC];
#pragma unroll
                for (int v = 0; v < VEC; ++v) part[v] = BF ? acc[v] : 0.f;  // bf16: one running sum
                int t = 0;
#pragma unroll 1
                for (; t + 8 <= n; t += 8) {
                    uint4 w[8];
                    uint32_t av[8];
#pragma unroll
                    for (int u = 0; u < 8; ++u) {
                        w[u] = load_b(__shfl_sync(kFullMask, col, t + u));
                        av[u] = __shfl_sync(kFullMask, val, t + u);
                    }
#pragma unroll
                    for (int u = 0; u < 8; ++u) fma_b(part, av[u], w[u]);
                }
#pragma unroll 1
                for (; t < n; ++t) {
                    const uint4 w = load_b(__shfl_sync(kFullMask, col, t));
                    fma_b(part, __shfl_sync(kFullMask, val, t), w);
                }
#pragma unroll
                for (int v = 0; v < VEC; ++v) acc[v] = BF ? part[v] : acc[v] + part[v];
            }
            if (any) {
                float* crow = a.C + (long long)r * a.ldc + c0;
                if (full) {
#pragma unroll
                    for (int v = 0; v < VEC; v += 4)
                        *reinterpret_cast<float4*>(crow + v) = make_float4(acc[v], acc[v + 1], acc[v + 2], acc[v + 3]);
                } else {
#pragma unroll
                    for (int v = 0; v < VEC; ++v)
                        if (c0 + v < a.N) crow[v] = acc[v];
                }
            }
        }
    }
}

__global__ void fill_f32_kernel(float* C, int M, int N, long long ldc) {
    const long long total = (long long)M * N;
    for (long long i = blockIdx.x * (long long)blockDim.x + threadIdx.x; i < total;
         i += (long long)gridDim.x * blockDim.x) {
        const long long r = i / N, c = i % N;
        C[r * ldc + c] = 0.f;
    }
}

}  // namespace
}  // namespace usm
