// CSR SpMM, C = A·B, for sm_103a.
//
// "Sparse GPU Kernels for Deep Learning" (Gale et al., SC 2020), summary
// card "Summary": SpMM on plain CSR with 1-D tiling, vector memory access on
// misaligned sparse rows and a load-balancing order kept apart from how the
// work is split ("Interesting ideas" I4).  The design below is written for
// GB300, not taken from the V100 kernels:
//
// * 1-D tiles.  A CTA owns MT = R·W rows of A (taken in row-swizzle order,
//   interleaved across its W warps so every warp gets a similar share) and
//   one strip of NT output columns.  Each output element is accumulated by
//   exactly one lane group in a fixed order: results do not depend on the
//   swizzle.  Two CTAs share an SM, so one CTA's barrier waits and prologue
//   overlap the other's arithmetic.
// * Dense operand staging.  The CTA walks K in chunks of KC rows.  For each
//   chunk one thread issues TMA tensor copies of B[k0:k0+KC, n0:n0+NT] into a
//   shared-memory stage (completion on an mbarrier, bounded wait; one or two
//   stages).  Only the chunks between the smallest and largest column index of
//   the CTA's rows are fetched, so block-diagonal (batched) matrices stay
//   cheap.
// * Sparse operand.  For each (row, chunk) a warp reads the next 32 column
//   indices and values of the row with coalesced loads (the window after the
//   row's cursor, so a misaligned row start costs nothing), keeps the prefix
//   whose columns fall in the chunk (ballot) and writes (stage offset, value)
//   entries to a per-warp list.  The next row's window is prefetched while
//   the current one computes.
// * Inner loop.  G = 32/L lane groups split the list into contiguous blocks.
//   Four steps at a time a group reads its four entries with 128-bit
//   broadcast loads (then 0-3 single steps), each lane reads 16 (fp32) or 8
//   (bf16) bytes of the staged B row (a group covers whole rows,
//   conflict-free) and does 4 FMAs: packed f32x2 FMA for fp32,
//   fma.rn.f32.bf16 on the bf16 halves for bf16.  The G partial rows are
//   added across groups at the end.
// * Accuracy.  In fp32 each window of ≤ 32 nonzeros is summed into a fresh
//   accumulator, windows are added into a per-(row, chunk) partial and those
//   into the row total: with ≤ 32 + 7 + K/KC additions along any output's
//   path the worst-case rounding bound stays below 1e-5·Σ|a||b| while
//   K/KC ≤ 128 (K up to 12288 with KC = 96).
#include <climits>
#include <type_traits>

#include "usm_device.cuh"
#include "usm_internal.h"

namespace usm {
namespace {

template <bool BF, int L, int R, int W, int KC, int NS>
struct SpmmCfg {
    static constexpr int ES = BF ? 2 : 4;          // element bytes
    static constexpr int NT = L * 4;               // output columns per CTA (4 per lane)
    static constexpr int G = 32 / L;               // lane groups (nonzeros per warp step)
    static constexpr int LANE_BYTES = 4 * ES;      // B bytes per lane per step
    static constexpr int PITCH = L * LANE_BYTES;   // bytes per staged B row
    static constexpr int STAGE = KC * PITCH;
    static constexpr int MT = R * W;
    static constexpr int BOX_ROWS = KC <= 256 ? KC : (KC % 256 == 0 ? 256 : (KC % 192 == 0 ? 192 : 128));
    static constexpr int THREADS = W * 32;
    static constexpr int ENTRY = BF ? 4 : 8;       // list entry bytes
    static constexpr int LIST_BYTES = W * 32 * ENTRY;
    static constexpr int SMEM = NS * STAGE + 64 + LIST_BYTES;
    static_assert(NS == 1 || NS == 2, "one or two stages");
    static_assert(32 % L == 0, "L must divide the warp");
    static_assert(KC % BOX_ROWS == 0 && BOX_ROWS <= 256, "TMA box height");
    static_assert(!BF || STAGE / 8 < 65536, "bf16 entry offsets are 16-bit multiples of 8 bytes");
};

// Window of 32 consecutive nonzeros of a row starting at `pos`: lane i gets
// nonzero pos+i (column INT_MAX past the row end).
template <bool BF>
__device__ __forceinline__ void load_window(const SpmmArgs& a, int pos, int end, int lane, int& col,
                                            uint32_t& val) {
    const int p = pos + lane;
    if (p < end) {
        col = __ldg(a.col_indices + p);
        if (BF)
            val = __ldg(reinterpret_cast<const unsigned short*>(a.values) + p);
        else
            val = __ldg(reinterpret_cast<const unsigned int*>(a.values) + p);
    } else {
        col = INT_MAX;
        val = 0;
    }
}

template <bool BF, int L, int R, int W, int KC, int NS>
__global__ void __launch_bounds__(W * 32, 2)
    spmm_kernel(const __grid_constant__ CUtensorMap tmB, const SpmmArgs a) {
    using C_ = SpmmCfg<BF, L, R, W, KC, NS>;
    constexpr int G = C_::G, PITCH = C_::PITCH, STAGE = C_::STAGE, ENTRY = C_::ENTRY;

    extern __shared__ __align__(1024) unsigned char smem[];
    unsigned char* stages = smem;
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + NS * STAGE);
    int* kr = reinterpret_cast<int*>(smem + NS * STAGE + 16);  // [0]=min col, [1]=max col, [2]=abort
    unsigned char* lists = smem + NS * STAGE + 64;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int g = lane / L, l = lane % L;
    const int n0 = blockIdx.y * C_::NT;
    const int tile = blockIdx.x;

    if (threadIdx.x == 0) {
        kr[0] = INT_MAX;
        kr[1] = -1;
        kr[2] = 0;
        mbar_init(smem_addr(&bars[0]), 1);
        mbar_init(smem_addr(&bars[1]), 1);
        fence_barrier_init();
        prefetch_tensor_map(&tmB);
    }

    // Row slots of this warp: slot i is row perm[tile*MT + i*W + warp].
    int my_row = -1, my_start = 0, my_end = 0;
    if (lane < R) {
        const long long m = (long long)tile * C_::MT + (long long)lane * W + warp;
        if (m < a.M) {
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
    int c_lo = 0, nchunks = 0;
    {
        const int lo = max(kr[0], 0), hi = min(kr[1], a.K - 1);
        if (kr[1] >= 0 && lo <= hi) {
            c_lo = lo / KC;
            nchunks = hi / KC - c_lo + 1;
        }
    }

    auto issue = [&](int j) {
        const int s = j % NS;
        const uint32_t bar = smem_addr(&bars[s]);
        mbar_arrive_expect_tx(bar, STAGE);
        const uint32_t dst = smem_addr(stages + s * STAGE);
#pragma unroll
        for (int b = 0; b < KC / C_::BOX_ROWS; ++b)
            tma_load_2d(dst + b * C_::BOX_ROWS * PITCH, &tmB, n0, (c_lo + j) * KC + b * C_::BOX_ROWS,
                        bar);
    };
    if (threadIdx.x == 0) {
        if (nchunks > 0) issue(0);
        if (NS > 1 && nchunks > 1) issue(1);
    }

    float acc[R][4];
#pragma unroll
    for (int i = 0; i < R; ++i)
#pragma unroll
        for (int v = 0; v < 4; ++v) acc[i][v] = 0.f;

    int cur = my_start;  // lane i: cursor of row slot i
    int pcol;
    uint32_t pval;
    load_window<BF>(a, __shfl_sync(kFullMask, cur, 0), __shfl_sync(kFullMask, my_end, 0), lane, pcol,
                    pval);

    unsigned char* wl = lists + warp * 32 * ENTRY;
    const uint32_t wl_addr = smem_addr(wl);

    for (int j = 0; j < nchunks; ++j) {
        const int s = j % NS;
        const int k0 = (c_lo + j) * KC;
        const bool ok = mbar_wait_bounded(smem_addr(&bars[s]), (j / NS) & 1, kWaitLimitNs);
        if (!ok) kr[2] = 1;
        const uint32_t stage = smem_addr(stages + s * STAGE) + l * C_::LANE_BYTES;
        if (ok) {
#pragma unroll
            for (int i = 0; i < R; ++i) {
                int rc = __shfl_sync(kFullMask, cur, i);
                const int re = __shfl_sync(kFullMask, my_end, i);
                int col = pcol;
                uint32_t val = pval;
                if (i + 1 < R)
                    load_window<BF>(a, __shfl_sync(kFullMask, cur, i + 1),
                                    __shfl_sync(kFullMask, my_end, i + 1), lane, pcol, pval);
                float c4[4] = {0.f, 0.f, 0.f, 0.f};  // fp32: this window's partial sums (≤ 32 terms)
                float cc[4] = {0.f, 0.f, 0.f, 0.f};  // fp32: this chunk segment's windows
                while (true) {
                    const bool valid = (rc + lane < re) && ((unsigned)(col - k0) < (unsigned)KC);
                    const unsigned bal = __ballot_sync(kFullMask, valid);
                    const int n = (bal == kFullMask) ? 32 : (__ffs(~bal) - 1);  // valid prefix
                    if (n == 0) break;
                    // G == 1: exact count (0-3 single steps at the end).  G > 1: each
                    // group's block must start 16-byte aligned for the 128-bit
                    // entry loads, so pad to a multiple of 4·G.
                    const int npad = (G == 1) ? n : (n + 4 * G - 1) / (4 * G) * (4 * G);
                    if (lane < npad) {
                        const bool live = lane < n;
                        const uint32_t off = live ? (uint32_t)(col - k0) * PITCH : 0u;
                        if constexpr (BF) {
                            reinterpret_cast<uint32_t*>(wl)[lane] = live ? ((off >> 3) | (val << 16)) : 0u;
                        } else {
                            reinterpret_cast<uint2*>(wl)[lane] = live ? make_uint2(off, val) : make_uint2(0u, 0u);
                        }
                    }
                    __syncwarp();
                    const int q = npad / G;  // steps of each group
                    const int q4 = q & ~3;
                    const uint32_t gl = wl_addr + g * q * ENTRY;
                    // One bf16 step: entry e = (stage offset / 8) | value << 16.
                    auto step_bf16 = [&](uint32_t e) {
                        const uint2 b = lds64(stage + ((e & 0xffffu) << 3));
                        const uint16_t av = hi16(e);
                        acc[i][0] = fma_bf16(av, lo16(b.x), acc[i][0]);
                        acc[i][1] = fma_bf16(av, hi16(b.x), acc[i][1]);
                        acc[i][2] = fma_bf16(av, lo16(b.y), acc[i][2]);
                        acc[i][3] = fma_bf16(av, hi16(b.y), acc[i][3]);
                    };
                    // One fp32 step: staged row at byte offset off, value bits av.
                    auto step_f32 = [&](const uint4& b, uint32_t av) {
                        const float x = __uint_as_float(av);
                        const float2 a2 = make_float2(x, x);
                        float2 lo = make_float2(c4[0], c4[1]), hi = make_float2(c4[2], c4[3]);
                        lo = __ffma2_rn(a2, make_float2(__uint_as_float(b.x), __uint_as_float(b.y)), lo);
                        hi = __ffma2_rn(a2, make_float2(__uint_as_float(b.z), __uint_as_float(b.w)), hi);
                        c4[0] = lo.x;
                        c4[1] = lo.y;
                        c4[2] = hi.x;
                        c4[3] = hi.y;
                    };
#pragma unroll 1
                    for (int t = 0; t < q4; t += 4) {
                        if constexpr (BF) {
                            const uint4 e = lds128(gl + t * 4);
                            step_bf16(e.x);
                            step_bf16(e.y);
                            step_bf16(e.z);
                            step_bf16(e.w);
                        } else {
                            const uint4 e01 = lds128(gl + t * 8);
                            const uint4 e23 = lds128(gl + t * 8 + 16);
                            const uint4 b0 = lds128(stage + e01.x), b1 = lds128(stage + e01.z);
                            const uint4 b2 = lds128(stage + e23.x), b3 = lds128(stage + e23.z);
                            step_f32(b0, e01.y);
                            step_f32(b1, e01.w);
                            step_f32(b2, e23.y);
                            step_f32(b3, e23.w);
                        }
                    }
#pragma unroll 1
                    for (int t = q4; t < q; ++t) {  // 0-3 remaining steps (G == 1 only)
                        if constexpr (BF) {
                            step_bf16(lds32(gl + t * 4));
                        } else {
                            const uint2 e = lds64(gl + t * 8);
                            step_f32(lds128(stage + e.x), e.y);
                        }
                    }
                    __syncwarp();
                    if constexpr (!BF) {
#pragma unroll
                        for (int v = 0; v < 4; ++v) {
                            cc[v] += c4[v];
                            c4[v] = 0.f;
                        }
                    }
                    rc += n;
                    if (n < 32) break;
                    load_window<BF>(a, rc, re, lane, col, val);
                }
                if constexpr (!BF) {
#pragma unroll
                    for (int v = 0; v < 4; ++v) acc[i][v] += cc[v];
                }
                if (lane == i) cur = rc;
                if (i + 1 == R)
                    load_window<BF>(a, __shfl_sync(kFullMask, cur, 0), __shfl_sync(kFullMask, my_end, 0),
                                    lane, pcol, pval);
            }
        }
        __syncthreads();  // every warp is done with stage s
        if (kr[2]) break;
        if (threadIdx.x == 0 && j + NS < nchunks) {
            fence_proxy_async_smem();
            issue(j + NS);
        }
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
        for (int v = 0; v < 4; ++v) {
            float x = acc[i][v];
            if (G >= 2) x += __shfl_xor_sync(kFullMask, x, L);
            if (G >= 4) x += __shfl_xor_sync(kFullMask, x, 2 * L);
            if (G >= 8) x += __shfl_xor_sync(kFullMask, x, 4 * L);
            acc[i][v] = x;
        }

#pragma unroll
    for (int i = 0; i < R; ++i) {
        const int row = __shfl_sync(kFullMask, my_row, i);
        if (row < 0 || g != 0) continue;
        const int c0 = n0 + l * 4;
        float* dst = a.C + (long long)row * a.ldc + c0;
        if (c0 + 4 <= a.N) {
            *reinterpret_cast<float4*>(dst) = make_float4(acc[i][0], acc[i][1], acc[i][2], acc[i][3]);
        } else {
#pragma unroll
            for (int v = 0; v < 4; ++v)
                if (c0 + v < a.N) dst[v] = acc[i][v];
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

template <bool BF, int L, int R, int W, int KC, int NS>
int launch_cfg(const SpmmArgs& a, const void* B, int ldb, cudaStream_t stream) {
    using C_ = SpmmCfg<BF, L, R, W, KC, NS>;
    CUtensorMap map;
    if (!encode_tensor_map_2d(&map, B, BF, a.K, a.N, ldb, C_::NT, C_::BOX_ROWS)) return USM_ERR_CUDA;
    auto kern = spmm_kernel<BF, L, R, W, KC, NS>;
    static int configured_mask = 0;  // one bit per device
    int dev = 0;
    cudaGetDevice(&dev);
    if (dev < 31 && !(__atomic_load_n(&configured_mask, __ATOMIC_ACQUIRE) & (1 << dev))) {
        if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C_::SMEM) !=
            cudaSuccess)
            return USM_ERR_CUDA;
        __atomic_fetch_or(&configured_mask, 1 << dev, __ATOMIC_ACQ_REL);
    }
    // Row tiles on x (dispatched first, longest rows first under a swizzle),
    // column strips on y.
    const dim3 grid((a.M + C_::MT - 1) / C_::MT, (a.N + C_::NT - 1) / C_::NT);
    if (grid.y > 65535u) return USM_ERR_UNSUPPORTED;
    kern<<<grid, C_::THREADS, C_::SMEM, stream>>>(map, a);
    return cudaGetLastError() == cudaSuccess ? USM_OK : USM_ERR_CUDA;
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

// Tile choice: 128 output columns per CTA (4 per lane), or 64 when N ≤ 64;
// 4 rows per warp and 16 warps (64 rows per CTA), two CTAs per SM and one
// 96 KB stage per CTA: while one CTA waits for its next chunk the other
// computes, and the tall chunks (KC = 192 fp32 / 384 bf16 rows) halve the
// per-(row, chunk) work that a double-buffered 2 x 48 KB layout needs
// (measured: FFN step 7.69 against 8.90 ms).
#ifndef USM_SPMM_STAGES
#define USM_SPMM_STAGES 1
#endif
int launch_spmm(const SpmmArgs& a, const void* B, int ldb, bool bf16, cudaStream_t stream) {
    constexpr int W = 16, R = 4, NS = USM_SPMM_STAGES, F = 2 / NS;  // F: chunk growth with one stage
    if (!bf16) {
        if (a.N <= 64) return launch_cfg<false, 16, R, W, 192 * F, NS>(a, B, ldb, stream);
        return launch_cfg<false, 32, R, W, 96 * F, NS>(a, B, ldb, stream);
    }
    if (a.N <= 64) return launch_cfg<true, 16, R, W, 384 * F, NS>(a, B, ldb, stream);
    return launch_cfg<true, 32, R, W, 192 * F, NS>(a, B, ldb, stream);
}

}  // namespace usm
