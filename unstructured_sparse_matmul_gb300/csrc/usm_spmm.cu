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
//   shared-memory stage (double buffered, completion on an mbarrier, bounded
//   wait).  Only the chunks between the smallest and largest column index of
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
//   broadcast loads, then each lane reads 16 (fp32) or 8 (bf16) bytes of the
//   four staged B rows (a group covers whole rows, conflict-free) and does 4
//   FMAs per row: packed f32x2 FMA for fp32, fma.rn.f32.bf16 straight on the
//   bf16 halves for bf16.  The G partial rows are added across groups at the
//   end.
// * Accuracy.  In fp32 each (row, chunk) segment (≤ KC terms) is summed into
//   a fresh accumulator that is then added to the row total: every output is
//   a sum of ≤ KC-term partials, which keeps the worst-case rounding bound
//   below 1e-5·Σ|a||b| for K up to 4096 (KC = 96).
#include <climits>
#include <type_traits>

#include "usm_device.cuh"
#include "usm_internal.h"

namespace usm {
namespace {

template <bool BF, int L, int R, int W, int KC>
struct SpmmCfg {
    static constexpr int ES = BF ? 2 : 4;          // element bytes
    static constexpr int NT = L * 4;               // output columns per CTA (4 per lane)
    static constexpr int G = 32 / L;               // lane groups (nonzeros per warp step)
    static constexpr int LANE_BYTES = 4 * ES;      // B bytes per lane per step
    static constexpr int PITCH = L * LANE_BYTES;   // bytes per staged B row
    static constexpr int STAGE = KC * PITCH;
    static constexpr int MT = R * W;
    static constexpr int BOX_ROWS = KC <= 256 ? KC : KC / 2;
    static constexpr int THREADS = W * 32;
    static constexpr int ENTRY = BF ? 4 : 8;       // list entry bytes
    static constexpr int LIST_BYTES = W * 32 * ENTRY;
    static constexpr int SMEM = 2 * STAGE + 64 + LIST_BYTES;
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

template <bool BF, int L, int R, int W, int KC>
__global__ void __launch_bounds__(W * 32, 2)
    spmm_kernel(const __grid_constant__ CUtensorMap tmB, const SpmmArgs a) {
    using C_ = SpmmCfg<BF, L, R, W, KC>;
    constexpr int G = C_::G, PITCH = C_::PITCH, STAGE = C_::STAGE, ENTRY = C_::ENTRY;

    extern __shared__ __align__(1024) unsigned char smem[];
    unsigned char* stages = smem;
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + 2 * STAGE);
    int* kr = reinterpret_cast<int*>(smem + 2 * STAGE + 16);  // [0]=min col, [1]=max col, [2]=abort
    unsigned char* lists = smem + 2 * STAGE + 64;

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
        const int s = j & 1;
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
        if (nchunks > 1) issue(1);
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
        const int s = j & 1;
        const int k0 = (c_lo + j) * KC;
        const bool ok = mbar_wait_bounded(smem_addr(&bars[s]), (j >> 1) & 1, kWaitLimitNs);
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
                float c4[4] = {0.f, 0.f, 0.f, 0.f};  // fp32: this segment's partial sums
                while (true) {
                    const bool valid = (rc + lane < re) && ((unsigned)(col - k0) < (unsigned)KC);
                    const unsigned bal = __ballot_sync(kFullMask, valid);
                    const int n = (bal == kFullMask) ? 32 : (__ffs(~bal) - 1);  // valid prefix
                    if (n == 0) break;
                    const int npad = (n + 4 * G - 1) / (4 * G) * (4 * G);
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
                    const int q = npad / G;  // steps of each group, multiple of 4
                    const uint32_t gl = wl_addr + g * q * ENTRY;
#pragma unroll 1
                    for (int t = 0; t < q; t += 4) {
                        if constexpr (BF) {
                            const uint4 e = lds128(gl + t * 4);
                            const uint32_t ev[4] = {e.x, e.y, e.z, e.w};
                            uint2 b[4];
#pragma unroll
                            for (int u = 0; u < 4; ++u) b[u] = lds64(stage + ((ev[u] & 0xffffu) << 3));
#pragma unroll
                            for (int u = 0; u < 4; ++u) {
                                acc[i][0] = fma_bf16_hl(ev[u], b[u].x, acc[i][0]);
                                acc[i][1] = fma_bf16_hh(ev[u], b[u].x, acc[i][1]);
                                acc[i][2] = fma_bf16_hl(ev[u], b[u].y, acc[i][2]);
                                acc[i][3] = fma_bf16_hh(ev[u], b[u].y, acc[i][3]);
                            }
                        } else {
                            const uint4 e01 = lds128(gl + t * 8);
                            const uint4 e23 = lds128(gl + t * 8 + 16);
                            const uint32_t off[4] = {e01.x, e01.z, e23.x, e23.z};
                            const uint32_t av[4] = {e01.y, e01.w, e23.y, e23.w};
                            uint4 b[4];
#pragma unroll
                            for (int u = 0; u < 4; ++u) b[u] = lds128(stage + off[u]);
                            float2 lo = make_float2(c4[0], c4[1]), hi = make_float2(c4[2], c4[3]);
#pragma unroll
                            for (int u = 0; u < 4; ++u) {
                                const float x = __uint_as_float(av[u]);
                                const float2 a2 = make_float2(x, x);
                                lo = __ffma2_rn(a2, make_float2(__uint_as_float(b[u].x), __uint_as_float(b[u].y)), lo);
                                hi = __ffma2_rn(a2, make_float2(__uint_as_float(b[u].z), __uint_as_float(b[u].w)), hi);
                            }
                            c4[0] = lo.x;
                            c4[1] = lo.y;
                            c4[2] = hi.x;
                            c4[3] = hi.y;
                        }
                    }
                    __syncwarp();
                    rc += n;
                    if (n < 32) break;
                    load_window<BF>(a, rc, re, lane, col, val);
                }
                if constexpr (!BF) {
#pragma unroll
                    for (int v = 0; v < 4; ++v) acc[i][v] += c4[v];
                }
                if (lane == i) cur = rc;
                if (i + 1 == R)
                    load_window<BF>(a, __shfl_sync(kFullMask, cur, 0), __shfl_sync(kFullMask, my_end, 0),
                                    lane, pcol, pval);
            }
        }
        __syncthreads();  // every warp is done with stage s
        if (kr[2]) break;
        if (threadIdx.x == 0 && j + 2 < nchunks) {
            fence_proxy_async_smem();
            issue(j + 2);
        }
    }

    if (kr[2]) {
        // A transfer never completed: record it, wait (bounded) for the copies
        // still in flight so none lands after the CTA exits, and leave.
        if (threadIdx.x == 0) {
            record_status(a.status, USM_ERR_TIMEOUT);
            for (int b = 0; b < nchunks && b < 2; ++b) {
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

template <bool BF, int L, int R, int W, int KC>
int launch_cfg(const SpmmArgs& a, const void* B, int ldb, cudaStream_t stream) {
    using C_ = SpmmCfg<BF, L, R, W, KC>;
    CUtensorMap map;
    if (!encode_tensor_map_2d(&map, B, BF, a.K, a.N, ldb, C_::NT, C_::BOX_ROWS)) return USM_ERR_CUDA;
    auto kern = spmm_kernel<BF, L, R, W, KC>;
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
// 4 rows per warp and 16 warps (64 rows per CTA), two CTAs per SM; stages
// of 48 KB.
int launch_spmm(const SpmmArgs& a, const void* B, int ldb, bool bf16, cudaStream_t stream) {
    constexpr int W = 16, R = 4;
    if (!bf16) {
        if (a.N <= 64) return launch_cfg<false, 16, R, W, 192>(a, B, ldb, stream);
        return launch_cfg<false, 32, R, W, 96>(a, B, ldb, stream);
    }
    if (a.N <= 64) return launch_cfg<true, 16, R, W, 384>(a, B, ldb, stream);
    return launch_cfg<true, 32, R, W, 192>(a, B, ldb, stream);
}

}  // namespace usm
