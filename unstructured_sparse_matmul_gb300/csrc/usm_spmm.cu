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
//   exactly one lane in a fixed order: results do not depend on the swizzle.
// * Dense operand staging.  The CTA walks K in chunks of KC rows.  For each
//   chunk one thread issues TMA tensor copies of B[k0:k0+KC, n0:n0+NT] into a
//   shared-memory stage (double buffered, completion on an mbarrier, bounded
//   wait).  Only the chunks between the smallest and largest column index of
//   the CTA's rows are fetched, so block-diagonal (batched) matrices stay
//   cheap.
// * Sparse operand.  For each (row, chunk) a warp reads the next 32 column
//   indices and values of the row with coalesced loads (the window of the
//   row after its cursor, so a misaligned row start costs nothing), keeps the
//   prefix whose columns fall in the chunk (ballot), and writes
//   (byte offset into the stage, value) entries to a per-warp list.  The
//   window of the next row is prefetched while the current row computes.
// * Inner loop.  G = 32/L lane groups each take one list entry per step:
//   every lane reads 16 bytes of the staged B row (one LDS.128; a group
//   covers a whole 16·L-byte row, conflict-free) and does EPV FMAs into its
//   accumulators (fp32 via packed f32x2 FMA; bf16 operands are widened
//   exactly first).  At the end the G partial rows are added across groups.
// * Accuracy.  In fp32 each (row, chunk) segment (≤ KC terms) is summed into
//   a fresh accumulator that is then added to the row total, so every output
//   is a sum of ≤ KC-term partials: the worst-case rounding bound stays
//   below 1e-5·Σ|a||b| for K up to 4096 with KC = 128.
#include <climits>
#include <type_traits>

#include "usm_device.cuh"
#include "usm_internal.h"

namespace usm {
namespace {

template <bool BF>
struct SpmmEntry;
template <>
struct SpmmEntry<false> {  // fp32: byte offset, value bits
    using T = uint2;
};
template <>
struct SpmmEntry<true> {  // bf16: (byte offset / 16) | bf16 value << 16
    using T = uint32_t;
};

template <bool BF, int L, int R, int W, int KC>
struct SpmmCfg {
    static constexpr int EPV = BF ? 8 : 4;  // elements per 16-byte vector
    static constexpr int NT = L * EPV;      // output columns per CTA
    static constexpr int G = 32 / L;        // nonzeros per warp step
    static constexpr int PITCH = L * 16;    // bytes per staged B row
    static constexpr int STAGE = KC * PITCH;
    static constexpr int MT = R * W;
    static constexpr int BOX_ROWS = KC < 256 ? KC : 256;
    static constexpr int THREADS = W * 32;
    using Entry = typename SpmmEntry<BF>::T;
    static constexpr int LIST_BYTES = W * 32 * (int)sizeof(Entry);
    static constexpr int SMEM = 2 * STAGE + 64 + LIST_BYTES;
    static_assert(32 % L == 0, "L must divide the warp");
    static_assert(KC % BOX_ROWS == 0, "KC must be a multiple of the TMA box height");
    static_assert(STAGE <= 65536 * 16, "stage offsets must fit the entry encoding");
};

__device__ __forceinline__ uint4 lds128(uint32_t addr) {
    uint4 v;
    asm volatile("ld.shared.v4.u32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "r"(addr));
    return v;
}

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
__global__ void __launch_bounds__(W * 32, 1)
    spmm_kernel(const __grid_constant__ CUtensorMap tmB, const SpmmArgs a) {
    using C_ = SpmmCfg<BF, L, R, W, KC>;
    using Entry = typename C_::Entry;
    constexpr int EPV = C_::EPV, G = C_::G, PITCH = C_::PITCH, STAGE = C_::STAGE;

    extern __shared__ __align__(1024) unsigned char smem[];
    unsigned char* stages = smem;
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + 2 * STAGE);
    int* kr = reinterpret_cast<int*>(smem + 2 * STAGE + 16);  // [0]=min col, [1]=max col, [2]=abort
    Entry* lists = reinterpret_cast<Entry*>(smem + 2 * STAGE + 64);

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

    float acc[R][EPV];
#pragma unroll
    for (int i = 0; i < R; ++i)
#pragma unroll
        for (int v = 0; v < EPV; ++v) acc[i][v] = 0.f;

    int cur = my_start;  // lane i: cursor of row slot i
    int pcol;
    uint32_t pval;
    load_window<BF>(a, __shfl_sync(kFullMask, cur, 0), __shfl_sync(kFullMask, my_end, 0), lane, pcol,
                    pval);

    Entry* wl = lists + warp * 32;
    bool timed_out = false;

    for (int j = 0; j < nchunks; ++j) {
        const int s = j & 1;
        const int k0 = (c_lo + j) * KC;
        const bool ok = mbar_wait_bounded(smem_addr(&bars[s]), (j >> 1) & 1, kWaitLimitNs);
        if (!ok) {
            timed_out = true;
            kr[2] = 1;
        }
        const uint32_t stage = smem_addr(stages + s * STAGE) + l * 16;
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
                float accc[EPV];
#pragma unroll
                for (int v = 0; v < EPV; ++v) accc[v] = 0.f;
                while (true) {
                    const bool valid = (rc + lane < re) && ((unsigned)(col - k0) < (unsigned)KC);
                    const unsigned bal = __ballot_sync(kFullMask, valid);
                    const int n = (bal == kFullMask) ? 32 : (__ffs(~bal) - 1);  // valid prefix
                    if (n == 0) break;
                    const int npad = (n + G - 1) / G * G;
                    if (lane < npad) {
                        const bool live = lane < n;
                        const uint32_t off = live ? (uint32_t)(col - k0) * PITCH : 0u;
                        if constexpr (BF) {
                            wl[lane] = live ? ((off >> 4) | (val << 16)) : 0u;
                        } else {
                            wl[lane] = live ? make_uint2(off, val) : make_uint2(0u, 0u);
                        }
                    }
                    __syncwarp();
#pragma unroll 4
                    for (int t = g; t < npad; t += G) {
                        if constexpr (BF) {
                            const uint32_t e = wl[t];
                            const uint4 b = lds128(stage + ((e & 0xffffu) << 4));
                            const float av = __uint_as_float(e & 0xffff0000u);
                            const float2 a2 = make_float2(av, av);
                            const uint32_t w[4] = {b.x, b.y, b.z, b.w};
#pragma unroll
                            for (int q = 0; q < 4; ++q) {
                                float2 c2 = make_float2(acc[i][2 * q], acc[i][2 * q + 1]);
                                c2 = __ffma2_rn(a2, make_float2(bf16lo(w[q]), bf16hi(w[q])), c2);
                                acc[i][2 * q] = c2.x;
                                acc[i][2 * q + 1] = c2.y;
                            }
                        } else {
                            const uint2 e = wl[t];
                            const uint4 b = lds128(stage + e.x);
                            const float av = __uint_as_float(e.y);
                            const float2 a2 = make_float2(av, av);
                            float2 c0 = make_float2(accc[0], accc[1]);
                            float2 c1 = make_float2(accc[2], accc[3]);
                            c0 = __ffma2_rn(a2, make_float2(__uint_as_float(b.x), __uint_as_float(b.y)), c0);
                            c1 = __ffma2_rn(a2, make_float2(__uint_as_float(b.z), __uint_as_float(b.w)), c1);
                            accc[0] = c0.x;
                            accc[1] = c0.y;
                            accc[2] = c1.x;
                            accc[3] = c1.y;
                        }
                    }
                    __syncwarp();
                    rc += n;
                    if (n < 32) break;
                    load_window<BF>(a, rc, re, lane, col, val);
                }
                if constexpr (!BF) {
#pragma unroll
                    for (int v = 0; v < EPV; ++v) acc[i][v] += accc[v];
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
            for (int j = 0; j < nchunks && j < 2; ++j) {
                // Stages hold chunks whose phases are unknown here; wait on both
                // parities briefly (each wait ends by itself).
                mbar_wait_bounded(smem_addr(&bars[j]), 0, 1000000ull);
                mbar_wait_bounded(smem_addr(&bars[j]), 1, 1000000ull);
            }
        }
        (void)timed_out;
        return;
    }

    // Add the G partial rows held by the lane groups.
#pragma unroll
    for (int i = 0; i < R; ++i)
#pragma unroll
        for (int v = 0; v < EPV; ++v) {
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
        const int c0 = n0 + l * EPV;
        float* dst = a.C + (long long)row * a.ldc + c0;
        if (c0 + EPV <= a.N) {
#pragma unroll
            for (int v = 0; v < EPV; v += 4)
                *reinterpret_cast<float4*>(dst + v) =
                    make_float4(acc[i][v], acc[i][v + 1], acc[i][v + 2], acc[i][v + 3]);
        } else {
#pragma unroll
            for (int v = 0; v < EPV; ++v)
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

// Tile choice: the widest column strip the lanes can cover without waste,
// and the most rows per CTA (best reuse of each staged B chunk) that still
// gives every SM at least ~2 CTAs.
int launch_spmm(const SpmmArgs& a, const void* B, int ldb, bool bf16, cudaStream_t stream) {
    const int sms = sm_count_current_device();
    auto ctas = [&](int nt, int mt) {
        return (long long)((a.N + nt - 1) / nt) * ((a.M + mt - 1) / mt);
    };
    constexpr int W = 16;
    if (!bf16) {
        if (a.N <= 64) {
            if (ctas(64, 8 * W) >= 2 * sms) return launch_cfg<false, 16, 8, W, 256>(a, B, ldb, stream);
            return launch_cfg<false, 16, 4, W, 256>(a, B, ldb, stream);
        }
        if (ctas(128, 8 * W) >= 2 * sms) return launch_cfg<false, 32, 8, W, 128>(a, B, ldb, stream);
        return launch_cfg<false, 32, 4, W, 128>(a, B, ldb, stream);
    }
    if (a.N <= 64) {
        if (ctas(64, 8 * W) >= 2 * sms) return launch_cfg<true, 8, 8, W, 512>(a, B, ldb, stream);
        return launch_cfg<true, 8, 4, W, 512>(a, B, ldb, stream);
    }
    if (ctas(256, 8 * W) >= 2 * sms) return launch_cfg<true, 32, 8, W, 128>(a, B, ldb, stream);
    return launch_cfg<true, 32, 4, W, 128>(a, B, ldb, stream);
}

}  // namespace usm
