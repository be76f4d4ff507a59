// Row swizzle for sm_103a.
//
// "Sparse GPU Kernels for Deep Learning" (Gale et al., SC 2020), summary
// card: the kernels use a decoupled load-balancing scheme ("Summary"), the
// "row swizzle", which balances work independently of how the computation is
// split across processing elements ("Interesting ideas" I4).  Reading used
// here: the processing order lists rows by decreasing length, rows of equal
// length by increasing index; with seg_rows > 0 the order is built inside
// each run of seg_rows consecutive rows.
//
// Build: a stable least-significant-digit radix sort of the row ids on the
// key (segment, K - length), 8 bits per pass.  The same sort (keyed by column
// index) gives the CSR transpose its order.  The input is the identity
// order, so stability supplies the ascending-index tie-break and the result
// is unique and bit-exact.  Each pass is three kernels: per-tile digit
// histograms, one exclusive scan over (digit, tile), and a stable scatter in
// which each tile ranks equal digits with warp match masks and per-warp
// counts.  Everything is integer arithmetic.
#include <climits>

#include "usm_device.cuh"
#include "usm_internal.h"

namespace usm {
namespace {

constexpr int kTile = 2048;   // items per tile
constexpr int kThreads = 256; // threads per tile block
constexpr int kWarps = kThreads / 32;

__device__ __forceinline__ unsigned long long item_key(const SortSpec& c, int item) {
    if (c.kind == SortKey::Column) {
        int col = __ldg(c.col_indices + item);
        col = min(max(col, 0), max(c.K - 1, 0));
        return (unsigned long long)col;
    }
    int s = __ldg(c.row_offsets + item), e = __ldg(c.row_offsets + item + 1);
    long long len = (long long)e - s;
    if (len < 0) len = 0;
    if (len > c.K) len = c.K;
    const unsigned long long seg = (unsigned long long)(item / c.seg_rows);
    return (seg << c.len_bits) | (unsigned long long)(c.K - len);
}

__device__ __forceinline__ int digit_of(unsigned long long key, int shift) {
    return (int)((key >> shift) & 0xffull);
}

__global__ void radix_hist_kernel(SortSpec c, const int* __restrict__ in, int shift, int ntiles,
                                  int* __restrict__ hist) {
    __shared__ int h[256];
    for (int i = threadIdx.x; i < 256; i += blockDim.x) h[i] = 0;
    __syncthreads();
    const int tile = blockIdx.x;
    const long long base = (long long)tile * kTile;
    for (int i = threadIdx.x; i < kTile; i += blockDim.x) {
        const long long idx = base + i;
        if (idx < c.n) {
            const int it = in ? __ldg(in + idx) : (int)idx;
            atomicAdd(&h[digit_of(item_key(c, it), shift)], 1);
        }
    }
    __syncthreads();
    for (int d = threadIdx.x; d < 256; d += blockDim.x) hist[(long long)d * ntiles + tile] = h[d];
}

__global__ void radix_scatter_kernel(SortSpec c, const int* __restrict__ in, int shift, int ntiles,
                                     const int* __restrict__ offsets, int* __restrict__ out) {
    __shared__ int running[256];
    __shared__ int wcount[kWarps][256];
    const int tile = blockIdx.x;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    for (int d = threadIdx.x; d < 256; d += blockDim.x)
        running[d] = offsets[(long long)d * ntiles + tile];
    const long long base = (long long)tile * kTile;
    for (int round = 0; round < kTile / kThreads; ++round) {
        for (int i = threadIdx.x; i < kWarps * 256; i += blockDim.x) (&wcount[0][0])[i] = 0;
        __syncthreads();
        const long long idx = base + round * kThreads + threadIdx.x;
        const bool live = idx < c.n;
        int it = 0, d = -1;
        if (live) {
            it = in ? __ldg(in + idx) : (int)idx;
            d = digit_of(item_key(c, it), shift);
        }
        // Lanes of this warp holding the same digit, and this lane's rank
        // among them (lanes are in item order, so ranks are stable).
        const unsigned peers = __match_any_sync(kFullMask, d);
        const int rank_in_warp = __popc(peers & ((1u << lane) - 1u));
        if (live && rank_in_warp == 0) wcount[warp][d] = __popc(peers);
        __syncthreads();
        // Per digit: prefix over warps of this round, then advance `running`.
        for (int dd = threadIdx.x; dd < 256; dd += blockDim.x) {
            int run = running[dd];
            for (int w = 0; w < kWarps; ++w) {
                const int v = wcount[w][dd];
                wcount[w][dd] = run;
                run += v;
            }
            running[dd] = run;
        }
        __syncthreads();
        if (live) out[wcount[warp][d] + rank_in_warp] = it;
        __syncthreads();
    }
}

// Exclusive scan of n ints in place, one block (sums kept in 64 bits).
__global__ void exclusive_scan_kernel(int* __restrict__ data, long long n) {
    __shared__ long long sums[1024];
    const int t = threadIdx.x;
    const long long per = (n + blockDim.x - 1) / blockDim.x;
    const long long b = t * per, e = min(n, b + per);
    long long s = 0;
    for (long long i = b; i < e; ++i) s += data[i];
    sums[t] = s;
    __syncthreads();
    if (t == 0) {
        long long run = 0;
        for (int i = 0; i < (int)blockDim.x; ++i) {
            const long long v = sums[i];
            sums[i] = run;
            run += v;
        }
    }
    __syncthreads();
    long long run = sums[t];
    for (long long i = b; i < e; ++i) {
        const int v = data[i];
        data[i] = (int)run;
        run += v;
    }
}

}  // namespace

int launch_exclusive_scan(int* data, long long n, cudaStream_t stream) {
    if (n <= 0) return USM_OK;
    exclusive_scan_kernel<<<1, 1024, 0, stream>>>(data, n);
    return cudaGetLastError() == cudaSuccess ? USM_OK : USM_ERR_CUDA;
}

int bits_for(long long v) {  // bits needed to hold 0..v
    int b = 0;
    while (b < 62 && (v >> b) != 0) ++b;
    return b;
}

size_t stable_sort_workspace_bytes(long long n) {
    if (n <= 0) return 0;
    const long long ntiles = (n + kTile - 1) / kTile;
    return (size_t)n * sizeof(int) + (size_t)(256 * ntiles) * sizeof(int);
}

int launch_stable_sort(const SortSpec& spec, int key_bits, int* out, void* ws, size_t ws_bytes,
                       cudaStream_t stream) {
    if (spec.n <= 0) return USM_OK;
    if (ws == nullptr || ws_bytes < stable_sort_workspace_bytes(spec.n)) return USM_ERR_WORKSPACE;
    const int ntiles = (int)((spec.n + kTile - 1) / kTile);
    int* tmp = static_cast<int*>(ws);
    int* hist = tmp + spec.n;
    int passes = (key_bits + 7) / 8;
    if (passes == 0) passes = 1;
    // Ping-pong so the last pass lands in `out`.
    const int* src = nullptr;  // identity order on the first pass
    for (int p = 0; p < passes; ++p) {
        int* dst = ((passes - 1 - p) % 2 == 0) ? out : tmp;
        radix_hist_kernel<<<ntiles, kThreads, 0, stream>>>(spec, src, 8 * p, ntiles, hist);
        exclusive_scan_kernel<<<1, 1024, 0, stream>>>(hist, 256LL * ntiles);
        radix_scatter_kernel<<<ntiles, kThreads, 0, stream>>>(spec, src, 8 * p, ntiles, hist, dst);
        if (cudaGetLastError() != cudaSuccess) return USM_ERR_CUDA;
        src = dst;
    }
    return USM_OK;
}

size_t swizzle_workspace_bytes(int M, int K) {
    (void)K;
    return stable_sort_workspace_bytes(M);
}

int launch_row_swizzle(int M, int K, int seg_rows, const int* row_offsets, int* perm, void* ws,
                       size_t ws_bytes, cudaStream_t stream) {
    if (M <= 0) return USM_OK;
    if (seg_rows <= 0 || seg_rows > M) seg_rows = M;
    SortSpec c{SortKey::RowSwizzle, row_offsets, nullptr, M, K, seg_rows, bits_for(K)};
    const int seg_bits = bits_for((M - 1) / seg_rows);
    return launch_stable_sort(c, c.len_bits + seg_bits, perm, ws, ws_bytes, stream);
}

}  // namespace usm
