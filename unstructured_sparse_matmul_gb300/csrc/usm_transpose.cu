// CSR transpose for sm_103a: Aᵀ (K×M) in CSR from A (M×K).
//
// The sparse layer's input gradient is Aᵀ·dY, an SpMM on the transposed
// weight; "Sparse GPU Kernels for Deep Learning" (Gale et al., SC 2020)
// targets both inference and training (summary card, "Summary").  Rows of Aᵀ
// list their column indices (rows of A) in increasing order, so the result is
// the unique transposed CSR and the transpose is bit-exact.
//
// Steps, all on the GPU:
//   1. row id of every nonzero (each warp expands one row at a time);
//   2. stable radix sort of the nonzero positions by column index — the
//      input order is row-major, so stability leaves the rows of each column
//      in increasing order;
//   3. row_offsets of Aᵀ: per-column counts (integer atomics, exact) and an
//      exclusive scan;
//   4. gather: col_indices_t[q] = rowid[perm[q]], values_t[q] = values[perm[q]].
// The permutation can be returned so later steps re-gather new values with
// csr_permute_values without sorting again (the pattern is fixed while the
// weights change).
#include "usm_device.cuh"
#include "usm_internal.h"

namespace usm {
namespace {

__global__ void expand_rowid_kernel(int M, int nnz, const int* __restrict__ ro, int* __restrict__ rowid) {
    const int lane = threadIdx.x & 31;
    const int warps = (gridDim.x * blockDim.x) >> 5;
    for (int r = (blockIdx.x * blockDim.x + threadIdx.x) >> 5; r < M; r += warps) {
        int s = __ldg(ro + r), e = __ldg(ro + r + 1);
        s = min(max(s, 0), nnz);
        e = min(max(e, s), nnz);
        for (int p = s + lane; p < e; p += 32) rowid[p] = r;
    }
}

__global__ void column_count_kernel(int nnz, int K, const int* __restrict__ ci, int* __restrict__ counts) {
    for (long long p = blockIdx.x * (long long)blockDim.x + threadIdx.x; p < nnz;
         p += (long long)gridDim.x * blockDim.x) {
        const int c = min(max(__ldg(ci + p), 0), K - 1);
        atomicAdd(counts + c, 1);
    }
}

__global__ void zero_ints_kernel(int* __restrict__ x, long long n) {
    for (long long i = blockIdx.x * (long long)blockDim.x + threadIdx.x; i < n;
         i += (long long)gridDim.x * blockDim.x)
        x[i] = 0;
}

template <typename T>
__global__ void gather_kernel(int nnz, const int* __restrict__ perm, const int* __restrict__ rowid,
                              const T* __restrict__ vals, int* __restrict__ ci_t, T* __restrict__ vals_t,
                              int* __restrict__ perm_out) {
    for (long long q = blockIdx.x * (long long)blockDim.x + threadIdx.x; q < nnz;
         q += (long long)gridDim.x * blockDim.x) {
        const int p = __ldg(perm + q);
        ci_t[q] = __ldg(rowid + p);
        if (vals_t) vals_t[q] = vals[p];
        if (perm_out) perm_out[q] = p;
    }
}

template <typename T>
__global__ void permute_kernel(int nnz, const int* __restrict__ perm, const T* __restrict__ vals,
                               T* __restrict__ out) {
    for (long long q = blockIdx.x * (long long)blockDim.x + threadIdx.x; q < nnz;
         q += (long long)gridDim.x * blockDim.x)
        out[q] = vals[__ldg(perm + q)];
}

int grid_for(long long n) {
    long long b = (n + 255) / 256;
    const long long cap = 8LL * sm_count_current_device();
    if (b > cap) b = cap;
    return (int)(b < 1 ? 1 : b);
}

}  // namespace

size_t transpose_workspace_bytes(int M, int K, int nnz) {
    (void)M;
    (void)K;
    if (nnz <= 0) return 0;
    // rowid[nnz] + perm[nnz] + sort scratch, each region 256-byte aligned
    auto al = [](size_t b) { return (b + 255) / 256 * 256; };
    return al((size_t)nnz * 4) * 2 + al(stable_sort_workspace_bytes(nnz));
}

int launch_csr_transpose(int M, int K, int nnz, const int* ro, const int* ci, const void* values, bool bf16,
                         int* ro_t, int* ci_t, void* values_t, int* perm_out, void* ws, size_t ws_bytes,
                         cudaStream_t stream) {
    // Row offsets of Aᵀ: counts per column, then an exclusive scan over K+1.
    zero_ints_kernel<<<grid_for(K + 1), 256, 0, stream>>>(ro_t, (long long)K + 1);
    if (nnz > 0) column_count_kernel<<<grid_for(nnz), 256, 0, stream>>>(nnz, K, ci, ro_t);
    if (cudaGetLastError() != cudaSuccess) return USM_ERR_CUDA;
    int st = launch_exclusive_scan(ro_t, (long long)K + 1, stream);
    if (st != USM_OK || nnz == 0) return st;
    if (ws == nullptr || ws_bytes < transpose_workspace_bytes(M, K, nnz)) return USM_ERR_WORKSPACE;
    auto al = [](size_t b) { return (b + 255) / 256 * 256; };
    unsigned char* w = static_cast<unsigned char*>(ws);
    int* rowid = reinterpret_cast<int*>(w);
    int* perm = reinterpret_cast<int*>(w + al((size_t)nnz * 4));
    void* sort_ws = w + 2 * al((size_t)nnz * 4);
    expand_rowid_kernel<<<grid_for((long long)M * 32), 256, 0, stream>>>(M, nnz, ro, rowid);
    if (cudaGetLastError() != cudaSuccess) return USM_ERR_CUDA;
    SortSpec spec{SortKey::Column, nullptr, ci, nnz, K, 1, 0};
    st = launch_stable_sort(spec, bits_for(K > 0 ? K - 1 : 0), perm, sort_ws, stable_sort_workspace_bytes(nnz),
                            stream);
    if (st != USM_OK) return st;
    if (bf16)
        gather_kernel<uint16_t><<<grid_for(nnz), 256, 0, stream>>>(
            nnz, perm, rowid, static_cast<const uint16_t*>(values), ci_t, static_cast<uint16_t*>(values_t),
            perm_out);
    else
        gather_kernel<float><<<grid_for(nnz), 256, 0, stream>>>(nnz, perm, rowid, static_cast<const float*>(values),
                                                                ci_t, static_cast<float*>(values_t), perm_out);
    return cudaGetLastError() == cudaSuccess ? USM_OK : USM_ERR_CUDA;
}

int launch_permute_values(int nnz, const int* perm, const void* values, bool bf16, void* out,
                          cudaStream_t stream) {
    if (nnz <= 0) return USM_OK;
    if (bf16)
        permute_kernel<uint16_t><<<grid_for(nnz), 256, 0, stream>>>(nnz, perm, static_cast<const uint16_t*>(values),
                                                                    static_cast<uint16_t*>(out));
    else
        permute_kernel<float><<<grid_for(nnz), 256, 0, stream>>>(nnz, perm, static_cast<const float*>(values),
                                                                 static_cast<float*>(out));
    return cudaGetLastError() == cudaSuccess ? USM_OK : USM_ERR_CUDA;
}

}  // namespace usm
