// Row-wise softmax over the stored entries of each CSR row, for the sparse
// attention chain SDDMM → softmax → SpMM (the sparse-attention use of the
// kernels, "Sparse GPU Kernels for Deep Learning", summary card,
// "Interesting ideas" I3):
//     out[p] = exp(s[p] - m_r) / Σ_{q in row r} exp(s[q] - m_r),  m_r = max s.
// One warp per row, three passes over the row (max, sum, write) so no
// running rescale adds error (row_softmax_stats, softmax_prob: the same
// routines the SpMM with a fused softmax uses, so the two agree bit for bit).

#include "usm_device.cuh"
#include "usm_internal.h"

namespace usm {
namespace {

__global__ void row_softmax_kernel(int M, int nnz, const int* __restrict__ ro, const float* __restrict__ s,
                                   void* out, int out_bf16) {
    const int lane = threadIdx.x & 31;
    const int warps = (gridDim.x * blockDim.x) >> 5;
    for (int r = (blockIdx.x * blockDim.x + threadIdx.x) >> 5; r < M; r += warps) {
        int b = __ldg(ro + r), e = __ldg(ro + r + 1);
        b = min(max(b, 0), nnz);
        e = min(max(e, b), nnz);
        if (b == e) continue;
        float m, rz;
        row_softmax_stats(s, b, e, lane, m, rz);
        for (int p = b + lane; p < e; p += 32) {
            const float v = softmax_prob(__ldg(s + p), m, rz);
            if (out_bf16)
                reinterpret_cast<uint16_t*>(out)[p] = f32_to_bf16_rne(v);
            else
                reinterpret_cast<float*>(out)[p] = v;
        }
    }
}

}  // namespace

int launch_row_softmax(int M, int nnz, const int* ro, const float* scores, void* out, bool out_bf16,
                       cudaStream_t stream) {
    if (M <= 0) return USM_OK;
    long long blocks = ((long long)M * 32 + 255) / 256;
    const long long cap = 16LL * sm_count_current_device();
    if (blocks > cap) blocks = cap;
    row_softmax_kernel<<<(int)blocks, 256, 0, stream>>>(M, nnz, ro, scores, out, out_bf16 ? 1 : 0);
    return cudaGetLastError() == cudaSuccess ? USM_OK : USM_ERR_CUDA;
}

}  // namespace usm
