// CSR contract check on the device: the plain CSR the kernels take
// ("Sparse GPU Kernels for Deep Learning", summary card, "Interesting ideas"
// I5: standard CSR, no structural constraint), with the reading that each
// row's column indices are strictly increasing.  Reports the first violation
// in a fixed order: row_offsets[0] = 0, then non-decreasing offsets (first
// row that decreases), then row_offsets[M] = nnz, then the first nonzero
// position whose column is outside [0, K) or not above its predecessor in
// the row (the range test first at a tied position).
//
// Every read is in bounds whatever the input: offsets are read at r and r+1
// for r < M, and a row's entries only inside [0, nnz) after clamping its
// offsets, so a malformed CSR is reported, never followed.
#include <climits>

#include "usm_device.cuh"
#include "usm_internal.h"

namespace usm {
namespace {

// result[0] code, result[1] index, result[2] first decreasing row,
// result[3] first column out of range, result[4] first column out of order.
__global__ void validate_init_kernel(int* result) {
    if (threadIdx.x == 0) {
        result[0] = USM_CSR_VALID;
        result[1] = -1;
        result[2] = INT_MAX;
        result[3] = INT_MAX;
        result[4] = INT_MAX;
    }
}

// A warp per row: lane 0 compares the row's two offsets, the lanes stride
// over the row's entries (clamped to [0, nnz)).
__global__ void validate_scan_kernel(int M, int K, int nnz, const int* __restrict__ ro, const int* __restrict__ ci,
                                     int* result) {
    const int lane = threadIdx.x & 31;
    const long long warps = ((long long)gridDim.x * blockDim.x) >> 5;
    int bad_range = INT_MAX, bad_order = INT_MAX;
    for (long long r = ((long long)blockIdx.x * blockDim.x + threadIdx.x) >> 5; r < M; r += warps) {
        const int b = __ldg(ro + r), e = __ldg(ro + r + 1);
        if (lane == 0 && e < b) atomicMin(result + 2, (int)r);
        const long long s = min(max((long long)b, 0LL), (long long)nnz);
        const long long t = min(max((long long)e, s), (long long)nnz);
        for (long long p = s + lane; p < t; p += 32) {
            const int c = __ldg(ci + p);
            if (c < 0 || c >= K) bad_range = min(bad_range, (int)p);
            if (p > s && c <= __ldg(ci + p - 1)) bad_order = min(bad_order, (int)p);
        }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        bad_range = min(bad_range, __shfl_xor_sync(kFullMask, bad_range, o));
        bad_order = min(bad_order, __shfl_xor_sync(kFullMask, bad_order, o));
    }
    if (lane == 0) {
        if (bad_range != INT_MAX) atomicMin(result + 3, bad_range);
        if (bad_order != INT_MAX) atomicMin(result + 4, bad_order);
    }
}

__global__ void validate_finish_kernel(int M, int nnz, const int* __restrict__ ro, int* result) {
    if (threadIdx.x != 0) return;
    int code = USM_CSR_VALID, index = -1;
    if (ro[0] != 0) {
        code = USM_CSR_FIRST_OFFSET;
        index = 0;
    } else if (result[2] != INT_MAX) {
        code = USM_CSR_OFFSETS_DECREASE;
        index = result[2];
    } else if (ro[M] != nnz) {
        code = USM_CSR_LAST_OFFSET;
        index = M;
    } else if (result[3] != INT_MAX || result[4] != INT_MAX) {
        const bool range_first = result[3] <= result[4];
        code = range_first ? USM_CSR_COLUMN_RANGE : USM_CSR_COLUMN_ORDER;
        index = range_first ? result[3] : result[4];
    }
    result[0] = code;
    result[1] = index;
}

}  // namespace

int launch_csr_validate(int M, int K, int nnz, const int* row_offsets, const int* col_indices, int* result,
                        cudaStream_t stream) {
    validate_init_kernel<<<1, 32, 0, stream>>>(result);
    if (M > 0) {
        long long blocks = ((long long)M * 32 + 255) / 256;
        const long long cap = 16LL * sm_count_current_device();
        if (blocks > cap) blocks = cap;
        validate_scan_kernel<<<(int)blocks, 256, 0, stream>>>(M, K, nnz, row_offsets, col_indices, result);
    }
    validate_finish_kernel<<<1, 32, 0, stream>>>(M, nnz, row_offsets, result);
    return cudaGetLastError() == cudaSuccess ? USM_OK : USM_ERR_CUDA;
}

}  // namespace usm
