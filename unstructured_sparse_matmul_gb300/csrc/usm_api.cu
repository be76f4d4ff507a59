// C ABI of the library: argument checks, dispatch, status word, tensor maps.
// The declarations and their contracts are in include/usm.h.
#include <cudaTypedefs.h>

#include <atomic>
#include <mutex>

#include "usm_device.cuh"
#include "usm_internal.h"

namespace usm {

// One status word per device (a __device__ variable exists once in every
// device context that loads this module).
__device__ int g_status_word;

namespace {

constexpr int kMaxDevices = 64;
std::atomic<int> g_sm_count[kMaxDevices];
std::once_flag g_encode_once;
PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;
std::once_flag g_ctx_once;
PFN_cuCtxGetCurrent_v4000 g_ctx_get_current = nullptr;
PFN_cuCtxGetId_v12000 g_ctx_get_id = nullptr;
std::mutex g_symbol_mutex;

void* driver_entry(const char* name, unsigned version) {
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion(name, &fn, version, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
        return fn;
    return nullptr;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

cudaStream_t as_stream(void* s) { return reinterpret_cast<cudaStream_t>(s); }

__global__ void wait_timeout_selftest_kernel(long long limit_ns, int* status) {
    __shared__ uint64_t bar;
    if (threadIdx.x == 0) {
        mbar_init(smem_addr(&bar), 1);
        fence_barrier_init();
    }
    __syncthreads();
    // Nothing ever arrives on this barrier: the wait must give up by itself.
    if (threadIdx.x == 0 && !mbar_wait_bounded(smem_addr(&bar), 0, (unsigned long long)limit_ns))
        record_status(status, USM_ERR_TIMEOUT);
}

}  // namespace

unsigned long long current_context_id() {
    std::call_once(g_ctx_once, [] {
        g_ctx_get_current = reinterpret_cast<PFN_cuCtxGetCurrent_v4000>(driver_entry("cuCtxGetCurrent", 4000));
        g_ctx_get_id = reinterpret_cast<PFN_cuCtxGetId_v12000>(driver_entry("cuCtxGetId", 12000));
    });
    if (!g_ctx_get_current || !g_ctx_get_id) return 0;
    CUcontext ctx = nullptr;
    if (g_ctx_get_current(&ctx) != CUDA_SUCCESS || ctx == nullptr) return 0;
    unsigned long long id = 0;
    if (g_ctx_get_id(ctx, &id) != CUDA_SUCCESS) return 0;
    return id;
}

void* SymbolAddressCache::get() {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
    std::lock_guard<std::mutex> lock(g_symbol_mutex);
    const unsigned long long ctx = current_context_id();
    if (ctx != 0 && ctx == ctx_[dev] && addr_[dev] != nullptr) return addr_[dev];
    // First use in this context (or no context current yet): the lookup
    // makes the device's primary context current and may load the module.
    void* addr = nullptr;
    if (cudaGetSymbolAddress(&addr, symbol_) != cudaSuccess || addr == nullptr) return nullptr;
    ctx_[dev] = current_context_id();
    addr_[dev] = addr;
    return addr;
}

namespace {
SymbolAddressCache g_status_cache(&g_status_word);
}  // namespace

int* status_word_for_current_device() { return static_cast<int*>(g_status_cache.get()); }

int sm_count_current_device() {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return 148;
    int n = g_sm_count[dev].load(std::memory_order_relaxed);
    if (n > 0) return n;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0)
        n = 148;
    g_sm_count[dev].store(n, std::memory_order_relaxed);
    return n;
}

bool encode_tensor_map_2d(CUtensorMap* map, const void* base, bool bf16, long long rows,
                          long long cols, long long ld_elems, int box_cols, int box_rows) {
    std::call_once(g_encode_once, [] {
        g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(driver_entry("cuTensorMapEncodeTiled", 12000));
    });
    if (!g_encode) return false;
    const int es = bf16 ? 2 : 4;
    cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
    cuuint64_t strides[1] = {(cuuint64_t)(ld_elems * es)};
    cuuint32_t box[2] = {(cuuint32_t)box_cols, (cuuint32_t)box_rows};
    cuuint32_t estr[2] = {1, 1};
    CUresult r = g_encode(map, bf16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2,
                          const_cast<void*>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                          CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                          CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

int launch_wait_timeout_selftest(long long limit_ns, int* status, cudaStream_t stream) {
    wait_timeout_selftest_kernel<<<1, 32, 0, stream>>>(limit_ns, status);
    return cudaGetLastError() == cudaSuccess ? USM_OK : USM_ERR_CUDA;
}

}  // namespace usm

using namespace usm;

namespace {
std::atomic<int> g_override_rows{0}, g_override_tiles{0}, g_override_splits{0};
}  // namespace

namespace usm {
ScheduleOverride schedule_override() {
    return {g_override_rows.load(std::memory_order_relaxed), g_override_tiles.load(std::memory_order_relaxed),
            g_override_splits.load(std::memory_order_relaxed)};
}
}  // namespace usm

extern "C" {

int csr_spmm(int M, int K, int N, int nnz, const int* row_offsets, const int* col_indices,
             const void* values, const int* row_swizzle, int seg_rows, const void* B, int ldb, float* C,
             int ldc, usm_dtype dtype, void* stream) {
    if (M < 0 || K < 0 || N < 0 || nnz < 0) return USM_ERR_INVALID_ARG;
    if (dtype != USM_F32 && dtype != USM_BF16) return USM_ERR_INVALID_ARG;
    if (M == 0 || N == 0) return USM_OK;
    if (ldc < N) return USM_ERR_INVALID_ARG;
    if (!C || !row_offsets) return USM_ERR_INVALID_ARG;
    if (!aligned16(C) || (ldc % 4) != 0) return USM_ERR_ALIGNMENT;
    if (nnz > 0 && K == 0) return USM_ERR_INVALID_ARG;
    cudaStream_t st = as_stream(stream);
    if (nnz == 0) return launch_fill_f32(C, M, N, ldc, st);
    if (!col_indices || !values || !B) return USM_ERR_INVALID_ARG;
    if (ldb < N) return USM_ERR_INVALID_ARG;
    const int es = dtype == USM_BF16 ? 2 : 4;
    if (!aligned16(B) || ((long long)ldb * es) % 16 != 0) return USM_ERR_ALIGNMENT;
    int* status = status_word_for_current_device();
    if (!status) return USM_ERR_CUDA;
    SpmmArgs a{M, K, N, nnz, row_offsets, col_indices, values, row_swizzle, effective_seg(M, seg_rows), C, ldc,
               status};
    return launch_spmm(a, B, ldb, dtype == USM_BF16, st);
}

int csr_spmm_row_softmax(int M, int K, int N, int nnz, const int* row_offsets, const int* col_indices,
                         const float* scores, const int* row_swizzle, int seg_rows, const void* B, int ldb, float* C,
                         int ldc, usm_dtype dtype, void* stream) {
    if (M < 0 || K < 0 || N < 0 || nnz < 0) return USM_ERR_INVALID_ARG;
    if (dtype != USM_F32 && dtype != USM_BF16) return USM_ERR_INVALID_ARG;
    if (M == 0 || N == 0) return USM_OK;
    if (ldc < N) return USM_ERR_INVALID_ARG;
    if (!C || !row_offsets) return USM_ERR_INVALID_ARG;
    if (!aligned16(C) || (ldc % 4) != 0) return USM_ERR_ALIGNMENT;
    if (nnz > 0 && K == 0) return USM_ERR_INVALID_ARG;
    cudaStream_t st = as_stream(stream);
    if (nnz == 0) return launch_fill_f32(C, M, N, ldc, st);
    if (!col_indices || !scores || !B) return USM_ERR_INVALID_ARG;
    if (ldb < N) return USM_ERR_INVALID_ARG;
    const int es = dtype == USM_BF16 ? 2 : 4;
    if (!aligned16(B) || ((long long)ldb * es) % 16 != 0) return USM_ERR_ALIGNMENT;
    int* status = status_word_for_current_device();
    if (!status) return USM_ERR_CUDA;
    SpmmArgs a{M, K, N, nnz, row_offsets, col_indices, scores, row_swizzle, effective_seg(M, seg_rows), C, ldc,
               status};
    return launch_spmm(a, B, ldb, dtype == USM_BF16, st, true);
}

size_t csr_sddmm_workspace_bytes(int M, int K, int D, int nnz, usm_dtype in_dtype) {
    if (M <= 0 || K < 0 || D <= 0 || nnz <= 0) return 0;
    return sddmm_workspace_bytes(M, K, D, nnz, in_dtype == USM_BF16);
}

int csr_sddmm(int M, int K, int D, int nnz, const int* row_offsets, const int* col_indices,
              const int* row_swizzle, int seg_rows, const void* X, int ldx, const void* Y, int ldy, void* out,
              usm_dtype in_dtype, usm_dtype out_dtype, void* workspace, size_t workspace_bytes,
              void* stream) {
    if (M < 0 || K < 0 || D < 0 || nnz < 0) return USM_ERR_INVALID_ARG;
    if ((in_dtype != USM_F32 && in_dtype != USM_BF16) || (out_dtype != USM_F32 && out_dtype != USM_BF16))
        return USM_ERR_INVALID_ARG;
    if (M == 0 || nnz == 0) return USM_OK;
    if (!out || !row_offsets || !col_indices) return USM_ERR_INVALID_ARG;
    if (K == 0) return USM_ERR_INVALID_ARG;
    cudaStream_t st = as_stream(stream);
    if (D == 0) return launch_fill_out(out, nnz, out_dtype == USM_BF16, st);
    if (!X || !Y || ldx < D || ldy < D) return USM_ERR_INVALID_ARG;
    const int es = in_dtype == USM_BF16 ? 2 : 4;
    if (!aligned16(X) || !aligned16(Y) || ((long long)ldx * es) % 16 != 0 ||
        ((long long)ldy * es) % 16 != 0)
        return USM_ERR_ALIGNMENT;
    const size_t need = sddmm_workspace_bytes(M, K, D, nnz, in_dtype == USM_BF16);
    if (need > 0 && (workspace == nullptr || workspace_bytes < need)) return USM_ERR_WORKSPACE;
    if (need > 0 && !aligned16(workspace)) return USM_ERR_ALIGNMENT;
    int* status = status_word_for_current_device();
    if (!status) return USM_ERR_CUDA;
    SddmmArgs a{M, K, D, nnz, row_offsets, col_indices, row_swizzle, effective_seg(M, seg_rows), X, ldx, out, 0,
                out_dtype == USM_BF16 ? 1 : 0, 1, status};
    return launch_sddmm(a, Y, ldy, in_dtype == USM_BF16, workspace, workspace_bytes, st);
}

size_t row_swizzle_workspace_bytes(int M, int K) {
    if (M <= 0 || K < 0) return 0;
    return swizzle_workspace_bytes(M, K);
}

int row_swizzle_build(int M, int K, int seg_rows, const int* row_offsets, int* swizzle_out,
                      void* workspace, size_t workspace_bytes, void* stream) {
    if (M < 0 || K < 0) return USM_ERR_INVALID_ARG;
    if (M == 0) return USM_OK;
    if (!row_offsets || !swizzle_out) return USM_ERR_INVALID_ARG;
    if (!workspace || workspace_bytes < swizzle_workspace_bytes(M, K)) return USM_ERR_WORKSPACE;
    if ((reinterpret_cast<uintptr_t>(workspace) & 3u) != 0) return USM_ERR_ALIGNMENT;
    return launch_row_swizzle(M, K, seg_rows, row_offsets, swizzle_out, workspace, workspace_bytes,
                              as_stream(stream));
}

namespace {
size_t align256(size_t b) { return (b + 255) / 256 * 256; }
// Leading dimension of the transposed Y the general SDDMM builds (16-byte rows).
long long yt_ld(int D, bool bf16) {
    const int per = bf16 ? 8 : 4;
    return ((long long)D + per - 1) / per * per;
}
size_t general_yt_bytes(int K, int D, bool bf16, int y_transposed) {
    if (y_transposed || K <= 0 || D <= 0) return 0;
    return align256((size_t)K * (size_t)yt_ld(D, bf16) * (bf16 ? 2 : 4));
}
}  // namespace

size_t csr_sddmm_general_workspace_bytes(int M, int K, int D, int nnz, usm_dtype in_dtype, int y_transposed) {
    if (M <= 0 || K < 0 || D <= 0 || nnz <= 0) return 0;
    const bool bf = in_dtype == USM_BF16;
    return general_yt_bytes(K, D, bf, y_transposed) + sddmm_workspace_bytes(M, K, D, nnz, bf);
}

int csr_sddmm_general(int M, int K, int D, int nnz, const int* row_offsets, const int* col_indices,
                      const void* values, const int* row_swizzle, int seg_rows, const void* X, int ldx,
                      const void* Y, int ldy,
                      int y_transposed, void* out, usm_dtype in_dtype, usm_dtype out_dtype, void* workspace,
                      size_t workspace_bytes, void* stream) {
    if (M < 0 || K < 0 || D < 0 || nnz < 0) return USM_ERR_INVALID_ARG;
    if ((in_dtype != USM_F32 && in_dtype != USM_BF16) || (out_dtype != USM_F32 && out_dtype != USM_BF16))
        return USM_ERR_INVALID_ARG;
    if (y_transposed != 0 && y_transposed != 1) return USM_ERR_INVALID_ARG;
    if (M == 0 || nnz == 0) return USM_OK;
    if (!out || !row_offsets || !col_indices) return USM_ERR_INVALID_ARG;
    if (K == 0) return USM_ERR_INVALID_ARG;
    cudaStream_t st = as_stream(stream);
    if (D == 0) return launch_fill_out(out, nnz, out_dtype == USM_BF16, st);
    const bool bf = in_dtype == USM_BF16;
    const int es = bf ? 2 : 4;
    if (!X || !Y || ldx < D) return USM_ERR_INVALID_ARG;
    if (y_transposed ? ldy < D : ldy < K) return USM_ERR_INVALID_ARG;
    if (!aligned16(X) || ((long long)ldx * es) % 16 != 0) return USM_ERR_ALIGNMENT;
    if (y_transposed && (!aligned16(Y) || ((long long)ldy * es) % 16 != 0)) return USM_ERR_ALIGNMENT;
    const size_t yt_bytes = general_yt_bytes(K, D, bf, y_transposed);
    const size_t part_bytes = sddmm_workspace_bytes(M, K, D, nnz, bf);
    const size_t need = yt_bytes + part_bytes;
    if (need > 0 && (workspace == nullptr || workspace_bytes < need)) return USM_ERR_WORKSPACE;
    if (need > 0 && (reinterpret_cast<uintptr_t>(workspace) & 255u) != 0) return USM_ERR_ALIGNMENT;
    int* status = status_word_for_current_device();
    if (!status) return USM_ERR_CUDA;
    const void* Yk = Y;
    long long ldyk = ldy;
    if (!y_transposed) {
        ldyk = yt_ld(D, bf);
        const int r = launch_dense_transpose(Y, ldy, D, K, bf, workspace, ldyk, st);
        if (r != USM_OK) return r;
        Yk = workspace;
    }
    if (ldyk > 0x7fffffffLL) return USM_ERR_UNSUPPORTED;
    SddmmArgs a{M, K, D, nnz, row_offsets, col_indices, row_swizzle, effective_seg(M, seg_rows), X, ldx, out, 0,
                out_dtype == USM_BF16 ? 1 : 0, 1, status, values, bf ? 1 : 0};
    void* part = part_bytes ? static_cast<unsigned char*>(workspace) + yt_bytes : nullptr;
    return launch_sddmm(a, Yk, (int)ldyk, bf, part, part_bytes, st);
}

int csr_row_softmax(int M, int nnz, const int* row_offsets, const float* scores, void* out, usm_dtype out_dtype,
                    void* stream) {
    if (M < 0 || nnz < 0) return USM_ERR_INVALID_ARG;
    if (out_dtype != USM_F32 && out_dtype != USM_BF16) return USM_ERR_INVALID_ARG;
    if (M == 0 || nnz == 0) return USM_OK;
    if (!row_offsets || !scores || !out) return USM_ERR_INVALID_ARG;
    return launch_row_softmax(M, nnz, row_offsets, scores, out, out_dtype == USM_BF16, as_stream(stream));
}

size_t csr_transpose_workspace_bytes(int M, int K, int nnz) {
    if (M < 0 || K < 0 || nnz <= 0) return 0;
    return transpose_workspace_bytes(M, K, nnz);
}

int csr_transpose(int M, int K, int nnz, const int* row_offsets, const int* col_indices, const void* values,
                  usm_dtype dtype, int* row_offsets_t, int* col_indices_t, void* values_t, int* perm_out,
                  void* workspace, size_t workspace_bytes, void* stream) {
    if (M < 0 || K < 0 || nnz < 0) return USM_ERR_INVALID_ARG;
    if (dtype != USM_F32 && dtype != USM_BF16) return USM_ERR_INVALID_ARG;
    if (!row_offsets_t) return USM_ERR_INVALID_ARG;
    if (nnz > 0 && (K == 0 || !row_offsets || !col_indices || !col_indices_t)) return USM_ERR_INVALID_ARG;
    if ((values == nullptr) != (values_t == nullptr)) return USM_ERR_INVALID_ARG;
    const size_t need = transpose_workspace_bytes(M, K, nnz);
    if (need > 0 && (workspace == nullptr || workspace_bytes < need)) return USM_ERR_WORKSPACE;
    if (need > 0 && (reinterpret_cast<uintptr_t>(workspace) & 255u) != 0) return USM_ERR_ALIGNMENT;
    return launch_csr_transpose(M, K, nnz, row_offsets, col_indices, values, dtype == USM_BF16, row_offsets_t,
                                col_indices_t, values_t, perm_out, workspace, workspace_bytes, as_stream(stream));
}

int csr_permute_values(int nnz, const int* perm, const void* values, usm_dtype dtype, void* out, void* stream) {
    if (nnz < 0) return USM_ERR_INVALID_ARG;
    if (dtype != USM_F32 && dtype != USM_BF16) return USM_ERR_INVALID_ARG;
    if (nnz == 0) return USM_OK;
    if (!perm || !values || !out) return USM_ERR_INVALID_ARG;
    return launch_permute_values(nnz, perm, values, dtype == USM_BF16, out, as_stream(stream));
}

int csr_validate(int M, int K, int nnz, const int* row_offsets, const int* col_indices, int* result, void* stream) {
    if (M < 0 || K < 0 || nnz < 0) return USM_ERR_INVALID_ARG;
    if (!row_offsets || !result || (nnz > 0 && !col_indices)) return USM_ERR_INVALID_ARG;
    if ((uintptr_t)result % alignof(int) != 0) return USM_ERR_ALIGNMENT;
    return launch_csr_validate(M, K, nnz, row_offsets, col_indices, result, as_stream(stream));
}

int usm_poll_status(void* stream) {
    cudaStream_t st = as_stream(stream);
    if (cudaStreamSynchronize(st) != cudaSuccess) return USM_ERR_CUDA;
    int* status = status_word_for_current_device();
    if (!status) return USM_ERR_CUDA;
    int v = 0;
    if (cudaMemcpyAsync(&v, status, sizeof(int), cudaMemcpyDeviceToHost, st) != cudaSuccess)
        return USM_ERR_CUDA;
    if (cudaMemsetAsync(status, 0, sizeof(int), st) != cudaSuccess) return USM_ERR_CUDA;
    if (cudaStreamSynchronize(st) != cudaSuccess) return USM_ERR_CUDA;
    return v;
}

const char* usm_status_string(int status) {
    switch (status) {
        case USM_OK: return "USM_OK";
        case USM_ERR_INVALID_ARG: return "USM_ERR_INVALID_ARG";
        case USM_ERR_ALIGNMENT: return "USM_ERR_ALIGNMENT";
        case USM_ERR_UNSUPPORTED: return "USM_ERR_UNSUPPORTED";
        case USM_ERR_CUDA: return "USM_ERR_CUDA";
        case USM_ERR_TIMEOUT: return "USM_ERR_TIMEOUT";
        case USM_ERR_WORKSPACE: return "USM_ERR_WORKSPACE";
        default: return "USM_UNKNOWN_STATUS";
    }
}

int usm_set_schedule_override(int rows_per_warp, int tiles_per_block, int k_splits) {
    const bool r_ok = rows_per_warp == 0 || (rows_per_warp <= 32 && (rows_per_warp & (rows_per_warp - 1)) == 0);
    if (!r_ok || tiles_per_block < 0 || k_splits < 0 || k_splits > 65535) return USM_ERR_INVALID_ARG;
    g_override_rows.store(rows_per_warp, std::memory_order_relaxed);
    g_override_tiles.store(tiles_per_block, std::memory_order_relaxed);
    g_override_splits.store(k_splits, std::memory_order_relaxed);
    return USM_OK;
}

int usm_selftest_wait_timeout(long long limit_ns, void* stream) {
    if (limit_ns < 1000 || limit_ns > 1000000000LL) return USM_ERR_INVALID_ARG;
    int* status = status_word_for_current_device();
    if (!status) return USM_ERR_CUDA;
    return launch_wait_timeout_selftest(limit_ns, status, as_stream(stream));
}

}  // extern "C"
