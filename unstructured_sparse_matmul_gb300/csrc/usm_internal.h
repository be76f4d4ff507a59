// Host-side declarations shared by the translation units of the library.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include "usm.h"
#include "usm_args.h"

namespace usm {

// Device address of a __device__ variable (`symbol`: its host-side name,
// which is not a device address) in the calling thread's current context,
// looked up with cudaGetSymbolAddress.  The lookup may load the module that
// holds the variable.  The address is cached per device and per context:
// after a device reset or a new primary context the next call looks it up
// again.  Thread-safe.  nullptr if it cannot be resolved.
class SymbolAddressCache {
  public:
    explicit SymbolAddressCache(const void* symbol) : symbol_(symbol) {}
    void* get();

  private:
    static constexpr int kMaxDevices = 64;
    const void* symbol_;
    unsigned long long ctx_[kMaxDevices] = {};  // context id the address belongs to (0: none)
    void* addr_[kMaxDevices] = {};
};

// Unique id of the calling thread's current CUDA context (cuCtxGetId), or 0
// when no context is current or the driver entry points are missing.
unsigned long long current_context_id();

// Device status word of the current device (null if it cannot be resolved).
int* status_word_for_current_device();

// Number of SMs of the current device (cached per device).
int sm_count_current_device();

// Whether chunks of kc_tall staged rows walk K in fewer chunks than chunks of
// kc.  A taller chunk means fewer CTA barriers and refills, but when it saves
// no chunk it only stages more rows past K (zero-filled by the copy).
inline bool taller_chunk_pays(int K, int kc, int kc_tall) {
    return (K + kc_tall - 1) / kc_tall < (K + kc - 1) / kc;
}

// Encode a 2-D row-major tensor map (inner dim = cols) with box
// {box_cols, box_rows}.  Returns false if the driver entry point is missing
// or the encode fails.
bool encode_tensor_map_2d(CUtensorMap* map, const void* base, bool bf16, long long rows,
                          long long cols, long long ld_elems, int box_cols, int box_rows);

// softmax: a.values are fp32 scores and each row's values are their softmax
// probabilities, rounded to B's element type (csr_spmm_row_softmax).
int launch_spmm(const SpmmArgs& a, const void* B, int ldb, bool bf16, cudaStream_t stream, bool softmax = false);
int launch_fill_f32(float* C, int M, int N, long long ldc, cudaStream_t stream);

size_t sddmm_workspace_bytes(int M, int K, int D, int nnz, bool bf16);
// Elements between two strips of SDDMM partials: nnz rounded up to a multiple of 4.
long long partial_stride(long long nnz);
int launch_sddmm(SddmmArgs a, const void* Y, int ldy, bool in_bf16, void* workspace,
                 size_t workspace_bytes, cudaStream_t stream);
int launch_fill_out(void* out, long long n, bool bf16, cudaStream_t stream);
// Dense transpose: dst (cols × rows, leading dimension ldd) = srcᵀ (rows × cols, lds).
int launch_dense_transpose(const void* src, long long lds, int rows, int cols, bool bf16, void* dst,
                           long long ldd, cudaStream_t stream);
int launch_row_softmax(int M, int nnz, const int* row_offsets, const float* scores, void* out, bool out_bf16,
                       cudaStream_t stream);
int launch_csr_validate(int M, int K, int nnz, const int* row_offsets, const int* col_indices, int* result,
                        cudaStream_t stream);

// Stable LSD radix sort of item ids 0..n-1 by a key (8 bits per pass).
enum class SortKey { RowSwizzle, Column };
struct SortSpec {
    SortKey kind;
    const int* row_offsets;  // RowSwizzle: key = (segment, K - row length)
    const int* col_indices;  // Column: key = col_indices[item]
    long long n;             // number of items
    int K;
    int seg_rows;
    int len_bits;
};
size_t stable_sort_workspace_bytes(long long n);
int launch_stable_sort(const SortSpec& spec, int key_bits, int* out, void* ws, size_t ws_bytes,
                       cudaStream_t stream);
int bits_for(long long v);
int launch_exclusive_scan(int* data, long long n, cudaStream_t stream);  // in place, one block

size_t swizzle_workspace_bytes(int M, int K);
int launch_row_swizzle(int M, int K, int seg_rows, const int* row_offsets, int* perm,
                       void* workspace, size_t workspace_bytes, cudaStream_t stream);

size_t transpose_workspace_bytes(int M, int K, int nnz);
int launch_csr_transpose(int M, int K, int nnz, const int* row_offsets, const int* col_indices,
                         const void* values, bool bf16, int* ro_t, int* ci_t, void* values_t, int* perm_out,
                         void* ws, size_t ws_bytes, cudaStream_t stream);
int launch_permute_values(int nnz, const int* perm, const void* values, bool bf16, void* out,
                          cudaStream_t stream);

inline long long block_count(int M, int seg) { return (M + seg - 1) / seg; }
inline int effective_seg(int M, int seg_rows) { return (seg_rows <= 0 || seg_rows > M) ? M : seg_rows; }

int launch_wait_timeout_selftest(long long limit_ns, int* status, cudaStream_t stream);

// Launch shape forced by usm_set_schedule_override (0: the library's choice).
struct ScheduleOverride {
    int rows_per_warp, tiles_per_block, k_splits;
};
ScheduleOverride schedule_override();

}  // namespace usm
