// csr_sddmm_static_scratch: csr_sddmm for callers that cannot allocate
// device memory.
//
// csr_sddmm needs scratch memory whenever D spans more than one column
// strip (the per-strip partial sums).  Some callers cannot provide it: code
// that runs where no allocator is reachable (a plugin handed only raw
// pointers by its host framework, a real-time loop whose memory was fixed at
// start-up, an embedding that forbids cudaMalloc after initialisation).  This
// entry point takes its scratch from one fixed array in the library's own
// device image instead, so it allocates nothing on any call.
//
// The array below is sized kStaticScratchBytes (32 MiB).  It is reserved on a
// device when this file's module is loaded there: CUDA loads modules lazily,
// so that happens at the first call on the device (the address lookup
// below), and the 32 MiB stay reserved until the context ends.  In host code
// the array's name is only a host-side stand-in for the symbol, never a
// device address: the device address is looked up with cudaGetSymbolAddress
// (with that device current) and passed to the kernels; it is looked up again
// after a device reset or in a new context.
#include "usm_device.cuh"
#include "usm_internal.h"

namespace {

constexpr size_t kStaticScratchBytes = size_t(32) << 20;  // 32 MiB

static __device__ __align__(256) float g_sddmm_static_scratch[kStaticScratchBytes / sizeof(float)];

usm::SymbolAddressCache g_scratch_cache(&g_sddmm_static_scratch);

}  // namespace

extern "C" int csr_sddmm_static_scratch(int M, int K, int D, int nnz, const int* row_offsets,
                                        const int* col_indices, const int* row_swizzle, int seg_rows,
                                        const void* X, int ldx, const void* Y, int ldy, void* out,
                                        usm_dtype in_dtype, usm_dtype out_dtype, void* stream) {
    const size_t need = csr_sddmm_workspace_bytes(M, K, D, nnz, in_dtype);
    if (need > kStaticScratchBytes) return USM_ERR_UNSUPPORTED;
    void* scratch = nullptr;
    if (need > 0) {
        scratch = g_scratch_cache.get();
        if (scratch == nullptr) return USM_ERR_CUDA;
    }
    // On a valid CSR every strip writes its partial for every nonzero before
    // the strip sum reads it, so nothing an earlier call left in the array is
    // read and nothing needs clearing.
    return csr_sddmm(M, K, D, nnz, row_offsets, col_indices, row_swizzle, seg_rows, X, ldx, Y, ldy, out, in_dtype,
                     out_dtype, scratch, need > 0 ? kStaticScratchBytes : 0, stream);
}
