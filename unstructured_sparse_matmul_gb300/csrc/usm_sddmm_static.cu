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
// The array below is sized kStaticScratchBytes (32 MiB).  Every GPU that
// loads this library keeps those 32 MiB until the process exits.  In host
// code the array's name is only a host-side stand-in for the symbol, never a
// device address: the device address is looked up once per device with
// cudaGetSymbolAddress (with that device current) and passed to the kernels.
#include <atomic>

#include "usm_device.cuh"
#include "usm_internal.h"

namespace {

constexpr size_t kStaticScratchBytes = size_t(32) << 20;  // 32 MiB

static __device__ __align__(256) float g_sddmm_static_scratch[kStaticScratchBytes / sizeof(float)];

constexpr int kMaxDevices = 64;
std::atomic<void*> g_scratch_addr[kMaxDevices];

// Device address of the scratch array on the current device.  The first
// call on a device resolves it; later calls reuse it.
int scratch_for_current_device(void** out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return USM_ERR_CUDA;
    if (dev < 0 || dev >= kMaxDevices) return USM_ERR_UNSUPPORTED;
    void* p = g_scratch_addr[dev].load(std::memory_order_acquire);
    if (p == nullptr) {
        const cudaError_t err = cudaGetSymbolAddress(&p, g_sddmm_static_scratch);
        if (err != cudaSuccess || p == nullptr) return USM_ERR_CUDA;
        g_scratch_addr[dev].store(p, std::memory_order_release);
    }
    *out = p;
    return USM_OK;
}

}  // namespace

extern "C" int csr_sddmm_static_scratch(int M, int K, int D, int nnz, const int* row_offsets,
                                        const int* col_indices, const int* row_swizzle, int seg_rows,
                                        const void* X, int ldx, const void* Y, int ldy, void* out,
                                        usm_dtype in_dtype, usm_dtype out_dtype, void* stream) {
    const size_t need = csr_sddmm_workspace_bytes(M, K, D, nnz, in_dtype);
    if (need > kStaticScratchBytes) return USM_ERR_UNSUPPORTED;
    void* scratch = nullptr;
    if (need > 0) {
        const int st = scratch_for_current_device(&scratch);
        if (st != USM_OK) return st;
    }
    // Every strip writes its partial for every nonzero before the strip sum
    // reads it, so nothing left in the array by an earlier call is ever read:
    // no clearing is needed.
    return csr_sddmm(M, K, D, nnz, row_offsets, col_indices, row_swizzle, seg_rows, X, ldx, Y, ldy, out, in_dtype,
                     out_dtype, scratch, need > 0 ? kStaticScratchBytes : 0, stream);
}
