// Device-side building blocks shared by the kernels of this library:
// shared-memory barriers (mbarrier), TMA tensor copies, bounded waits and
// bf16 unpacking.  Everything is inline PTX for sm_103a.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "usm.h"

namespace usm {

constexpr unsigned kFullMask = 0xffffffffu;

// Upper bound for any wait on a TMA transfer.  A healthy transfer lands in
// microseconds; after this long the kernel records USM_ERR_TIMEOUT and
// returns instead of spinning forever.
constexpr unsigned long long kWaitLimitNs = 2000000000ull;  // 2 s

__device__ __forceinline__ uint32_t smem_addr(const void* p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ unsigned long long global_timer_ns() {
    unsigned long long t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

// ---------------------------------------------------------------- mbarrier
__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

__device__ __forceinline__ void fence_barrier_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void fence_proxy_async_smem() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(bar), "r"(parity)
        : "memory");
    return ok != 0;
}

// Wait for phase `parity` of the barrier to complete, giving up after
// limit_ns.  Returns false on timeout.
__device__ __forceinline__ bool mbar_wait_bounded(uint32_t bar, uint32_t parity,
                                                  unsigned long long limit_ns) {
    if (mbar_try_wait(bar, parity)) return true;
    const unsigned long long t0 = global_timer_ns();
    while (true) {
#pragma unroll 1
        for (int i = 0; i < 32; ++i)
            if (mbar_try_wait(bar, parity)) return true;
        if (global_timer_ns() - t0 > limit_ns) return false;
    }
}

// ------------------------------------------------------------------- TMA
// 2-D tiled bulk tensor copy global -> shared, completion counted in bytes on
// the barrier.  x is the inner (contiguous) coordinate in elements and must
// be a multiple of 16 bytes / element size; y is the row.
__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap* map, int x, int y,
                                            uint32_t bar) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes "
        "[%0], [%1, {%2, %3}], [%4];" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(bar)
        : "memory");
}

__device__ __forceinline__ void prefetch_tensor_map(const CUtensorMap* map) {
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}

// ------------------------------------------------------------ status word
__device__ __forceinline__ void record_status(int* status, int code) {
    if (status) atomicCAS(status, 0, code);
}

// ------------------------------------------------------------- bf16 bits
// bf16 is the top half of an fp32 bit pattern: widening is exact.
__device__ __forceinline__ uint16_t f32_to_bf16_rne(float x) {
    // Round to nearest, ties to even, on the bit pattern (inputs finite).
    uint32_t u = __float_as_uint(x);
    u += 0x7fffu + ((u >> 16) & 1u);
    return static_cast<uint16_t>(u >> 16);
}

// fp32 += bf16 × bf16: fma.rn.f32.bf16 multiplies the two bf16 values
// exactly and adds in fp32 with one rounding; on sm_103a it issues at the
// full FP32 rate.  Its operands are 16-bit registers: taking them as the low
// or high half of a 32-bit word in C (lo16/hi16) lets the compiler select the
// half for free, where an explicit split inside the asm costs extra
// instructions (measured: 10.6 against 16.2 cycles per warp step).
__device__ __forceinline__ float fma_bf16(uint16_t a, uint16_t b, float c) {
    float d;
    asm("fma.rn.f32.bf16 %0, %1, %2, %3;" : "=f"(d) : "h"(a), "h"(b), "f"(c));
    return d;
}
__device__ __forceinline__ uint16_t lo16(uint32_t w) { return static_cast<uint16_t>(w); }
__device__ __forceinline__ uint16_t hi16(uint32_t w) { return static_cast<uint16_t>(w >> 16); }

// Shared-memory loads by 32-bit shared address.  volatile keeps them after
// the barrier waits that publish the data they read.
__device__ __forceinline__ uint4 lds128(uint32_t addr) {
    uint4 v;
    asm volatile("ld.shared.v4.u32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "r"(addr));
    return v;
}
__device__ __forceinline__ uint2 lds64(uint32_t addr) {
    uint2 v;
    asm volatile("ld.shared.v2.u32 {%0,%1}, [%2];" : "=r"(v.x), "=r"(v.y) : "r"(addr));
    return v;
}
__device__ __forceinline__ uint32_t lds32(uint32_t addr) {
    uint32_t v;
    asm volatile("ld.shared.u32 %0, [%1];" : "=r"(v) : "r"(addr));
    return v;
}
__device__ __forceinline__ uint16_t lds16(uint32_t addr) {
    uint16_t v;
    asm volatile("ld.shared.u16 %0, [%1];" : "=h"(v) : "r"(addr));
    return v;
}

// Row scheduler.  The row swizzle lists rows by decreasing length (inside
// each diagonal block of seg rows); the kernels map swizzled positions to
// (row tile, slot) in a boustrophedon order: tile t of a block takes
// positions t, 2T-1-t, 2T+t, ... (T tiles per block), so every tile gets a
// similar mix of long and short rows, and a tile never spans two blocks.
// The launcher picks T ≥ ceil(seg / slots per tile), so no tile overflows;
// more tiles than that hold fewer rows each (to fill the last wave of CTAs).
// Slots alternate over the warps the same way.  Returns the position in the
// swizzle, or -1 past the block or the matrix.
__device__ __forceinline__ long long sched_pos(int tile, int slot, int T, int seg, int M) {
    const int b = tile / T, t = tile - b * T;  // T: tiles per block
    const long long p = (long long)slot * T + ((slot & 1) ? (T - 1 - t) : t);
    if (p >= seg) return -1;
    const long long m = (long long)b * seg + p;
    return m < M ? m : -1;
}
__device__ __forceinline__ int sched_slot(int i, int warp, int W) {
    return i * W + ((i & 1) ? (W - 1 - warp) : warp);
}

}  // namespace usm
