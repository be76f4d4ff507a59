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

// Rows of one TMA box for a chunk of kc staged rows: the largest divisor of kc
// that is at most 256 (a box dimension's limit), so whole boxes tile the chunk.
constexpr int tma_box_rows(int kc) {
    for (int b = kc < 256 ? kc : 256; b > 1; --b)
        if (kc % b == 0) return b;
    return 1;
}

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

// ----------------------------------------------------------- tensor memory
// Tensor memory (TMEM, 128 lanes x 512 columns of 32 bits per SM) as a
// second store for staged dense rows: tcgen05.ld reads it through its own
// path, beside the shared-memory loads.  A warp may read only the 32 lanes
// of its subpartition (warp id mod 4).  Addresses: lane << 16 | column.

// Allocate `cols` columns (a power of two >= 32) for the CTA; one full warp
// executes it and the base address lands in shared memory at `dst`.
__device__ __forceinline__ void tmem_alloc(uint32_t dst, uint32_t cols) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(dst), "r"(cols) : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t base, uint32_t cols) {
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(base), "r"(cols) : "memory");
}
__device__ __forceinline__ void tmem_fence_before_sync() {
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tmem_fence_after_sync() {
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// Shared-memory matrix descriptor, no swizzle: start, leading- and
// stride-dimension byte offsets (each >> 4), fixed 0b001 at bits 46-48.
__device__ __forceinline__ uint64_t smem_desc(uint32_t saddr, uint32_t lbo, uint32_t sbo) {
    return (uint64_t)((saddr & 0x3FFFFu) >> 4) | ((uint64_t)((lbo & 0x3FFFFu) >> 4) << 16) |
           ((uint64_t)((sbo & 0x3FFFFu) >> 4) << 32) | ((uint64_t)1 << 46);
}

// Copy 512 contiguous bytes of shared memory at `saddr` (32 rows of 16
// bytes) into TMEM columns col..col+3 of lanes 0..31 of every subpartition:
// row i lands in lane i (measured on GB300: bit-exact for every word).
// Asynchronous; issued by one thread.
__device__ __forceinline__ void tmem_cp_512b_x4(uint32_t tcol, uint32_t saddr) {
    asm volatile("tcgen05.cp.cta_group::1.32x128b.warpx4 [%0], %1;" ::"r"(tcol), "l"(smem_desc(saddr, 128, 128))
                 : "memory");
}
// Arrive once on the barrier when every tcgen05 copy this thread issued so
// far has completed.
__device__ __forceinline__ void tmem_commit(uint32_t bar) {
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar) : "memory");
}

// Eight 32-bit columns of this thread's TMEM lane, starting at taddr.  The
// wait is in the same statement, so the results are complete when used.
__device__ __forceinline__ void tmem_ld8(uint32_t taddr, uint32_t (&w)[8]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x8.b32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8];\n\t"
        "tcgen05.wait::ld.sync.aligned;"
        : "=r"(w[0]), "=r"(w[1]), "=r"(w[2]), "=r"(w[3]), "=r"(w[4]), "=r"(w[5]), "=r"(w[6]), "=r"(w[7])
        : "r"(taddr)
        : "memory");
}
// Four loads of four columns (16 bytes a lane) behind one wait.
__device__ __forceinline__ void tmem_ld4x4(uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3, uint4& w0, uint4& w1,
                                           uint4& w2, uint4& w3) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x4.b32 {%0,%1,%2,%3}, [%16];\n\t"
        "tcgen05.ld.sync.aligned.32x32b.x4.b32 {%4,%5,%6,%7}, [%17];\n\t"
        "tcgen05.ld.sync.aligned.32x32b.x4.b32 {%8,%9,%10,%11}, [%18];\n\t"
        "tcgen05.ld.sync.aligned.32x32b.x4.b32 {%12,%13,%14,%15}, [%19];\n\t"
        "tcgen05.wait::ld.sync.aligned;"
        : "=r"(w0.x), "=r"(w0.y), "=r"(w0.z), "=r"(w0.w), "=r"(w1.x), "=r"(w1.y), "=r"(w1.z), "=r"(w1.w),
          "=r"(w2.x), "=r"(w2.y), "=r"(w2.z), "=r"(w2.w), "=r"(w3.x), "=r"(w3.y), "=r"(w3.z), "=r"(w3.w)
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3)
        : "memory");
}
__device__ __forceinline__ uint4 tmem_ld4(uint32_t a) {
    uint4 w;
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x4.b32 {%0,%1,%2,%3}, [%4];\n\t"
        "tcgen05.wait::ld.sync.aligned;"
        : "=r"(w.x), "=r"(w.y), "=r"(w.z), "=r"(w.w)
        : "r"(a)
        : "memory");
    return w;
}
// Two loads of eight columns issued without a wait (results are not ready
// until tmem_wait_tied).  The accumulators c are tied in so that FMAs on
// them that come after this call in program order stay after the loads.
__device__ __forceinline__ void tmem_ld8x2_nowait(uint32_t a0, uint32_t a1, uint32_t (&w0)[8], uint32_t (&w1)[8],
                                                  float (&c)[8]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x8.b32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%24];\n\t"
        "tcgen05.ld.sync.aligned.32x32b.x8.b32 {%8,%9,%10,%11,%12,%13,%14,%15}, [%25];"
        : "=r"(w0[0]), "=r"(w0[1]), "=r"(w0[2]), "=r"(w0[3]), "=r"(w0[4]), "=r"(w0[5]), "=r"(w0[6]), "=r"(w0[7]),
          "=r"(w1[0]), "=r"(w1[1]), "=r"(w1[2]), "=r"(w1[3]), "=r"(w1[4]), "=r"(w1[5]), "=r"(w1[6]), "=r"(w1[7]),
          "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3]), "+f"(c[4]), "+f"(c[5]), "+f"(c[6]), "+f"(c[7])
        : "r"(a0), "r"(a1)
        : "memory");
}
// Wait for every tcgen05.ld this thread issued.  The loaded registers are
// tied in (their uses stay after the wait) and so are the accumulators (the
// FMAs issued between the loads and this wait stay before it).
__device__ __forceinline__ void tmem_wait_tied(uint32_t (&w0)[8], uint32_t (&w1)[8], float (&c)[8]) {
    asm volatile("tcgen05.wait::ld.sync.aligned;"
                 : "+r"(w0[0]), "+r"(w0[1]), "+r"(w0[2]), "+r"(w0[3]), "+r"(w0[4]), "+r"(w0[5]), "+r"(w0[6]),
                   "+r"(w0[7]), "+r"(w1[0]), "+r"(w1[1]), "+r"(w1[2]), "+r"(w1[3]), "+r"(w1[4]), "+r"(w1[5]),
                   "+r"(w1[6]), "+r"(w1[7]), "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3]), "+f"(c[4]), "+f"(c[5]),
                   "+f"(c[6]), "+f"(c[7])
                 :
                 : "memory");
}
// Four such loads in flight before one wait.
__device__ __forceinline__ void tmem_ld8x4(uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3, uint32_t (&w0)[8],
                                           uint32_t (&w1)[8], uint32_t (&w2)[8], uint32_t (&w3)[8]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x8.b32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%32];\n\t"
        "tcgen05.ld.sync.aligned.32x32b.x8.b32 {%8,%9,%10,%11,%12,%13,%14,%15}, [%33];\n\t"
        "tcgen05.ld.sync.aligned.32x32b.x8.b32 {%16,%17,%18,%19,%20,%21,%22,%23}, [%34];\n\t"
        "tcgen05.ld.sync.aligned.32x32b.x8.b32 {%24,%25,%26,%27,%28,%29,%30,%31}, [%35];\n\t"
        "tcgen05.wait::ld.sync.aligned;"
        : "=r"(w0[0]), "=r"(w0[1]), "=r"(w0[2]), "=r"(w0[3]), "=r"(w0[4]), "=r"(w0[5]), "=r"(w0[6]), "=r"(w0[7]),
          "=r"(w1[0]), "=r"(w1[1]), "=r"(w1[2]), "=r"(w1[3]), "=r"(w1[4]), "=r"(w1[5]), "=r"(w1[6]), "=r"(w1[7]),
          "=r"(w2[0]), "=r"(w2[1]), "=r"(w2[2]), "=r"(w2[3]), "=r"(w2[4]), "=r"(w2[5]), "=r"(w2[6]), "=r"(w2[7]),
          "=r"(w3[0]), "=r"(w3[1]), "=r"(w3[2]), "=r"(w3[3]), "=r"(w3[4]), "=r"(w3[5]), "=r"(w3[6]), "=r"(w3[7])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3)
        : "memory");
}

// ------------------------------------------------------------ status word
__device__ __forceinline__ void record_status(int* status, int code) {
    if (status) atomicCAS(status, 0, code);
}

// ------------------------------------------------------------- bf16 bits
// bf16 is the top half of an fp32 bit pattern: widening is exact.
__device__ __forceinline__ uint16_t f32_to_bf16_rne(float x) {
    // Round to nearest, ties to even (the hardware conversion).
    uint16_t h;
    asm("cvt.rn.bf16.f32 %0, %1;" : "=h"(h) : "f"(x));
    return h;
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

// Drop the 128-byte line at p (128-byte aligned) from L2 without writing it
// back: its contents become undefined.  For scratch data that is dead.
__device__ __forceinline__ void l2_discard_line(const void* p) {
    asm volatile("discard.global.L2 [%0], 128;" ::"l"(p) : "memory");
}

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

// Softmax over the stored entries of one CSR row, s[b..e): the maximum m and
// the reciprocal rz of z = Σ exp(s - m), computed by the 32 lanes of a warp
// (lane i takes entries b+i, b+i+32, ...; the lanes' results are combined by
// a butterfly).  A probability is softmax_prob(s, m, rz) = exp(s - m)·rz.
// Both kernels that need softmax probabilities use these two routines, so a
// probability has the same bits wherever it is formed.  The exponential is
// CUDA's fast __expf (documented error at most 2 + 1.17·|x| ulp; x = s - m
// <= 0, and terms with x below about -20 are under 2^-28 of the largest).
// Rounding: a lane's about n/32 terms go into four partial sums (about n/128
// additions each), joined in a 2-level tree, then the butterfly's 5 levels,
// the reciprocal and the product: about n/128 + 9 fp32 roundings on top of
// the exponentials' error.
__device__ __forceinline__ void row_softmax_stats(const float* __restrict__ s, int b, int e, int lane, float& m,
                                                  float& rz) {
    // Eight loads in flight a lane (the scores come from L2): the maximum,
    // then the sum in four interleaved partial sums.
    constexpr int U = 8;
    m = -3.402823466e38f;
    int p = b + lane;
    for (; p + (U - 1) * 32 < e; p += U * 32) {
        float v[U];
#pragma unroll
        for (int u = 0; u < U; ++u) v[u] = __ldg(s + p + 32 * u);
#pragma unroll
        for (int u = 0; u < U; ++u) m = fmaxf(m, v[u]);
    }
    for (; p < e; p += 32) m = fmaxf(m, __ldg(s + p));
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(kFullMask, m, o));
    float z[4] = {0.f, 0.f, 0.f, 0.f};
    p = b + lane;
    for (; p + (U - 1) * 32 < e; p += U * 32) {
        float v[U];
#pragma unroll
        for (int u = 0; u < U; ++u) v[u] = __ldg(s + p + 32 * u);
#pragma unroll
        for (int u = 0; u < U; ++u) z[u & 3] += __expf(v[u] - m);
    }
    for (int u = 0; p < e; p += 32, ++u) z[u & 3] += __expf(__ldg(s + p) - m);
    float t = (z[0] + z[1]) + (z[2] + z[3]);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) t += __shfl_xor_sync(kFullMask, t, o);
    rz = 1.f / t;
}
__device__ __forceinline__ float softmax_prob(float s, float m, float rz) { return __expf(s - m) * rz; }

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
