// Tensor-memory copy probe (sm_103a), one CTA of 16 warps on one SM.
//
// Checks the layout the SpMM kernel's tensor-memory rows rely on:
// tcgen05.cp.cta_group::1.32x128b.warpx4 from a no-swizzle shared-memory
// descriptor (leading and stride byte offsets 128) puts row i (16 bytes) of
// a 512-byte shared-memory block into lane i of every subpartition, columns
// +0..3.  128 such copies fill all 512 columns; every word of every lane is
// compared with the shared-memory source (mismatches are counted).  Also
// times those 64 KB fills (one issuing thread) and tcgen05.ld 32x32b at
// random columns: x2/x4/x8/x16 with four loads per wait, x8 with a wait
// after every load.
//
// Every mbarrier wait is bounded (2 s via %globaltimer); the tensor memory is
// always freed before the CTA exits.  Prints one JSON object per line.
#include <cstdio>
#include <cstdint>
#include <cstdlib>
#include <cuda_runtime.h>

#define CK(x) do { cudaError_t e_ = (x); if (e_ != cudaSuccess) { \
    fprintf(stderr, "%s:%d %s\n", __FILE__, __LINE__, cudaGetErrorString(e_)); exit(1); } } while (0)

__device__ __forceinline__ uint32_t smem_u32(const void* p) { return (uint32_t)__cvta_generic_to_shared(p); }
__device__ __forceinline__ unsigned long long gtime() {
    unsigned long long t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity) {
    const unsigned long long t0 = gtime();
    while (true) {
        uint32_t ok;
        asm volatile("{\n\t.reg .pred p;\n\tmbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
                     "selp.u32 %0, 1, 0, p;\n\t}" : "=r"(ok) : "r"(bar), "r"(parity) : "memory");
        if (ok) return true;
        if (gtime() - t0 > 2000000000ull) return false;
    }
}

// Shared-memory descriptor: start >> 4 (bits 0-13), LBO >> 4 (16-29),
// SBO >> 4 (32-45), fixed 0b001 at bits 46-48, no swizzle (61-63 = 0).
__device__ __forceinline__ uint64_t sdesc(uint32_t saddr, uint32_t lbo, uint32_t sbo) {
    uint64_t d = 0;
    d |= (uint64_t)((saddr & 0x3FFFFu) >> 4);
    d |= (uint64_t)((lbo & 0x3FFFFu) >> 4) << 16;
    d |= (uint64_t)((sbo & 0x3FFFFu) >> 4) << 32;
    d |= (uint64_t)1 << 46;
    return d;
}

constexpr int BUF = 64 * 1024;

struct Res {
    int mismatches, timeouts;
    uint32_t first_bad[8][4];  // lane, col, got, want
    unsigned long long fill_cycles, fills;
    unsigned long long ld_cycles[5];
};

__global__ void __launch_bounds__(512, 1) cp_probe(Res* res, int fills) {
    extern __shared__ __align__(1024) unsigned char buf[];
    __shared__ uint32_t tmem_base;
    __shared__ __align__(8) uint64_t bar;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    for (int i = threadIdx.x; i < BUF / 4; i += 512) reinterpret_cast<uint32_t*>(buf)[i] = (uint32_t)i * 2654435761u ^ 0x5bd1e995u;
    if (warp == 0) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], 512;" ::"r"(smem_u32(&tmem_base)));
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;");
    }
    if (threadIdx.x == 0) {
        asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(smem_u32(&bar)));
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");  // generic smem writes -> async proxy
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
    __syncthreads();
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
    const uint32_t tb = tmem_base;
    const uint32_t b0 = smem_u32(buf);
    uint32_t phase = 0;
    int timeouts = 0;
    unsigned long long fill_cyc = 0;
    for (int f = 0; f < fills; ++f) {
        const unsigned long long c0 = clock64();
        if (threadIdx.x == 0) {
            for (int b = 0; b < 128; ++b) {
                const uint64_t d = sdesc(b0 + 512 * b, 128, 128);
                asm volatile("tcgen05.cp.cta_group::1.32x128b.warpx4 [%0], %1;" ::"r"(tb + 4 * b), "l"(d) : "memory");
            }
            asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];"
                         ::"r"(smem_u32(&bar)) : "memory");
        }
        if (!mbar_wait(smem_u32(&bar), phase)) ++timeouts;
        phase ^= 1;
        asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
        fill_cyc += clock64() - c0;
        __syncthreads();
    }
    // check every TMEM word of this warp's subpartition
    int bad = 0;
    for (int c = 0; c < 512; c += 8) {
        uint32_t v[8];
        asm volatile("tcgen05.ld.sync.aligned.32x32b.x8.b32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8];\n\t"
                     "tcgen05.wait::ld.sync.aligned;"
                     : "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3]), "=r"(v[4]), "=r"(v[5]), "=r"(v[6]), "=r"(v[7])
                     : "r"(tb + ((uint32_t)(32 * (warp & 3)) << 16) + c));
        for (int j = 0; j < 8; ++j) {
            const int col = c + j, blk = col / 4, w = col % 4;
            const uint32_t want = reinterpret_cast<const uint32_t*>(buf)[(512 * blk + 16 * lane + 4 * w) / 4];
            if (v[j] != want) {
                ++bad;
                const int k = atomicAdd(&res->mismatches, 1);
                if (k < 8) {
                    res->first_bad[k][0] = 32 * (warp & 3) + lane;
                    res->first_bad[k][1] = col;
                    res->first_bad[k][2] = v[j];
                    res->first_bad[k][3] = want;
                }
            }
        }
    }
    (void)bad;
    // tcgen05.ld rates at random columns: shapes x2, x4, x8, x16 (4 loads per
    // wait) and x8 with a wait after every load
    uint32_t x = 0, seed = 99u + warp;
    const uint32_t tw = tb + ((uint32_t)(32 * (warp & 3)) << 16);
    const int iters = 20000;
    for (int mode = 0; mode < 5; ++mode) {
        __syncthreads();
        const unsigned long long c0 = clock64();
        for (int it = 0; it < iters; ++it) {
            seed = seed * 1664525u + 1013904223u;
            const uint32_t col = ((seed >> 8) & 511u) & ~63u;
            if (mode == 0) {
                uint32_t a[8];
                asm volatile("tcgen05.ld.sync.aligned.32x32b.x2.b32 {%0,%1}, [%8];\n\t"
                             "tcgen05.ld.sync.aligned.32x32b.x2.b32 {%2,%3}, [%9];\n\t"
                             "tcgen05.ld.sync.aligned.32x32b.x2.b32 {%4,%5}, [%10];\n\t"
                             "tcgen05.ld.sync.aligned.32x32b.x2.b32 {%6,%7}, [%11];\n\t"
                             "tcgen05.wait::ld.sync.aligned;"
                             : "=r"(a[0]), "=r"(a[1]), "=r"(a[2]), "=r"(a[3]), "=r"(a[4]), "=r"(a[5]), "=r"(a[6]), "=r"(a[7])
                             : "r"(tw + col), "r"(tw + col + 16), "r"(tw + col + 32), "r"(tw + col + 48));
                for (int q = 0; q < 8; ++q) x ^= a[q];
            } else if (mode == 1) {
                uint32_t a[16];
                asm volatile("tcgen05.ld.sync.aligned.32x32b.x4.b32 {%0,%1,%2,%3}, [%16];\n\t"
                             "tcgen05.ld.sync.aligned.32x32b.x4.b32 {%4,%5,%6,%7}, [%17];\n\t"
                             "tcgen05.ld.sync.aligned.32x32b.x4.b32 {%8,%9,%10,%11}, [%18];\n\t"
                             "tcgen05.ld.sync.aligned.32x32b.x4.b32 {%12,%13,%14,%15}, [%19];\n\t"
                             "tcgen05.wait::ld.sync.aligned;"
                             : "=r"(a[0]), "=r"(a[1]), "=r"(a[2]), "=r"(a[3]), "=r"(a[4]), "=r"(a[5]), "=r"(a[6]), "=r"(a[7]),
                               "=r"(a[8]), "=r"(a[9]), "=r"(a[10]), "=r"(a[11]), "=r"(a[12]), "=r"(a[13]), "=r"(a[14]), "=r"(a[15])
                             : "r"(tw + col), "r"(tw + col + 16), "r"(tw + col + 32), "r"(tw + col + 48));
                for (int q = 0; q < 16; ++q) x ^= a[q];
            } else if (mode == 2 || mode == 4) {
                uint32_t a[32];
                if (mode == 2) {
                    asm volatile("tcgen05.ld.sync.aligned.32x32b.x8.b32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%32];\n\t"
                                 "tcgen05.ld.sync.aligned.32x32b.x8.b32 {%8,%9,%10,%11,%12,%13,%14,%15}, [%33];\n\t"
                                 "tcgen05.ld.sync.aligned.32x32b.x8.b32 {%16,%17,%18,%19,%20,%21,%22,%23}, [%34];\n\t"
                                 "tcgen05.ld.sync.aligned.32x32b.x8.b32 {%24,%25,%26,%27,%28,%29,%30,%31}, [%35];\n\t"
                                 "tcgen05.wait::ld.sync.aligned;"
                                 : "=r"(a[0]), "=r"(a[1]), "=r"(a[2]), "=r"(a[3]), "=r"(a[4]), "=r"(a[5]), "=r"(a[6]), "=r"(a[7]),
                                   "=r"(a[8]), "=r"(a[9]), "=r"(a[10]), "=r"(a[11]), "=r"(a[12]), "=r"(a[13]), "=r"(a[14]), "=r"(a[15]),
                                   "=r"(a[16]), "=r"(a[17]), "=r"(a[18]), "=r"(a[19]), "=r"(a[20]), "=r"(a[21]), "=r"(a[22]), "=r"(a[23]),
                                   "=r"(a[24]), "=r"(a[25]), "=r"(a[26]), "=r"(a[27]), "=r"(a[28]), "=r"(a[29]), "=r"(a[30]), "=r"(a[31])
                                 : "r"(tw + col), "r"(tw + col + 16), "r"(tw + col + 32), "r"(tw + col + 48));
                } else {
                    for (int q = 0; q < 4; ++q)
                        asm volatile("tcgen05.ld.sync.aligned.32x32b.x8.b32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8];\n\t"
                                     "tcgen05.wait::ld.sync.aligned;"
                                     : "=r"(a[8 * q]), "=r"(a[8 * q + 1]), "=r"(a[8 * q + 2]), "=r"(a[8 * q + 3]),
                                       "=r"(a[8 * q + 4]), "=r"(a[8 * q + 5]), "=r"(a[8 * q + 6]), "=r"(a[8 * q + 7])
                                     : "r"(tw + col + 16 * q));
                }
                for (int q = 0; q < 32; ++q) x ^= a[q];
            } else {
                uint32_t a[64];
                asm volatile("tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%64];\n\t"
                             "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%65];\n\t"
                             "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%32,%33,%34,%35,%36,%37,%38,%39,%40,%41,%42,%43,%44,%45,%46,%47}, [%66];\n\t"
                             "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%48,%49,%50,%51,%52,%53,%54,%55,%56,%57,%58,%59,%60,%61,%62,%63}, [%67];\n\t"
                             "tcgen05.wait::ld.sync.aligned;"
                             : "=r"(a[0]), "=r"(a[1]), "=r"(a[2]), "=r"(a[3]), "=r"(a[4]), "=r"(a[5]), "=r"(a[6]), "=r"(a[7]),
                               "=r"(a[8]), "=r"(a[9]), "=r"(a[10]), "=r"(a[11]), "=r"(a[12]), "=r"(a[13]), "=r"(a[14]), "=r"(a[15]),
                               "=r"(a[16]), "=r"(a[17]), "=r"(a[18]), "=r"(a[19]), "=r"(a[20]), "=r"(a[21]), "=r"(a[22]), "=r"(a[23]),
                               "=r"(a[24]), "=r"(a[25]), "=r"(a[26]), "=r"(a[27]), "=r"(a[28]), "=r"(a[29]), "=r"(a[30]), "=r"(a[31]),
                               "=r"(a[32]), "=r"(a[33]), "=r"(a[34]), "=r"(a[35]), "=r"(a[36]), "=r"(a[37]), "=r"(a[38]), "=r"(a[39]),
                               "=r"(a[40]), "=r"(a[41]), "=r"(a[42]), "=r"(a[43]), "=r"(a[44]), "=r"(a[45]), "=r"(a[46]), "=r"(a[47]),
                               "=r"(a[48]), "=r"(a[49]), "=r"(a[50]), "=r"(a[51]), "=r"(a[52]), "=r"(a[53]), "=r"(a[54]), "=r"(a[55]),
                               "=r"(a[56]), "=r"(a[57]), "=r"(a[58]), "=r"(a[59]), "=r"(a[60]), "=r"(a[61]), "=r"(a[62]), "=r"(a[63])
                             : "r"(tw + col), "r"(tw + col + 16), "r"(tw + col + 32), "r"(tw + col + 48));
                for (int q = 0; q < 64; ++q) x ^= a[q];
            }
        }
        __syncthreads();
        if (threadIdx.x == 0) res->ld_cycles[mode] = clock64() - c0;
    }
    if (x == 0x12345u) res->mismatches += 1000000;
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
    __syncthreads();
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
    if (warp == 0) asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, 512;" ::"r"(tb));
    if (threadIdx.x == 0) {
        res->timeouts = timeouts;
        res->fill_cycles = fill_cyc;
        res->fills = fills;
    }
}

int main() {
    CK(cudaSetDevice(0));
    Res* d;
    CK(cudaMalloc(&d, sizeof(Res)));
    CK(cudaMemset(d, 0, sizeof(Res)));
    CK(cudaFuncSetAttribute(cp_probe, cudaFuncAttributeMaxDynamicSharedMemorySize, BUF));
    cp_probe<<<1, 512, BUF>>>(d, 200);
    CK(cudaGetLastError());
    CK(cudaDeviceSynchronize());
    Res h;
    CK(cudaMemcpy(&h, d, sizeof(Res), cudaMemcpyDeviceToHost));
    printf("{\"probe\": \"tcgen05_cp_32x128b_warpx4\", \"mismatches\": %d, \"checked_words\": %d, \"timeouts\": %d, "
           "\"fill_bytes\": 65536, \"cycles_per_fill\": %.1f, \"bytes_per_clk\": %.2f}\n",
           h.mismatches, 128 * 512, h.timeouts, (double)h.fill_cycles / h.fills,
           65536.0 * h.fills / (double)h.fill_cycles);
    for (int k = 0; k < 8 && k < h.mismatches; ++k)
        printf("{\"bad\": [%u, %u, \"0x%08x\", \"0x%08x\"]}\n", h.first_bad[k][0], h.first_bad[k][1], h.first_bad[k][2],
               h.first_bad[k][3]);
    // one CTA, 16 warps: per mode iters x 4 loads x (32 lanes x 4 B x N) per warp
    const char* names[5] = {"x2_4perwait", "x4_4perwait", "x8_4perwait", "x16_4perwait", "x8_waiteach"};
    const int n[5] = {2, 4, 8, 16, 8};
    for (int m = 0; m < 5; ++m)
        printf("{\"probe\": \"tcgen05_ld_32x32b_%s\", \"bytes_per_clk_sm_16warps\": %.2f}\n", names[m],
               20000.0 * 16 * 4 * 128 * n[m] / (double)h.ld_cycles[m]);
    return 0;
}
