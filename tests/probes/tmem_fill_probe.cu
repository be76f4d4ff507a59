// Tensor-memory fill-rate probe (sm_103a), one CTA of 16 warps on one SM:
//  A) tcgen05.cp.32x128b.warpx4 (512 B source, replicated to 4 subpartitions)
//     issued by 1, 4 or 16 threads (one per warp), 64 KB per fill;
//  B) tcgen05.cp.128x256b (4 KB source, no replication) issued by 1 or 4 threads,
//     128 KB per fill;
//  C) tcgen05.st.32x32b.x8 from registers by all 16 warps, 256 KB per fill
//     (each subpartition 64 KB), also with the LDS.128 reads of the source.
// Every mbarrier wait is bounded (2 s); the tensor memory is always freed.
// Prints one JSON object per line.
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
__device__ __forceinline__ uint64_t sdesc(uint32_t saddr, uint32_t lbo, uint32_t sbo) {
    uint64_t d = 0;
    d |= (uint64_t)((saddr & 0x3FFFFu) >> 4);
    d |= (uint64_t)((lbo & 0x3FFFFu) >> 4) << 16;
    d |= (uint64_t)((sbo & 0x3FFFFu) >> 4) << 32;
    d |= (uint64_t)1 << 46;
    return d;
}

constexpr int BUF = 128 * 1024;

struct Res {
    int timeouts, mismatches;
    unsigned long long cyc[8];
};

// mode 0/1/2: 32x128b.warpx4 from 1/4/16 issuing threads (64 KB distinct per fill)
// mode 3/4:   128x256b from 1/4 issuing threads (128 KB per fill: 32 instr of 4 KB)
// mode 5:     tcgen05.st.32x32b.x8 by all warps (each subpartition 32 KB: 128 KB per fill)
// mode 6:     LDS.128 x2 + tcgen05.st.32x32b.x8 by all warps (same bytes)
__global__ void __launch_bounds__(512, 1) fill_probe(Res* res, int fills) {
    extern __shared__ __align__(1024) unsigned char buf[];
    __shared__ uint32_t tmem_base;
    __shared__ __align__(8) uint64_t bar[4];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    for (int i = threadIdx.x; i < BUF / 4; i += 512) reinterpret_cast<uint32_t*>(buf)[i] = (uint32_t)i * 2654435761u;
    if (warp == 0) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], 512;" ::"r"(smem_u32(&tmem_base)));
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;");
    }
    if (threadIdx.x < 4) {
        asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(smem_u32(&bar[threadIdx.x])));
    }
    if (threadIdx.x == 0) asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
    __syncthreads();
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
    const uint32_t tb = tmem_base, b0 = smem_u32(buf);
    uint32_t ph[4] = {0, 0, 0, 0};
    uint32_t ph16 = 0;
    int timeouts = 0;
    __shared__ __align__(8) uint64_t bar16[16];
    if (threadIdx.x < 16) asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(smem_u32(&bar16[threadIdx.x])));
    if (threadIdx.x == 0) asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    __syncthreads();
    for (int mode = 0; mode < 7; ++mode) {
        __syncthreads();
        const unsigned long long c0 = clock64();
        for (int f = 0; f < fills; ++f) {
            if (mode <= 2) {
                const int nthr = mode == 0 ? 1 : (mode == 1 ? 4 : 16);
                const int per = 128 / nthr;  // 512-byte blocks per issuing thread
                if (lane == 0 && warp < nthr) {
                    for (int b = warp * per; b < (warp + 1) * per; ++b)
                        asm volatile("tcgen05.cp.cta_group::1.32x128b.warpx4 [%0], %1;"
                                     ::"r"(tb + 4 * b), "l"(sdesc(b0 + 512 * b, 128, 128)) : "memory");
                    const uint32_t bb = nthr == 16 ? smem_u32(&bar16[warp]) : smem_u32(&bar[warp]);
                    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];"
                                 ::"r"(bb) : "memory");
                }
                if (nthr == 16) {
                    if (lane == 0 && !mbar_wait(smem_u32(&bar16[warp]), ph16)) ++timeouts;
                } else {
                    for (int w = 0; w < nthr; ++w)
                        if (!mbar_wait(smem_u32(&bar[w]), ph[w])) ++timeouts;
                }
                if (nthr == 16) ph16 ^= 1;
                else for (int w = 0; w < nthr; ++w) ph[w] ^= 1;
            } else if (mode <= 4) {
                const int nthr = mode == 3 ? 1 : 4;
                const int per = 32 / nthr;  // 4 KB instructions per issuing thread (128 KB)
                if (lane == 0 && warp < nthr) {
                    for (int b = warp * per; b < (warp + 1) * per; ++b)
                        // 128 rows of 32 B: row i first 16 B at 16 i (groups of 8 rows 128 B apart),
                        // second 16 B at +2048; TMEM lanes 0..127, columns 8b..8b+7
                        asm volatile("tcgen05.cp.cta_group::1.128x256b [%0], %1;"
                                     ::"r"(tb + 8 * b), "l"(sdesc(b0 + 4096 * b, 2048, 128)) : "memory");
                    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];"
                                 ::"r"(smem_u32(&bar[warp])) : "memory");
                }
                for (int w = 0; w < nthr; ++w)
                    if (!mbar_wait(smem_u32(&bar[w]), ph[w])) ++timeouts;
                for (int w = 0; w < nthr; ++w) ph[w] ^= 1;
            } else {
                // each warp writes 32 TMEM columns x 8 ... : warp w (subpartition w & 3, quarter w >> 2)
                // stores 16 column-groups of 8: 16 x 32 lanes x 32 B = 16 KB; all 16 warps: 256 KB
                const uint32_t tw = tb + ((uint32_t)(32 * (warp & 3)) << 16) + 128 * (warp >> 2);
                for (int g = 0; g < 16; ++g) {
                    uint32_t v[8];
                    if (mode == 6) {
                        const uint32_t a = b0 + ((g * 16 + warp) % 128) * 1024 + 16 * lane;
                        asm volatile("ld.shared.v4.u32 {%0,%1,%2,%3}, [%4];" : "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3]) : "r"(a));
                        asm volatile("ld.shared.v4.u32 {%0,%1,%2,%3}, [%4];" : "=r"(v[4]), "=r"(v[5]), "=r"(v[6]), "=r"(v[7]) : "r"(a + 512));
                    } else {
#pragma unroll
                        for (int q = 0; q < 8; ++q) v[q] = g * 8 + q + lane;
                    }
                    asm volatile("tcgen05.st.sync.aligned.32x32b.x8.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8};"
                                 ::"r"(tw + 8 * g), "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]),
                                   "r"(v[6]), "r"(v[7]) : "memory");
                }
                asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
            }
            asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
            __syncthreads();
            asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
        }
        if (threadIdx.x == 0) res->cyc[mode] = clock64() - c0;
    }
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
    __syncthreads();
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
    if (warp == 0) asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, 512;" ::"r"(tb));
    if (timeouts) atomicAdd(&res->timeouts, timeouts);
}

int main() {
    CK(cudaSetDevice(0));
    Res* d;
    CK(cudaMalloc(&d, sizeof(Res)));
    CK(cudaMemset(d, 0, sizeof(Res)));
    CK(cudaFuncSetAttribute(fill_probe, cudaFuncAttributeMaxDynamicSharedMemorySize, BUF));
    const int fills = 100;
    fill_probe<<<1, 512, BUF>>>(d, fills);
    CK(cudaGetLastError());
    CK(cudaDeviceSynchronize());
    Res h;
    CK(cudaMemcpy(&h, d, sizeof(Res), cudaMemcpyDeviceToHost));
    const char* names[7] = {"cp32x128b_warpx4_1thr", "cp32x128b_warpx4_4thr", "cp32x128b_warpx4_16thr",
                            "cp128x256b_1thr", "cp128x256b_4thr", "st32x32b_x8_16warps", "lds128_then_st_x8_16warps"};
    // source bytes per fill: modes 0-2: 64 KB (written 4x); 3-4: 128 KB; 5-6: 256 KB
    const double src[7] = {65536, 65536, 65536, 131072, 131072, 262144, 262144};
    const double tm[7] = {262144, 262144, 262144, 131072, 131072, 262144, 262144};
    for (int m = 0; m < 7; ++m)
        printf("{\"probe\": \"%s\", \"cycles_per_fill\": %.0f, \"source_bytes_per_clk\": %.2f, "
               "\"tmem_bytes_written_per_clk\": %.2f}\n", names[m], (double)h.cyc[m] / fills,
               src[m] * fills / (double)h.cyc[m], tm[m] * fills / (double)h.cyc[m]);
    printf("{\"timeouts\": %d}\n", h.timeouts);
    return 0;
}
