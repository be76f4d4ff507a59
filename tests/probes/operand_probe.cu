// Operand-delivery probes for GB300 (sm_103a): shared-memory load bandwidth
// at random staged rows (LDS.32/64/128), FP32 FMA rates (scalar fma.rn.f32,
// fma.rn.f32x2, fma.rn.f32.bf16) and tensor-memory loads (tcgen05.ld
// 32x32b.x4 at random columns, four loads per wait), alone and mixed with
// LDS.128 in one warp.  `operand_probe t` runs the tensor-memory probes too.
// Prints one JSON object per line.
//
// One CTA of 512 threads per SM (200 KB of dynamic shared memory forces it),
// grid = SM count.  Each CTA times itself with clock64(); bytes (or flops)
// per clock per SM = the CTA's work / its cycles, independent of the clock
// frequency.  CUDA events give the wall time too.
#include <cstdio>
#include <cstdint>
#include <cstdlib>
#include <cuda_runtime.h>

#define CK(x) do { cudaError_t e_ = (x); if (e_ != cudaSuccess) { \
    fprintf(stderr, "%s:%d %s\n", __FILE__, __LINE__, cudaGetErrorString(e_)); exit(1); } } while (0)

constexpr int THREADS = 512;
constexpr int SMEM = 200 * 1024;
constexpr int ROWS = 192;      // staged rows of 1 KB
constexpr int PITCH = 1024;

__device__ __forceinline__ uint32_t smem_u32(const void* p) { return (uint32_t)__cvta_generic_to_shared(p); }

// ---------------------------------------------------------------- LDS probes
// Each warp loads from random staged rows: row r (warp-uniform, from an LCG),
// lanes cover contiguous bytes of the row (conflict-free).  8 loads per
// iteration at rows r, r+1, ..., r+7 (r < ROWS - 8).
template <int BYTES>
__global__ void __launch_bounds__(THREADS, 1) lds_probe(int iters, unsigned long long* cycles, uint32_t* sink) {
    extern __shared__ __align__(1024) unsigned char smem[];
    for (int i = threadIdx.x; i < ROWS * PITCH / 4; i += THREADS) reinterpret_cast<uint32_t*>(smem)[i] = i * 2654435761u;
    __syncthreads();
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const uint32_t base = smem_u32(smem) + lane * BYTES;
    uint32_t x = 0, seed = 12345u + warp * 7919u + blockIdx.x;
    __syncthreads();
    const unsigned long long t0 = clock64();
#pragma unroll 1
    for (int it = 0; it < iters; ++it) {
        seed = seed * 1664525u + 1013904223u;
        const uint32_t r = (seed >> 8) % (ROWS - 8);
        const uint32_t a = base + r * PITCH;
#pragma unroll
        for (int k = 0; k < 8; ++k) {
            if constexpr (BYTES == 4) {
                uint32_t v;
                asm volatile("ld.shared.u32 %0, [%1];" : "=r"(v) : "r"(a + k * PITCH));
                x ^= v;
            } else if constexpr (BYTES == 8) {
                uint32_t v0, v1;
                asm volatile("ld.shared.v2.u32 {%0,%1}, [%2];" : "=r"(v0), "=r"(v1) : "r"(a + k * PITCH));
                x ^= v0 ^ v1;
            } else {
                uint32_t v0, v1, v2, v3;
                asm volatile("ld.shared.v4.u32 {%0,%1,%2,%3}, [%4];"
                             : "=r"(v0), "=r"(v1), "=r"(v2), "=r"(v3) : "r"(a + k * PITCH));
                x ^= v0 ^ v1 ^ v2 ^ v3;
            }
        }
    }
    __syncthreads();
    const unsigned long long t1 = clock64();
    if (threadIdx.x == 0) cycles[blockIdx.x] = t1 - t0;
    if (x == 0x9e3779b9u) sink[0] = x;
}

// ---------------------------------------------------------------- FMA probes
// 16 independent accumulator chains (fp32) per thread; MODE 0: scalar
// fma.rn.f32, 1: fma.rn.f32x2 (two lanes of work per instruction), 2:
// fma.rn.f32.bf16 (bf16 operands, fp32 accumulate).
template <int MODE>
__global__ void __launch_bounds__(THREADS, 1) fma_probe(int iters, float seedf, unsigned long long* cycles, float* sink) {
    float acc[16];
#pragma unroll
    for (int i = 0; i < 16; ++i) acc[i] = seedf * (i + 1) + threadIdx.x;
    const float b = seedf * 0.5f, c = 1.0f - seedf;
    const uint16_t hb = (uint16_t)(__float_as_uint(b) >> 16), hc = (uint16_t)(__float_as_uint(c) >> 16);
    __syncthreads();
    const unsigned long long t0 = clock64();
#pragma unroll 1
    for (int it = 0; it < iters; ++it) {
#pragma unroll
        for (int rep = 0; rep < 4; ++rep) {
            if constexpr (MODE == 0) {
#pragma unroll
                for (int i = 0; i < 16; ++i) asm volatile("fma.rn.f32 %0, %0, %1, %2;" : "+f"(acc[i]) : "f"(b), "f"(c));
            } else if constexpr (MODE == 1) {
#pragma unroll
                for (int i = 0; i < 16; i += 2) {
                    float2 a2 = make_float2(acc[i], acc[i + 1]);
                    a2 = __ffma2_rn(a2, make_float2(b, b), make_float2(c, c));
                    acc[i] = a2.x;
                    acc[i + 1] = a2.y;
                }
            } else {
#pragma unroll
                for (int i = 0; i < 16; ++i)
                    asm volatile("fma.rn.f32.bf16 %0, %1, %2, %0;" : "+f"(acc[i]) : "h"(hb), "h"(hc));
            }
        }
    }
    __syncthreads();
    const unsigned long long t1 = clock64();
    if (threadIdx.x == 0) cycles[blockIdx.x] = t1 - t0;
    float s = 0.f;
#pragma unroll
    for (int i = 0; i < 16; ++i) s += acc[i];
    if (s == 1234.5f) sink[0] = s;
}

// --------------------------------------------------------------- TMEM probe
// Warp 0 allocates all 512 columns of the SM's tensor memory (one CTA per
// SM), every warp reads its subpartition's 32 lanes with tcgen05.ld
// 32x32b.x4 (16 bytes a thread, 512 a warp) at a warp-uniform random
// column, four loads per wait; MIX also issues one LDS.128 of a random
// staged row per TMEM load.  Warp 0 frees the columns before the CTA exits.
template <bool MIX, bool TM>
__global__ void __launch_bounds__(THREADS, 1) tmem_probe(int iters, unsigned long long* cycles, uint32_t* sink) {
    extern __shared__ __align__(1024) unsigned char smem[];
    __shared__ uint32_t tmem_base;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    for (int i = threadIdx.x; i < ROWS * PITCH / 4; i += THREADS) reinterpret_cast<uint32_t*>(smem)[i] = i * 2654435761u;
    if (TM && warp == 0) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], 512;" ::"r"(smem_u32(&tmem_base)));
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;");
    }
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
    __syncthreads();
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
    const uint32_t tbase = TM ? tmem_base + ((uint32_t)((warp & 3) * 32) << 16) : 0u;
    const uint32_t sbase = smem_u32(smem) + lane * 16;
    uint32_t x = 0, seed = 777u + warp * 7919u + blockIdx.x;
    const unsigned long long t0 = clock64();
#pragma unroll 1
    for (int it = 0; it < iters; ++it) {
        seed = seed * 1664525u + 1013904223u;
        const uint32_t col = ((seed >> 8) & 511u) & ~15u;   // 4 loads at col, +4, +8, +12
        const uint32_t row = (seed >> 4) % (ROWS - 4);
        if constexpr (TM) {
            uint32_t v[16];
            asm volatile(
                "tcgen05.ld.sync.aligned.32x32b.x4.b32 {%0,%1,%2,%3}, [%16];\n\t"
                "tcgen05.ld.sync.aligned.32x32b.x4.b32 {%4,%5,%6,%7}, [%17];\n\t"
                "tcgen05.ld.sync.aligned.32x32b.x4.b32 {%8,%9,%10,%11}, [%18];\n\t"
                "tcgen05.ld.sync.aligned.32x32b.x4.b32 {%12,%13,%14,%15}, [%19];\n\t"
                "tcgen05.wait::ld.sync.aligned;"
                : "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3]), "=r"(v[4]), "=r"(v[5]), "=r"(v[6]), "=r"(v[7]),
                  "=r"(v[8]), "=r"(v[9]), "=r"(v[10]), "=r"(v[11]), "=r"(v[12]), "=r"(v[13]), "=r"(v[14]), "=r"(v[15])
                : "r"(tbase + col), "r"(tbase + col + 4), "r"(tbase + col + 8), "r"(tbase + col + 12));
#pragma unroll
            for (int q = 0; q < 16; ++q) x ^= v[q];
        }
        if constexpr (MIX || !TM) {
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                uint32_t v0, v1, v2, v3;
                asm volatile("ld.shared.v4.u32 {%0,%1,%2,%3}, [%4];"
                             : "=r"(v0), "=r"(v1), "=r"(v2), "=r"(v3) : "r"(sbase + (row + k) * PITCH));
                x ^= v0 ^ v1 ^ v2 ^ v3;
            }
        }
    }
    const unsigned long long t1 = clock64();
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
    __syncthreads();
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
    if (TM && warp == 0) asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, 512;" ::"r"(tmem_base));
    if (threadIdx.x == 0) cycles[blockIdx.x] = t1 - t0;
    if (x == 0x9e3779b9u) sink[0] = x;
}

template <typename F>
void run(const char* name, F launch, int sms, double work_per_cta, const char* unit, unsigned long long* d_cyc) {
    cudaEvent_t e0, e1;
    CK(cudaEventCreate(&e0));
    CK(cudaEventCreate(&e1));
    for (int w = 0; w < 3; ++w) launch();
    CK(cudaDeviceSynchronize());
    const int reps = 10;
    CK(cudaEventRecord(e0));
    for (int r = 0; r < reps; ++r) launch();
    CK(cudaEventRecord(e1));
    CK(cudaDeviceSynchronize());
    float ms = 0;
    CK(cudaEventElapsedTime(&ms, e0, e1));
    unsigned long long* h = (unsigned long long*)malloc(sizeof(unsigned long long) * sms);
    CK(cudaMemcpy(h, d_cyc, sizeof(unsigned long long) * sms, cudaMemcpyDeviceToHost));
    unsigned long long mx = 0, mn = ~0ull;
    double sum = 0;
    for (int i = 0; i < sms; ++i) {
        mx = h[i] > mx ? h[i] : mx;
        mn = h[i] < mn ? h[i] : mn;
        sum += (double)h[i];
    }
    const double mean = sum / sms;
    const double per_launch_s = ms * 1e-3 / reps;
    printf("{\"probe\": \"%s\", \"%s_per_clk_sm\": %.2f, \"%s_per_clk_sm_slowest_cta\": %.2f, "
           "\"cycles_mean\": %.0f, \"cycles_min\": %llu, \"cycles_max\": %llu, \"ms_per_launch\": %.4f, "
           "\"implied_sm_mhz\": %.0f, \"total_%s_per_s\": %.4g, \"launches_timed\": %d}\n",
           name, unit, work_per_cta / mean, unit, work_per_cta / (double)mx, mean, mn, mx, per_launch_s * 1e3,
           mean / per_launch_s / 1e6, unit, work_per_cta * sms / per_launch_s, reps);
    fflush(stdout);
    free(h);
}

int main(int argc, char** argv) {
    int dev = 0, sms = 0;
    CK(cudaSetDevice(dev));
    CK(cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev));
    unsigned long long* d_cyc;
    uint32_t* d_sink;
    CK(cudaMalloc(&d_cyc, sizeof(unsigned long long) * sms));
    CK(cudaMalloc(&d_sink, 64));
    const bool with_tmem = argc > 1 && argv[1][0] == 't';

    CK(cudaFuncSetAttribute(lds_probe<4>, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM));
    CK(cudaFuncSetAttribute(lds_probe<8>, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM));
    CK(cudaFuncSetAttribute(lds_probe<16>, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM));
    CK(cudaFuncSetAttribute(fma_probe<0>, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM));
    CK(cudaFuncSetAttribute(fma_probe<1>, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM));
    CK(cudaFuncSetAttribute(fma_probe<2>, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM));
    const int it = 200000;
    // bytes per CTA: iters x 8 loads x 16 warps x 32 lanes x BYTES
    run("lds32_random_rows", [&] { lds_probe<4><<<sms, THREADS, SMEM>>>(it, d_cyc, d_sink); }, sms,
        (double)it * 8 * 16 * 32 * 4, "bytes", d_cyc);
    run("lds64_random_rows", [&] { lds_probe<8><<<sms, THREADS, SMEM>>>(it, d_cyc, d_sink); }, sms,
        (double)it * 8 * 16 * 32 * 8, "bytes", d_cyc);
    run("lds128_random_rows", [&] { lds_probe<16><<<sms, THREADS, SMEM>>>(it / 2, d_cyc, d_sink); }, sms,
        (double)(it / 2) * 8 * 16 * 32 * 16, "bytes", d_cyc);
    // flops per CTA: iters x 4 reps x 16 chains x 2 flop x 512 threads
    const int fi = 100000;
    const double fl = (double)fi * 4 * 16 * 2 * THREADS;
    run("fma_f32_scalar", [&] { fma_probe<0><<<sms, THREADS, SMEM>>>(fi, 0.999f, d_cyc, (float*)d_sink); }, sms, fl,
        "flop", d_cyc);
    run("fma_f32x2", [&] { fma_probe<1><<<sms, THREADS, SMEM>>>(fi, 0.999f, d_cyc, (float*)d_sink); }, sms, fl,
        "flop", d_cyc);
    run("fma_f32_bf16", [&] { fma_probe<2><<<sms, THREADS, SMEM>>>(fi, 0.999f, d_cyc, (float*)d_sink); }, sms, fl,
        "flop", d_cyc);
    if (with_tmem) {
        CK(cudaFuncSetAttribute(tmem_probe<false, true>, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM));
        CK(cudaFuncSetAttribute(tmem_probe<true, true>, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM));
        CK(cudaFuncSetAttribute(tmem_probe<false, false>, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM));
        const int ti = 100000;
        // per iteration per warp: 4 TMEM loads of 512 B; MIX adds 4 LDS.128 of 512 B
        run("tmem_ld_32x32b_x4", [&] { tmem_probe<false, true><<<sms, THREADS, SMEM>>>(ti, d_cyc, d_sink); }, sms,
            (double)ti * 4 * 512 * 16, "bytes", d_cyc);
        run("lds128_same_loop", [&] { tmem_probe<false, false><<<sms, THREADS, SMEM>>>(ti, d_cyc, d_sink); }, sms,
            (double)ti * 4 * 512 * 16, "bytes", d_cyc);
        run("tmem_ld_plus_lds128_mixed", [&] { tmem_probe<true, true><<<sms, THREADS, SMEM>>>(ti, d_cyc, d_sink); },
            sms, (double)ti * 8 * 512 * 16, "bytes", d_cyc);
    }
    CK(cudaGetLastError());
    CK(cudaDeviceSynchronize());
    printf("{\"sms\": %d, \"done\": true}\n", sms);
    return 0;
}
