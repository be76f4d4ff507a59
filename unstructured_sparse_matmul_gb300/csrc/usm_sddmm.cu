// CSR SDDMM: host launch code (strip width, launch model, workspace, kernel
// launches).  The kernels and their design are in usm_sddmm_kernel.cuh.
#include <climits>

#include "usm_internal.h"
#include "usm_sddmm_kernel.cuh"

// Most K splits per tile the launch model may choose (1 turns splitting off).
#ifndef USM_SDDMM_MAX_SPLIT
#define USM_SDDMM_MAX_SPLIT 16
#endif

namespace usm {
namespace {

template <bool BF, int L, int VV, int W, int KC, int MINB, int NS, bool TM = false>
int launch_cfg(SddmmArgs a, const void* Y, int ldy, void* ws, size_t ws_bytes, cudaStream_t stream) {
    using C_ = SddmmCfg<BF, L, VV, W, KC, MINB, NS>;
    CUtensorMap map;
    if (!encode_tensor_map_2d(&map, Y, BF, a.K, a.D, ldy, C_::DT, C_::BOX_ROWS)) return USM_ERR_CUDA;
    auto kern = sddmm_kernel<BF, L, VV, W, KC, MINB, NS, TM>;
    static int configured_mask = 0;
    int dev = 0;
    cudaGetDevice(&dev);
    if (dev < 31 && !(__atomic_load_n(&configured_mask, __ATOMIC_ACQUIRE) & (1 << dev))) {
        if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C_::SMEM) !=
            cudaSuccess)
            return USM_ERR_CUDA;
        __atomic_fetch_or(&configured_mask, 1 << dev, __ATOMIC_ACQ_REL);
    }
    const int nstrips = (a.D + C_::DT - 1) / C_::DT;
    if (nstrips > 65535) return USM_ERR_UNSUPPORTED;
    void* final_out = a.out;
    // Strips of partials lie partial_stride(nnz) elements apart (a multiple of
    // 32: every strip starts 16-byte aligned for the strip sum's loads, and
    // 128-byte aligned when the workspace is, so no 128-byte line of partials
    // spans two strips).
    const long long stride = partial_stride(a.nnz);
    if (nstrips > 1) {
        if (ws == nullptr || ws_bytes < (size_t)nstrips * (size_t)stride * sizeof(float))
            return USM_ERR_WORKSPACE;
        a.out = ws;
        a.out_stride = stride;
    }
    const int sms = sm_count_current_device();
    const long long slots = (long long)sms * MINB;
    const int seg = a.seg_rows;  // rows per diagonal block (M without blocks)
    const long long nblk = block_count(a.M, seg);
    // A block-diagonal schedule (seg_rows < M) is taken to have square blocks.
    const double kspan = (seg > 0 && seg < a.M) ? (double)min(a.K, seg) : (double)a.K;
    const double mean_len = (double)a.nnz / (a.M > 0 ? a.M : 1);
    const int nch = max(1, (int)((kspan + KC - 1) / KC));
    // Rows per warp R, K splits S and tiles per block T from a launch time
    // model fitted to a sweep of the FFN launches (R ∈ {4..32}, every
    // effective S, T the fewest tiles or the most that still fit in the same
    // number of CTA waves; L2 flushed between calls; the model's choices sum
    // to 1.2% above the best per launch on 128-wide strips, 2% on 256-wide
    // ones).  Time = waves × per-CTA work, with waves = ceil(CTAs / resident
    // slots): CTAs of a launch have near-equal work (swizzled rows), so a
    // part-filled last wave costs a whole one and more, shorter tiles that
    // fill it are free.  Work is counted in consumed nonzeros: staging the
    // CTA's share of the K span (0.45 a staged row), the nonzeros of its rows
    // in its share of the span, a fixed start-up (6000: first copy, cursor
    // search, epilogue) and a latency per (row, chunk) that a warp's rows pay
    // one after another (880).  Splitting K costs no reduction (each nonzero
    // belongs to one split); only split counts that give every split a
    // different chunk range are tried.
    int R = 1, S = 1, T = 1;
    {
        double best = 0.0;
        const long long tmax = max(1, (seg + W - 1) / W);  // at least one row a warp
        for (int sp = 1; sp <= min(USM_SDDMM_MAX_SPLIT, nch); ++sp) {
            const int per = (nch + sp - 1) / sp;
            if ((nch + per - 1) / per != sp) continue;  // same ranges as a smaller count
            const long long ctas_per_t = nblk * nstrips * sp;
            for (int r = 1; r <= 32; r <<= 1) {
                const long long t0 = (seg + r * W - 1) / (r * W);
                const long long waves0 = (ctas_per_t * t0 + slots - 1) / slots;
                const long long t1 = min(max(tmax, t0), max(t0, waves0 * slots / ctas_per_t));
                for (const long long t : {t0, t1}) {
                    const long long rows = (seg + t - 1) / t;
                    const long long reff = (rows + W - 1) / W;
                    const double waves = (double)((ctas_per_t * t + slots - 1) / slots);
                    const double work =
                        (0.45 * kspan + (double)rows * mean_len) * per / nch + 6000.0 + 880.0 * per * reff;
                    const double c = waves * work;
                    if (best == 0.0 || c < best) {
                        best = c;
                        R = (int)reff;
                        S = sp;
                        T = (int)t;
                    }
                }
            }
        }
    }
    const ScheduleOverride ov = schedule_override();
    if (ov.rows_per_warp > 0 || ov.tiles_per_block > 0) {
        if (ov.rows_per_warp > 0) R = ov.rows_per_warp;
        T = max((seg + R * W - 1) / (R * W), ov.tiles_per_block);
    }
    if (ov.k_splits > 0) S = ov.k_splits;
    // Every row of a block must have a slot: tiles × R·W ≥ rows per block.
    if (R < 1 || R > 32 || T < 1 || (long long)T * R * W < seg) return USM_ERR_INVALID_ARG;
    a.rows_per_warp = R;
    a.tiles_per_block = T;
    const long long tiles = block_count(a.M, a.seg_rows) * a.tiles_per_block;
    if (tiles > 0x7fffffffLL) return USM_ERR_UNSUPPORTED;
    const dim3 grid((unsigned)tiles, nstrips, S);
    kern<<<grid, C_::THREADS, C_::SMEM, stream>>>(map, a);
    if (cudaGetLastError() != cudaSuccess) return USM_ERR_CUDA;
    if (nstrips > 1) {
        const size_t ob = a.out_bf16 ? 8 : 16, sb = a.scale_bf16 ? 8 : 16;
        const bool vec = (uintptr_t)ws % 16 == 0 && (uintptr_t)final_out % ob == 0 &&
                         (a.scale == nullptr || (uintptr_t)a.scale % sb == 0);
        const long long items = vec ? (a.nnz + 3) / 4 : a.nnz;
        long long blocks = (items + 255) / 256;
        if (blocks > 8 * sms) blocks = 8 * sms;
        const int discard = USM_PARTIAL_DISCARD && (uintptr_t)ws % 128 == 0;
        if (vec)
            sddmm_strip_sum4_kernel<<<(int)blocks, 256, 0, stream>>>(static_cast<const float*>(ws), a.nnz, stride,
                                                                     nstrips, final_out, a.out_bf16, a.scale,
                                                                     a.scale_bf16, discard);
        else
            sddmm_strip_sum_kernel<<<(int)blocks, 256, 0, stream>>>(static_cast<const float*>(ws), a.nnz, stride,
                                                                    nstrips, final_out, a.out_bf16, a.scale,
                                                                    a.scale_bf16);
        if (cudaGetLastError() != cudaSuccess) return USM_ERR_CUDA;
    }
    return USM_OK;
}

// Strip width by density, element type and D: 256 columns when at least a
// quarter of the mask is set, else 128 (bf16 with D <= 64: 64).  Wider strips
// halve the partials and the list work per FMA but double the work per (row,
// chunk), which dominates at high sparsity.  Measured on the FFN shapes, 256
// against 128: fp32 4-6% faster at 70% sparsity, -2..+2% at 80%, 3-11%
// slower at 90-95%; bf16 0-7% faster at 70%, -5..+2% at 80-90%, 9-13%
// slower at 95%.
int strip_width(int M, int K, int D, int nnz, bool bf16) {
    if (bf16 && D <= 64) return 64;
    return 4LL * nnz >= (long long)M * K ? 256 : 128;
}

}  // namespace

long long partial_stride(long long nnz) { return (nnz + 31) / 32 * 32; }

size_t sddmm_workspace_bytes(int M, int K, int D, int nnz, bool bf16) {
    if (D <= 0 || nnz <= 0) return 0;
    const int dt = strip_width(M, K, D, nnz, bf16);
    const long long nstrips = (D + dt - 1) / dt;
    return nstrips > 1 ? (size_t)nstrips * (size_t)partial_stride(nnz) * sizeof(float) : 0;
}


int launch_dense_transpose(const void* src, long long lds, int rows, int cols, bool bf16, void* dst,
                           long long ldd, cudaStream_t stream) {
    if ((long long)rows * cols == 0) return USM_OK;
    const dim3 grid((cols + 31) / 32, (rows + 31) / 32), block(32, 8);
    if (grid.y > 65535u) return USM_ERR_UNSUPPORTED;
    if (bf16)
        dense_transpose_kernel<uint16_t><<<grid, block, 0, stream>>>(static_cast<const uint16_t*>(src), lds, rows, cols,
                                                                     static_cast<uint16_t*>(dst), ldd);
    else
        dense_transpose_kernel<float><<<grid, block, 0, stream>>>(static_cast<const float*>(src), lds, rows, cols,
                                                                  static_cast<float*>(dst), ldd);
    return cudaGetLastError() == cudaSuccess ? USM_OK : USM_ERR_CUDA;
}

int launch_fill_out(void* out, long long n, bool bf16, cudaStream_t stream) {
    if (n <= 0) return USM_OK;
    long long blocks = (n + 255) / 256;
    if (blocks > 4096) blocks = 4096;
    fill_out_kernel<<<(int)blocks, 256, 0, stream>>>(out, n, bf16 ? 1 : 0);
    return cudaGetLastError() == cudaSuccess ? USM_OK : USM_ERR_CUDA;
}

#ifndef USM_SDDMM_STAGES
#define USM_SDDMM_STAGES 1
#endif
int launch_sddmm(SddmmArgs a, const void* Y, int ldy, bool in_bf16, void* ws, size_t ws_bytes,
                 cudaStream_t stream) {
    constexpr int W = 16, NS = USM_SDDMM_STAGES, F = 2 / NS;  // F: chunk growth with one stage
    // fp32: one CTA per SM, up to 128 registers, one stage of 192 KB or more
    // (KC = 384 or 416 rows of a 128-wide strip, 192 or 216 of a 256-wide
    // one).
    if (!in_bf16) {
        // 256-wide strips (masks at least a quarter set); USM_SDDMM_TMEM=1 also
        // reads the last 64 rows of every chunk from tensor memory.
// Measured 8-16% slower at 70% sparsity (those nonzeros go one a warp step
// with 8 products a lane, against 4 a step with 32 on the shared-memory path).
#ifndef USM_SDDMM_TMEM
#define USM_SDDMM_TMEM 0
#endif
        // Chunk rows: 216 (a 216 KB stage, what the shared memory leaves beside
        // the lists) where that saves a chunk against 192: 2-3% faster on the
        // FFN launches at 70% sparsity; 224 ran the same or slower.  The
        // results do not depend on the chunk height (each nonzero is one dot
        // product over the strip).
#ifndef USM_SDDMM_KC256
#define USM_SDDMM_KC256 (108 * F)
#endif
        if (strip_width(a.M, a.K, a.D, a.nnz, false) == 256) {
            constexpr bool TM = USM_SDDMM_TMEM && NS == 1;
            if (taller_chunk_pays(a.K, 96 * F, USM_SDDMM_KC256))
                return launch_cfg<false, 8, 8, W, USM_SDDMM_KC256, 1, NS, TM>(a, Y, ldy, ws, ws_bytes, stream);
            return launch_cfg<false, 8, 8, W, 96 * F, 1, NS, TM>(a, Y, ldy, ws, ws_bytes, stream);
        }
        // 128-wide strips hold half the X registers (80 a thread at 24 warps):
        // 24 warps hide more of the loads' latency.  Measured against 16 on the
        // FFN launches (80-95% sparsity): 5-6% faster at 80%, 9% at 90%,
        // 11-12% at 95%; 20 and 32 warps gained less.  (256-wide strips, 96
        // registers at 20 warps: no change, those launches are bound by
        // shared-memory bandwidth.)
        // Launch-bound problems (one or two CTAs: the 256x256 mask at 90%, 4.2
        // against 4.6 us a call) keep 16 warps, whose set-up is shorter.
#ifndef USM_SDDMM_W128
#define USM_SDDMM_W128 24
#endif
        // Chunk rows: 416 where that saves a chunk against 384 (FFN 1024x4096
        // at 80-95% sparsity 1.5-5% faster; with K = 1024, where it saves none,
        // 1-3% slower).
#ifndef USM_SDDMM_KC128
#define USM_SDDMM_KC128 (208 * F)
#endif
        if (a.nnz < 100000) return launch_cfg<false, 8, 4, W, 192 * F, 1, NS>(a, Y, ldy, ws, ws_bytes, stream);
        if (taller_chunk_pays(a.K, 192 * F, USM_SDDMM_KC128))
            return launch_cfg<false, 8, 4, USM_SDDMM_W128, USM_SDDMM_KC128, 1, NS>(a, Y, ldy, ws, ws_bytes, stream);
        return launch_cfg<false, 8, 4, USM_SDDMM_W128, 192 * F, 1, NS>(a, Y, ldy, ws, ws_bytes, stream);
    }
    // bf16: one CTA a SM of 28 warps (D > 64; 64-72 registers) or 32 (D <= 64;
    // 56), one 192 KB stage, against two CTAs of 16 warps with 96 KB each: the
    // same or more warps, twice the rows sharing each staged chunk and half the
    // chunk visits.  Measured on the FFN launches: 6% less bf16 SDDMM time in
    // all (70%: 8-16% faster, 80% -3..+2%, 90-95% 4-12%; 24 warps gained less,
    // 32 spilled); attention (D = 64, 32 warps): 7% faster, 24 warps slower.
#ifndef USM_SDDMM_BF_W
#define USM_SDDMM_BF_W 28
#endif
#ifndef USM_SDDMM_BF_MB
#define USM_SDDMM_BF_MB 1
#endif
#ifndef USM_SDDMM_BF64_W
#define USM_SDDMM_BF64_W 32
#endif
#ifndef USM_SDDMM_BF64_MB
#define USM_SDDMM_BF64_MB 1
#endif
    constexpr int BW = USM_SDDMM_BF_W, BMB = USM_SDDMM_BF_MB, SW = USM_SDDMM_BF64_W, SMB = USM_SDDMM_BF64_MB;
    if (a.D <= 64) return launch_cfg<true, 8, 1, SW, 768 * F / SMB, SMB, NS>(a, Y, ldy, ws, ws_bytes, stream);
    // Chunk rows: 416 (256-wide strips) and 832 (128-wide) where that saves a
    // chunk against 384 and 768: FFN 1024x4096 at 70% 1.6% faster, 80% 6%,
    // 90% 2.5%, 95% even (432 and 864 the same).
#ifndef USM_SDDMM_BF_KC_TALL
#define USM_SDDMM_BF_KC_TALL (208 * F / BMB)
#endif
#ifndef USM_SDDMM_BF128_KC_TALL
#define USM_SDDMM_BF128_KC_TALL (416 * F / BMB)
#endif
    if (strip_width(a.M, a.K, a.D, a.nnz, true) == 256) {
        if (taller_chunk_pays(a.K, 192 * F / BMB, USM_SDDMM_BF_KC_TALL))
            return launch_cfg<true, 8, 4, BW, USM_SDDMM_BF_KC_TALL, BMB, NS>(a, Y, ldy, ws, ws_bytes, stream);
        return launch_cfg<true, 8, 4, BW, 192 * F / BMB, BMB, NS>(a, Y, ldy, ws, ws_bytes, stream);
    }
    if (taller_chunk_pays(a.K, 384 * F / BMB, USM_SDDMM_BF128_KC_TALL))
        return launch_cfg<true, 8, 2, BW, USM_SDDMM_BF128_KC_TALL, BMB, NS>(a, Y, ldy, ws, ws_bytes, stream);
    return launch_cfg<true, 8, 2, BW, 384 * F / BMB, BMB, NS>(a, Y, ldy, ws, ws_bytes, stream);
}

}  // namespace usm
