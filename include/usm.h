/*
 * usm.h — C ABI of the GB300 (sm_103a) unstructured sparse matrix library.
 *
 * Operations from "Sparse GPU Kernels for Deep Learning" (Gale, Zaharia,
 * Young, Elsen, SC 2020): SpMM and SDDMM on plain CSR matrices with
 * unstructured, moderately sparse (70–98%) deep-learning sparsity, plus the
 * row-swizzle load-balancing order.  Every entry point takes plain pointers
 * and sizes; no C++ or framework type crosses this boundary.
 *
 * Conventions shared by every entry point
 * ---------------------------------------
 * Pointers.  Array arguments are DEVICE pointers owned by the caller.  The
 *   library never allocates, frees or keeps a pointer after the call returns.
 *   Scratch memory, where an operation needs it, is passed in by the caller
 *   ("workspace"); its size comes from the matching *_workspace_bytes call.
 * CSR.  row_offsets is int32[M+1] with row_offsets[0] = 0, non-decreasing,
 *   row_offsets[M] = nnz; col_indices is int32[nnz], each row's indices
 *   strictly increasing and in [0, K).  The compute calls do not scan the
 *   CSR (that would cost a pass over it; csr_validate does, on request); a
 *   CSR that breaks this contract gives
 *   undefined results but never an out-of-bounds dense access, because every
 *   column index is clamped into [0, K) before it addresses a dense operand.
 * Dense operands.  Row-major with a leading dimension (elements per row).
 *   Base pointers must be 16-byte aligned and ld·sizeof(element) a multiple
 *   of 16 bytes, else USM_ERR_ALIGNMENT.
 * Types.  usm_dtype names the INPUT element type (values and dense
 *   operands).  Products and sums are always fp32.  Dense outputs are fp32.
 * Asynchrony.  Calls enqueue work on `stream` (a cudaStream_t; NULL = the
 *   legacy default stream) and return without synchronising, except
 *   usm_poll_status.  Device-side failures (a bounded wait that timed out)
 *   are recorded in a per-device status word read by usm_poll_status.
 * Errors.  Every entry point returns USM_OK or a negative usm_status; none
 *   throws, aborts or prints.  Argument checks run on the host before any
 *   launch, so a rejected call touches no device memory.
 * Threads.  Calls may be issued from several host threads; the status word
 *   is shared by all calls on one device.  The library keeps the device
 *   address of that word (and of csr_sddmm_static_scratch's array) per device
 *   and per CUDA context, and looks it up again after a device reset.
 */
#ifndef USM_H_
#define USM_H_

#include <stddef.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum usm_dtype { USM_F32 = 0, USM_BF16 = 1 } usm_dtype;

typedef enum usm_status {
    USM_OK = 0,
    USM_ERR_INVALID_ARG = -1, /* negative size, NULL pointer with nonzero size, bad enum */
    USM_ERR_ALIGNMENT = -2,   /* dense pointer or leading dimension not 16-byte aligned */
    USM_ERR_UNSUPPORTED = -3, /* shape outside the documented limits */
    USM_ERR_CUDA = -4,        /* a CUDA runtime call or launch failed */
    USM_ERR_TIMEOUT = -5,     /* a device-side bounded wait gave up (see usm_poll_status) */
    USM_ERR_WORKSPACE = -6    /* workspace NULL or smaller than *_workspace_bytes */
} usm_status;

/*
 * csr_spmm — sparse × dense product, C = A · B.
 *
 * Source: "Sparse GPU Kernels for Deep Learning", summary card, "Summary"
 * (SpMM on plain CSR with unstructured sparsity; the sparse layer's forward
 * pass, and its input gradient when A is the transposed weight).
 *
 *   A : M×K sparse, CSR (row_offsets, col_indices, values[nnz] of `dtype`).
 *   B : K×N dense, row-major, leading dimension ldb ≥ N, elements of `dtype`.
 *   C : M×N dense fp32, row-major, leading dimension ldc ≥ N.  OVERWRITTEN:
 *       C[r][j] = Σ_{p in row r} values[p] · B[col_indices[p]][j]
 *       (rows of A with no nonzeros give zero rows of C).
 *   row_swizzle : NULL, or int32[M], a permutation of 0..M-1 giving the order
 *       in which rows are scheduled (see row_swizzle_build).  It changes only
 *       the schedule, never the result (each output row is computed by one
 *       unit in a fixed order).
 *   seg_rows : the rows per diagonal block the swizzle was built with (the
 *       seg_rows of row_swizzle_build); <= 0 or > M means one block.  The row
 *       scheduler deals each block's swizzled rows out to thread blocks so
 *       that every thread block gets a similar mix of row lengths and never
 *       rows of two blocks.  Like the swizzle, it never changes the result.
 * Limits: 0 ≤ M, K, N < 2^31, nnz < 2^31; ldc a multiple of 4.
 * Empty cases: M = 0 or N = 0 is a no-op; nnz = 0 zero-fills C.
 */
int csr_spmm(int M, int K, int N, int nnz,
             const int *row_offsets, const int *col_indices, const void *values,
             const int *row_swizzle, int seg_rows,
             const void *B, int ldb,
             float *C, int ldc,
             usm_dtype dtype, void *stream);

/*
 * csr_sddmm — sampled dense–dense product on the mask of A.
 *
 * Source: "Sparse GPU Kernels for Deep Learning", summary card, "Interesting
 * ideas" I3: the specialised form drops the element-wise scaling by A's
 * values and takes the second operand transposed, the form weight gradients
 * and sparse-attention scores need.
 *
 *   mask : M×K, CSR (row_offsets, col_indices); values are not read.
 *   X    : M×D dense, row-major, leading dimension ldx ≥ D, `in_dtype`.
 *   Y    : K×D dense, row-major, leading dimension ldy ≥ D, `in_dtype`
 *          (used transposed: the product is X·Yᵀ).
 *   out  : [nnz] in the mask's CSR order, element type `out_dtype`
 *          (USM_F32, or USM_BF16 rounded to nearest even from the fp32 sum):
 *          out[p] = Σ_{j<D} X[r][j] · Y[col_indices[p]][j],  p in row r.
 *   row_swizzle, seg_rows : as csr_spmm (schedule only).
 *   workspace : device scratch of at least
 *          csr_sddmm_workspace_bytes(M, K, D, nnz, in_dtype) bytes; may be
 *          NULL when that size is 0.  Its contents on entry are ignored and
 *          undefined on return (partials already summed are dropped from the
 *          L2 cache without being written back).
 * Limits: as csr_spmm.  nnz = 0 or M = 0 is a no-op; D = 0 zero-fills out.
 */
size_t csr_sddmm_workspace_bytes(int M, int K, int D, int nnz, usm_dtype in_dtype);

int csr_sddmm(int M, int K, int D, int nnz,
              const int *row_offsets, const int *col_indices,
              const int *row_swizzle, int seg_rows,
              const void *X, int ldx,
              const void *Y, int ldy,
              void *out, usm_dtype in_dtype, usm_dtype out_dtype,
              void *workspace, size_t workspace_bytes,
              void *stream);

/*
 * csr_sddmm_static_scratch — csr_sddmm for callers that cannot allocate.
 *
 * The paper has no counterpart to this entry point; it exists for callers
 * that cannot call cudaMalloc (a plugin that only receives raw pointers from
 * its host framework, a loop whose device memory was fixed at start-up, an
 * environment that forbids allocation after initialisation) and so cannot
 * supply csr_sddmm's workspace.  Same arguments, contract and result as
 * csr_sddmm, minus the workspace: the scratch comes from one fixed 32 MiB
 * array in the library's device image.
 *
 *   Limit: csr_sddmm_workspace_bytes(M, K, D, nnz, in_dtype) must not exceed
 *          32 MiB (33554432 bytes); larger problems return USM_ERR_UNSUPPORTED
 *          before anything is launched.  Problems that need no workspace
 *          (one column strip) always fit and never touch the array.
 *   Set-up: the first call on a device that needs the array (with that
 *          device current) looks up its device address with
 *          cudaGetSymbolAddress.  CUDA loads the library's device code
 *          lazily, so this first call may also load the module that holds
 *          the array and reserve its 32 MiB on that device; it returns
 *          USM_ERR_CUDA if the device has no room for it.  Make that first
 *          call during initialisation, before device memory is fixed and
 *          before any stream capture.  The 32 MiB stay reserved until the
 *          device's context ends; after a device reset the next call does
 *          the set-up again.
 *   Allocation: none on later calls (no cudaMalloc, cudaFree or allocating
 *          library routine).
 *   Sharing: every call on a device uses the same array, whose contents
 *          between calls are undefined.  On a CSR that meets the contract nothing in
 *          it needs to start at zero; on one that does not (see
 *          csr_validate), or after USM_ERR_TIMEOUT, the output may hold values
 *          left there by an earlier call.  Calls whose executions overlap on
 *          the GPU (other streams, other host threads) race on the array and
 *          give wrong results: serialise them.
 */
int csr_sddmm_static_scratch(int M, int K, int D, int nnz,
                             const int *row_offsets, const int *col_indices,
                             const int *row_swizzle, int seg_rows,
                             const void *X, int ldx,
                             const void *Y, int ldy,
                             void *out, usm_dtype in_dtype, usm_dtype out_dtype,
                             void *stream);

/*
 * row_swizzle_build — the row-swizzle processing order.
 *
 * Source: "Sparse GPU Kernels for Deep Learning", summary card, "Summary"
 * (a decoupled load-balancing scheme) and "Interesting ideas" I4 (row
 * swizzle balances work independently of how the computation is split).
 * Reading used here: rows are listed by decreasing length, rows of equal
 * length by increasing index, so the permutation is unique.  With
 * seg_rows > 0 the order is built separately inside each run of seg_rows
 * consecutive rows (the diagonal blocks of a batched block-diagonal matrix,
 * e.g. one block per attention head); seg_rows ≤ 0 means a single run.
 *
 *   row_offsets : int32[M+1] (only lengths are read).
 *   swizzle_out : int32[M], written with the permutation.
 *   workspace   : at least row_swizzle_workspace_bytes(M, K) bytes of device
 *                 scratch (contents ignored on entry).
 * Bit-exact and deterministic.  M = 0 is a no-op.
 */
size_t row_swizzle_workspace_bytes(int M, int K);

int row_swizzle_build(int M, int K, int seg_rows, const int *row_offsets, int *swizzle_out,
                      void *workspace, size_t workspace_bytes, void *stream);

/*
 * csr_sddmm_general — SDDMM with the element-wise scaling and operand
 * orientation the specialised form drops.
 *
 * Source: "Sparse GPU Kernels for Deep Learning", summary card, "Interesting
 * ideas" I3 (the general case, which the authors note is easy to add).
 *
 *   out[p] = s_p · Σ_{j<D} X[r][j] · Yop[col_indices[p]][j],  p in row r,
 *   s_p = values[p] (mask values, `in_dtype`) or 1 when values is NULL,
 *   Yop = Y when y_transposed = 1 (Y is K×D, ldy ≥ D, as csr_sddmm), or
 *   Yop = Yᵀ when y_transposed = 0 (Y is D×K row-major, ldy ≥ K; it is
 *   transposed into the workspace first, so it has no alignment rule).
 *   The scaling multiplies the fp32 dot product once (one extra rounding).
 *   workspace : csr_sddmm_general_workspace_bytes(M, K, D, nnz, in_dtype,
 *           y_transposed) bytes, 256-byte aligned, contents ignored.
 * Other arguments, limits and empty cases as csr_sddmm.
 */
size_t csr_sddmm_general_workspace_bytes(int M, int K, int D, int nnz, usm_dtype in_dtype, int y_transposed);

int csr_sddmm_general(int M, int K, int D, int nnz,
                      const int *row_offsets, const int *col_indices, const void *values,
                      const int *row_swizzle, int seg_rows,
                      const void *X, int ldx,
                      const void *Y, int ldy, int y_transposed,
                      void *out, usm_dtype in_dtype, usm_dtype out_dtype,
                      void *workspace, size_t workspace_bytes, void *stream);

/*
 * csr_row_softmax — softmax over the stored entries of each CSR row:
 *   out[p] = exp(s[p] - m_r) / Σ_{q in row r} exp(s[q] - m_r),  m_r = max_q s[q],
 * scores fp32 [nnz], out fp32 or bf16 (nearest even) [nnz]; empty rows write
 * nothing.  The normalisation step between the SDDMM scores and the SpMM of
 * sparse attention (the sparse-attention use of the kernels, "Interesting
 * ideas" I3).  Error: ≤ n/128 + 9 fp32 roundings per output for a row of n
 * entries (four partial sums a lane, a 2-level and a 5-level tree, a
 * reciprocal of the sum and one product) on top of the exponentials', which
 * use the fast hardware exp (CUDA's __expf: at most 2 + 1.17·|s - m| ulp).
 * csr_spmm_row_softmax forms the same values bit for bit.
 */
int csr_row_softmax(int M, int nnz, const int *row_offsets, const float *scores, void *out,
                    usm_dtype out_dtype, void *stream);

/*
 * csr_spmm_row_softmax — sparse attention's softmax fused into the SpMM:
 *   C[r][j] = Σ_{p in row r} P[p] · B[col_indices[p]][j],
 *   P[p] = exp(s[p] - m_r) / Σ_{q in row r} exp(s[q] - m_r),  m_r = max_{q in row r} s[q],
 * the row softmax over each row's stored entries of the fp32 `scores` (the
 * SDDMM output of the sparse-attention chain), taken inside the product.
 * Each P[p] is formed in fp32 exactly as csr_row_softmax forms it (same
 * operations in the same order, bit for bit), then rounded to `dtype`
 * (USM_BF16: nearest even; USM_F32: unchanged) and multiplied as csr_spmm
 * multiplies values: the result is bit-identical to csr_row_softmax into a
 * `dtype` buffer followed by csr_spmm on it, without that buffer's write and
 * read.  Source: "Sparse GPU Kernels for Deep Learning", summary card,
 * "Interesting ideas" I3 (the SDDMM and SpMM of sparse attention); the
 * softmax between them is this library's.
 *
 *   scores : fp32 [nnz] in the CSR order of (row_offsets, col_indices).
 *   B      : K×N dense, row-major, ldb ≥ N, elements of `dtype`.
 *   C      : M×N fp32, ldc ≥ N, overwritten; empty rows give zero rows.
 *   row_swizzle, seg_rows : as csr_spmm (schedule only).
 * Limits, alignment and empty cases as csr_spmm.
 */
int csr_spmm_row_softmax(int M, int K, int N, int nnz,
                         const int *row_offsets, const int *col_indices, const float *scores,
                         const int *row_swizzle, int seg_rows,
                         const void *B, int ldb,
                         float *C, int ldc,
                         usm_dtype dtype, void *stream);

/*
 * csr_transpose — Aᵀ in CSR, for the sparse layer's input gradient.
 *
 * Source: "Sparse GPU Kernels for Deep Learning", summary card, "Summary"
 * (the kernels serve training as well as inference; the input gradient of a
 * sparse layer C = A·B is dB = Aᵀ·dC, an SpMM on the transposed weight).
 *
 *   A     : M×K, CSR (row_offsets, col_indices, values of `dtype`; values may
 *           be NULL to transpose the structure only, then values_t is NULL).
 *   Aᵀ    : K×M, CSR written to row_offsets_t[K+1], col_indices_t[nnz] and
 *           values_t[nnz].  Each row of Aᵀ lists its column indices (rows of
 *           A) in increasing order, so the result is unique and bit-exact.
 *   perm_out : NULL, or int32[nnz] receiving, for each nonzero q of Aᵀ, the
 *           position in A's arrays it came from (values_t[q] = values[perm[q]]);
 *           csr_permute_values re-gathers new values with it.
 *   workspace : at least csr_transpose_workspace_bytes(M, K, nnz) bytes of
 *           device scratch, 256-byte aligned (contents ignored on entry).
 * Column indices outside [0, K) are clamped (contract violations give
 * undefined but in-bounds results).  nnz = 0 writes row_offsets_t = 0.
 */
size_t csr_transpose_workspace_bytes(int M, int K, int nnz);

int csr_transpose(int M, int K, int nnz,
                  const int *row_offsets, const int *col_indices, const void *values,
                  usm_dtype dtype,
                  int *row_offsets_t, int *col_indices_t, void *values_t, int *perm_out,
                  void *workspace, size_t workspace_bytes, void *stream);

/*
 * csr_permute_values — out[q] = values[perm[q]] for q < nnz (fp32 or bf16
 * elements): moves a CSR's values into the order of a fixed transpose
 * permutation (see csr_transpose), e.g. after each weight update.
 */
int csr_permute_values(int nnz, const int *perm, const void *values, usm_dtype dtype, void *out,
                       void *stream);

/*
 * usm_poll_status — synchronise `stream`, then return and clear the current
 * device's status word: USM_OK, or USM_ERR_TIMEOUT when a kernel's bounded
 * wait (on a TMA transfer) gave up and the kernel returned early (its output
 * is then incomplete).  Returns USM_ERR_CUDA if the synchronisation fails.
 */
int usm_poll_status(void *stream);

/* Human-readable name of a usm_status value (static string, never NULL). */
const char *usm_status_string(int status);

/*
 * csr_validate — checks the CSR contract above on the device, for callers
 * whose matrices come from outside (the pages give plain CSR, "Interesting
 * ideas" I5; the strictly increasing column order is this library's
 * reading).  The compute entry points never scan the CSR themselves.
 *   result : device int[USM_CSR_VALIDATE_INTS], caller-owned, 4-byte aligned;
 *            on completion (stream order) result[0] is a usm_csr_check code
 *            and result[1] the first offending index (the row for offset
 *            codes, M for USM_CSR_LAST_OFFSET, the nonzero position for
 *            column codes; -1 when valid).  Words 2.. are scratch.
 * Violations are reported in this order, the first that applies:
 * row_offsets[0] != 0; offsets decreasing (first such row r:
 * row_offsets[r+1] < row_offsets[r]); row_offsets[M] != nnz; then the first
 * nonzero position p whose column is outside [0, K) (range) or not above the
 * previous column of its row (order), range winning a tie.  Reads stay
 * inside row_offsets[0..M] and col_indices[0..nnz) whatever the contents.
 * Returns USM_ERR_INVALID_ARG for negative sizes or NULL pointers (col_indices
 * may be NULL when nnz = 0), else USM_OK / USM_ERR_CUDA for the launch.
 */
typedef enum usm_csr_check {
    USM_CSR_VALID = 0,
    USM_CSR_FIRST_OFFSET = 1,     /* row_offsets[0] != 0 */
    USM_CSR_OFFSETS_DECREASE = 2, /* row_offsets[r+1] < row_offsets[r] */
    USM_CSR_LAST_OFFSET = 3,      /* row_offsets[M] != nnz */
    USM_CSR_COLUMN_RANGE = 4,     /* col_indices[p] outside [0, K) */
    USM_CSR_COLUMN_ORDER = 5      /* col_indices[p] <= col_indices[p-1] within a row */
} usm_csr_check;

#define USM_CSR_VALIDATE_INTS 8

int csr_validate(int M, int K, int nnz, const int *row_offsets, const int *col_indices, int *result,
                 void *stream);

/*
 * usm_selftest_wait_timeout — checks the bounded-wait path without faulting
 * anything: launches one CTA that waits on a shared-memory barrier nothing
 * will ever complete, with a limit of `limit_ns` nanoseconds (1e3..1e9).
 * The kernel gives up, records USM_ERR_TIMEOUT in the status word and
 * returns, so the next usm_poll_status(stream) returns USM_ERR_TIMEOUT.
 */
int usm_selftest_wait_timeout(long long limit_ns, void *stream);

/*
 * usm_set_schedule_override — for tests and tuning (the pages have no
 * counterpart): forces the launch shape of later csr_spmm and csr_sddmm
 * calls (including the general and static-scratch forms) in this process.
 * A field of 0 keeps the library's own choice.
 *   rows_per_warp    row slots per warp, one of 1, 2, 4, 8, 16, 32
 *                    (csr_spmm has kernels for 2 and 4, and for 4 and 8 on
 *                    fp32 masks under 7% set with N > 64: a forced value it
 *                    has none for makes the call return USM_ERR_UNSUPPORTED);
 *   tiles_per_block  row tiles per diagonal block of the schedule (raised to
 *                    the fewest that hold a block, if below);
 *   k_splits         csr_sddmm: ranges of K chunks, one CTA each (split
 *                    counts above the chunk count leave CTAs idle);
 *                    csr_spmm accepts only 0 or 1.
 * Results do not depend on the schedule: an SDDMM output adds the same
 * terms in the same order under every schedule, and so does an SpMM output
 * under every schedule of one element type and strip width.  While an
 * override is set, csr_spmm always runs its staged kernels: fp32 masks
 * under 3% set with N <= 128, which it otherwise serves with a kernel that
 * gathers the rows of B without staging (and sums in another order), then
 * give results within the same tolerance but not the same bits.  The setting is
 * process-wide and not ordered with calls issued concurrently on other
 * threads.  Returns USM_ERR_INVALID_ARG (setting unchanged) for a value
 * outside these sets.
 */
int usm_set_schedule_override(int rows_per_warp, int tiles_per_block, int k_splits);

#ifdef __cplusplus
}
#endif

#endif /* USM_H_ */
