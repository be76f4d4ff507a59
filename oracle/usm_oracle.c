/*
 * CPU oracle for CSR SpMM / SDDMM — TEST INFRASTRUCTURE ONLY.
 *
 * Plain, slow, obviously correct restatements of the operations described in
 * "Sparse GPU Kernels for Deep Learning" (Gale, Zaharia, Young, Elsen,
 * SC 2020; summary card "Summary" and "Interesting ideas" I3, I4, I5).  Every
 * floating-point sum is accumulated in fp64 in CSR order; inputs arrive
 * already widened (exactly) to fp64.  No blocking, tiling or reordering.
 *
 * Only the test suite, the smoke check and the benchmark's CPU-baseline arm
 * may load this library.  It shares no source, header or helper with the CUDA
 * library; the two only ever see the same input arrays.
 *
 * Build: gcc -O2 -fopenmp -ffp-contract=off -shared -fPIC (contraction off so
 * x86-64 and aarch64 hosts give bit-identical results).
 */
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#include <math.h>
#ifdef _OPENMP
#include <omp.h>
#endif

/* Threads for the next parallel loop: nthreads > 0 asks for that many, 0 for
 * the process default (OMP_NUM_THREADS or all cores), captured on first use so
 * an earlier call with a fixed count does not shrink later "all cores" calls. */
static int g_default_threads = 0;

static int default_threads(void) {
#ifdef _OPENMP
    if (g_default_threads == 0) g_default_threads = omp_get_max_threads();
    return g_default_threads;
#else
    return 1;
#endif
}

static void set_threads(int nthreads) {
#ifdef _OPENMP
    omp_set_num_threads(nthreads > 0 ? nthreads : default_threads());
#else
    (void)nthreads;
#endif
}

int oracle_max_threads(void) { return default_threads(); }

/*
 * Plain CSR contract ("Interesting ideas" I5: standard CSR, no structural
 * constraint).  Reading taken where the pages are silent: column indices of a
 * row are strictly increasing (sorted, no duplicates).
 * Returns 0 when valid, a negative code naming the first violation otherwise.
 */
int oracle_csr_check(int M, int K, int64_t nnz, const int32_t *ro, const int32_t *ci) {
    if (M < 0 || K < 0 || nnz < 0) return -1;
    if (ro[0] != 0) return -2;
    for (int r = 0; r < M; ++r)
        if (ro[r + 1] < ro[r]) return -3;
    if ((int64_t)ro[M] != nnz) return -4;
    for (int r = 0; r < M; ++r) {
        for (int32_t p = ro[r]; p < ro[r + 1]; ++p) {
            if (ci[p] < 0 || ci[p] >= K) return -5;
            if (p > ro[r] && ci[p] <= ci[p - 1]) return -6;
        }
    }
    return 0;
}

/*
 * SpMM (summary card, "Summary"): C = A · B with A sparse M×K in CSR and B
 * dense K×N row-major.  C[r][j] = sum over the nonzeros p of row r of
 * a_p · B[col_p][j].  C is overwritten.
 */
void oracle_spmm(int M, int K, int N, const int32_t *ro, const int32_t *ci, const double *a,
                 const double *B, int64_t ldb, double *C, int64_t ldc, int nthreads) {
    (void)K;
    set_threads(nthreads);
#pragma omp parallel for schedule(dynamic, 16)
    for (int r = 0; r < M; ++r) {
        double *c = C + (int64_t)r * ldc;
        for (int j = 0; j < N; ++j) c[j] = 0.0;
        for (int32_t p = ro[r]; p < ro[r + 1]; ++p) {
            const double ap = a[p];
            const double *b = B + (int64_t)ci[p] * ldb;
            for (int j = 0; j < N; ++j) c[j] += ap * b[j];
        }
    }
}

/*
 * SDDMM in the specialised form the pages describe ("Interesting ideas" I3:
 * no element-wise scaling by A's values, and the second operand used
 * transposed): for every nonzero p = (r, col_p) of the mask,
 *     out[p] = sum_j X[r][j] · Y[col_p][j],
 * X dense M×D, Y dense K×D, both row-major.  out follows the mask's CSR order.
 */
void oracle_sddmm(int M, int K, int D, const int32_t *ro, const int32_t *ci, const double *X,
                  int64_t ldx, const double *Y, int64_t ldy, double *out, int nthreads) {
    (void)K;
    set_threads(nthreads);
#pragma omp parallel for schedule(dynamic, 16)
    for (int r = 0; r < M; ++r) {
        const double *x = X + (int64_t)r * ldx;
        for (int32_t p = ro[r]; p < ro[r + 1]; ++p) {
            const double *y = Y + (int64_t)ci[p] * ldy;
            double s = 0.0;
            for (int j = 0; j < D; ++j) s += x[j] * y[j];
            out[p] = s;
        }
    }
}

/*
 * General SDDMM, the extension the pages call easy to add ("Interesting
 * ideas" I3): out[p] = a_p^scale · sum_j X[r][j] · Yop[col_p][j], where
 * Yop = Y (K×D, "transposed operand", y_transposed = 1) or Yop = Yᵀ for Y
 * given D×K (y_transposed = 0), and the scaling by the mask's values a_p
 * is applied when scale_by_values = 1.
 */
void oracle_sddmm_general(int M, int K, int D, const int32_t *ro, const int32_t *ci,
                          const double *a, int scale_by_values, const double *X, int64_t ldx,
                          const double *Y, int64_t ldy, int y_transposed, double *out,
                          int nthreads) {
    (void)K;
    set_threads(nthreads);
#pragma omp parallel for schedule(dynamic, 16)
    for (int r = 0; r < M; ++r) {
        const double *x = X + (int64_t)r * ldx;
        for (int32_t p = ro[r]; p < ro[r + 1]; ++p) {
            double s = 0.0;
            for (int j = 0; j < D; ++j) {
                double y = y_transposed ? Y[(int64_t)ci[p] * ldy + j] : Y[(int64_t)j * ldy + ci[p]];
                s += x[j] * y;
            }
            out[p] = scale_by_values ? a[p] * s : s;
        }
    }
}

/*
 * Row swizzle ("Interesting ideas" I4: load balancing kept apart from how the
 * work is split).  Reading: the processing order lists rows by decreasing
 * length, ties by increasing row index, so the permutation is unique.  With
 * seg_rows > 0 the order is built independently inside each run of seg_rows
 * consecutive rows (the diagonal blocks of a batched, block-diagonal
 * matrix); seg_rows <= 0 means one run covering all M rows.
 */
static const int32_t *g_ro_for_sort;

static int cmp_rows(const void *pa, const void *pb) {
    int32_t a = *(const int32_t *)pa, b = *(const int32_t *)pb;
    int32_t la = g_ro_for_sort[a + 1] - g_ro_for_sort[a];
    int32_t lb = g_ro_for_sort[b + 1] - g_ro_for_sort[b];
    if (la != lb) return la > lb ? -1 : 1; /* longer rows first */
    return a < b ? -1 : (a > b ? 1 : 0);   /* ties: lower row index first */
}

void oracle_row_swizzle(int M, int seg_rows, const int32_t *ro, int32_t *perm) {
    if (seg_rows <= 0 || seg_rows > M) seg_rows = M;
    for (int r = 0; r < M; ++r) perm[r] = r;
    g_ro_for_sort = ro;
    for (int s = 0; s < M; s += seg_rows) {
        int n = (M - s < seg_rows) ? (M - s) : seg_rows;
        qsort(perm + s, (size_t)n, sizeof(int32_t), cmp_rows);
    }
    g_ro_for_sort = NULL;
}

/*
 * CSR transpose by counting sort: Aᵀ (K×M) in CSR, needed for the sparse
 * layer's input gradient Aᵀ·dY (the kernels serve "both inference and
 * training", summary card "Summary").  Rows of Aᵀ list their column indices
 * (rows of A) in increasing order; values move unchanged.
 */
void oracle_csr_transpose(int M, int K, const int32_t *ro, const int32_t *ci, const double *a,
                          int32_t *ro_t, int32_t *ci_t, double *a_t) {
    int32_t *fill = (int32_t *)calloc((size_t)K + 1, sizeof(int32_t));
    for (int c = 0; c <= K; ++c) ro_t[c] = 0;
    for (int r = 0; r < M; ++r)
        for (int32_t p = ro[r]; p < ro[r + 1]; ++p) ro_t[ci[p] + 1] += 1;
    for (int c = 0; c < K; ++c) ro_t[c + 1] += ro_t[c];
    for (int r = 0; r < M; ++r) {
        for (int32_t p = ro[r]; p < ro[r + 1]; ++p) {
            int c = ci[p];
            int32_t q = ro_t[c] + fill[c]++;
            ci_t[q] = r;
            a_t[q] = a[p];
        }
    }
    free(fill);
}

/*
 * Row-wise softmax over the stored entries of each CSR row (the missing
 * positions of the mask are excluded):
 *     out[p] = exp(s[p] - m_r) / sum_{q in row r} exp(s[q] - m_r),
 * m_r = max_{q in row r} s[q].  Empty rows produce nothing.
 */
void oracle_csr_softmax(int M, const int32_t *ro, const double *s, double *out, int nthreads) {
    set_threads(nthreads);
#pragma omp parallel for schedule(dynamic, 16)
    for (int r = 0; r < M; ++r) {
        int32_t b = ro[r], e = ro[r + 1];
        if (b == e) continue;
        double m = s[b];
        for (int32_t p = b + 1; p < e; ++p)
            if (s[p] > m) m = s[p];
        double z = 0.0;
        for (int32_t p = b; p < e; ++p) z += exp(s[p] - m);
        for (int32_t p = b; p < e; ++p) out[p] = exp(s[p] - m) / z;
    }
}

/*
 * Round fp64 to bfloat16 bits, round-to-nearest, ties to even, in one step
 * (no intermediate fp32).  bfloat16 keeps 8 significand bits (7 stored) and
 * fp32's exponent range; inputs here are finite and well inside that range.
 */
void oracle_round_to_bf16(int64_t n, const double *x, uint16_t *out) {
    for (int64_t i = 0; i < n; ++i) {
        double v = x[i];
        if (v == 0.0) {
            out[i] = signbit(v) ? 0x8000u : 0x0000u;
            continue;
        }
        int e;
        double m = frexp(fabs(v), &e);           /* |v| = m·2^e, m in [0.5, 1) */
        double scaled = ldexp(m, 8);              /* 8 significant bits above the point */
        double fl = floor(scaled);
        double rem = scaled - fl;
        if (rem > 0.5 || (rem == 0.5 && fmod(fl, 2.0) != 0.0)) fl += 1.0;
        double r = ldexp(fl, e - 8);              /* rounded magnitude */
        float f = (float)r;                       /* exact: 8 significant bits */
        uint32_t u;
        memcpy(&u, &f, sizeof u);
        uint16_t h = (uint16_t)(u >> 16);         /* low 16 bits are zero */
        out[i] = signbit(v) ? (uint16_t)(h | 0x8000u) : h;
    }
}
