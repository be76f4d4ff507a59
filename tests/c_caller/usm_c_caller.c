/*
 * A plain C caller of the library's C ABI (include/usm.h): no C++, no Python.
 *
 * usage: usm_c_caller DIR
 * Reads DIR/problem.bin, checks the CSR with csr_validate, runs
 * row_swizzle_build, csr_spmm and csr_sddmm on the GPU through the CUDA runtime, and writes DIR/C.bin (fp32 M×N) and
 * DIR/out.bin (fp32 nnz).  problem.bin: int32 M, K, N, D, nnz; then
 * int32 row_offsets[M+1], int32 col_indices[nnz], float values[nnz],
 * float B[K·N], float X[M·D], float Y[K·D] (all row-major).
 * Exit status 0 on success; a message on stderr otherwise.
 */
#include <stdio.h>
#include <stdlib.h>

#include <cuda_runtime_api.h>

#include "usm.h"

static int fail(const char *what, int code) {
    fprintf(stderr, "usm_c_caller: %s failed (%d: %s)\n", what, code, usm_status_string(code));
    return 1;
}

static void *read_all(const char *path, long *size) {
    FILE *f = fopen(path, "rb");
    if (!f) return NULL;
    fseek(f, 0, SEEK_END);
    *size = ftell(f);
    fseek(f, 0, SEEK_SET);
    void *buf = malloc((size_t)*size);
    if (buf && fread(buf, 1, (size_t)*size, f) != (size_t)*size) {
        free(buf);
        buf = NULL;
    }
    fclose(f);
    return buf;
}

static int write_all(const char *path, const void *data, size_t bytes) {
    FILE *f = fopen(path, "wb");
    if (!f) return 0;
    const size_t n = fwrite(data, 1, bytes, f);
    fclose(f);
    return n == bytes;
}

/* Device buffer of `bytes` (at least 16), filled from `host` unless NULL. */
static void *to_device(const void *host, size_t bytes) {
    void *d = NULL;
    if (cudaMalloc(&d, bytes ? bytes : 16) != cudaSuccess) return NULL;
    if (host && bytes && cudaMemcpy(d, host, bytes, cudaMemcpyHostToDevice) != cudaSuccess) return NULL;
    return d;
}

int main(int argc, char **argv) {
    if (argc != 2) {
        fprintf(stderr, "usage: %s DIR\n", argv[0]);
        return 2;
    }
    char path[4096];
    long size = 0;
    snprintf(path, sizeof path, "%s/problem.bin", argv[1]);
    const int *hdr = (const int *)read_all(path, &size);
    if (!hdr || size < 5 * (long)sizeof(int)) {
        fprintf(stderr, "usm_c_caller: cannot read %s\n", path);
        return 1;
    }
    const int M = hdr[0], K = hdr[1], N = hdr[2], D = hdr[3], nnz = hdr[4];
    const int *ro = hdr + 5;
    const int *ci = ro + (M + 1);
    const float *vals = (const float *)(ci + nnz);
    const float *B = vals + nnz;
    const float *X = B + (size_t)K * N;
    const float *Y = X + (size_t)M * D;

    int *d_ro = to_device(ro, sizeof(int) * (size_t)(M + 1));
    int *d_ci = to_device(ci, sizeof(int) * (size_t)nnz);
    float *d_vals = to_device(vals, sizeof(float) * (size_t)nnz);
    float *d_B = to_device(B, sizeof(float) * (size_t)K * N);
    float *d_X = to_device(X, sizeof(float) * (size_t)M * D);
    float *d_Y = to_device(Y, sizeof(float) * (size_t)K * D);
    float *d_C = to_device(NULL, sizeof(float) * (size_t)M * N);
    float *d_out = to_device(NULL, sizeof(float) * (size_t)nnz);
    int *d_perm = to_device(NULL, sizeof(int) * (size_t)M);
    if (!d_ro || !d_ci || !d_vals || !d_B || !d_X || !d_Y || !d_C || !d_out || !d_perm)
        return fail("cudaMalloc/cudaMemcpy", USM_ERR_CUDA);

    cudaStream_t stream;
    if (cudaStreamCreate(&stream) != cudaSuccess) return fail("cudaStreamCreate", USM_ERR_CUDA);

    int *d_check = to_device(NULL, sizeof(int) * USM_CSR_VALIDATE_INTS);
    if (!d_check) return fail("cudaMalloc", USM_ERR_CUDA);
    int st = csr_validate(M, K, nnz, d_ro, d_ci, d_check, stream);
    if (st != USM_OK) return fail("csr_validate", st);
    int check[2];
    if (cudaMemcpyAsync(check, d_check, sizeof check, cudaMemcpyDeviceToHost, stream) != cudaSuccess ||
        cudaStreamSynchronize(stream) != cudaSuccess)
        return fail("csr_validate result", USM_ERR_CUDA);
    if (check[0] != USM_CSR_VALID) {
        fprintf(stderr, "usm_c_caller: CSR violates the contract (code %d at %d)\n", check[0], check[1]);
        return 1;
    }

    const size_t swz_bytes = row_swizzle_workspace_bytes(M, K);
    void *d_swz = to_device(NULL, swz_bytes);
    st = row_swizzle_build(M, K, 0, d_ro, d_perm, d_swz, swz_bytes, stream);
    if (st != USM_OK) return fail("row_swizzle_build", st);

    st = csr_spmm(M, K, N, nnz, d_ro, d_ci, d_vals, d_perm, 0, d_B, N, d_C, N, USM_F32, stream);
    if (st != USM_OK) return fail("csr_spmm", st);

    const size_t ws_bytes = csr_sddmm_workspace_bytes(M, K, D, nnz, USM_F32);
    void *d_ws = to_device(NULL, ws_bytes);
    st = csr_sddmm(M, K, D, nnz, d_ro, d_ci, d_perm, 0, d_X, D, d_Y, D, d_out, USM_F32, USM_F32,
                   ws_bytes ? d_ws : NULL, ws_bytes, stream);
    if (st != USM_OK) return fail("csr_sddmm", st);

    st = usm_poll_status(stream);  /* synchronises the stream */
    if (st != USM_OK) return fail("device status", st);

    float *C = malloc(sizeof(float) * (size_t)M * N + 16);
    float *out = malloc(sizeof(float) * (size_t)nnz + 16);
    if (!C || !out) return fail("malloc", USM_ERR_INVALID_ARG);
    if (cudaMemcpy(C, d_C, sizeof(float) * (size_t)M * N, cudaMemcpyDeviceToHost) != cudaSuccess ||
        cudaMemcpy(out, d_out, sizeof(float) * (size_t)nnz, cudaMemcpyDeviceToHost) != cudaSuccess)
        return fail("cudaMemcpy back", USM_ERR_CUDA);
    snprintf(path, sizeof path, "%s/C.bin", argv[1]);
    if (!write_all(path, C, sizeof(float) * (size_t)M * N)) return fail("write C.bin", USM_ERR_INVALID_ARG);
    snprintf(path, sizeof path, "%s/out.bin", argv[1]);
    if (!write_all(path, out, sizeof(float) * (size_t)nnz)) return fail("write out.bin", USM_ERR_INVALID_ARG);
    return 0;
}
