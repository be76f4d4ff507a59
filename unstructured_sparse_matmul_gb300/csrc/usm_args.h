// Arguments the kernels receive by value (plain data, shared by the host
// launch code and the device code).
#pragma once

#include <stdint.h>

namespace usm {

struct SpmmArgs {
    int M, K, N, nnz;
    const int* row_offsets;
    const int* col_indices;
    const void* values;
    const int* perm;  // may be null (identity order)
    int seg_rows;     // rows per diagonal block of the schedule (> 0)
    float* C;
    long long ldc;
    int* status;
    int tiles_per_block = 0;  // row tiles per diagonal block (set by the launcher)
};

struct SddmmArgs {
    int M, K, D, nnz;
    const int* row_offsets;
    const int* col_indices;
    const int* perm;
    int seg_rows;
    const void* X;
    long long ldx;
    void* out;           // final output (single strip) or fp32 partials (several strips)
    long long out_stride;  // elements between strips of partials
    int out_bf16;        // final output element type is bf16
    int rows_per_warp;
    int* status;
    const void* scale;   // null, or the mask's values: out[p] is multiplied by scale[p]
    int scale_bf16;      // scale elements are bf16 (else fp32)
    int tiles_per_block = 0;  // row tiles per diagonal block (set by the launcher)
};

}  // namespace usm
