// gemm_common.cuh -- output stores and the balanced stream-K partition
// shared by the batched GEMM kernels.
#pragma once

#include <cuda_bf16.h>

#include "device_common.cuh"
#include "w12_internal.h"

namespace w12 {


// Store one output of a batched GEMV (y row-major [M][N], fp32 or bf16).
__device__ __forceinline__ void store_out(void *y, int y_dtype, int64_t N, int64_t m, int64_t n, float v) {
    if (y_dtype == W12_F32)
        static_cast<float *>(y)[m * N + n] = v;
    else
        static_cast<__nv_bfloat16 *>(y)[m * N + n] = __float2bfloat16_rn(v);
}

// Balanced partition of U stream-K units over the grid: CTA c takes the
// units [sk_unit_begin(c), sk_unit_begin(c + 1)).
__device__ __forceinline__ int sk_unit_begin(int c, int per, int rem) { return c * per + min(c, rem); }

__device__ __forceinline__ int sk_cta_of(int u, int per, int rem) {
    const int big = rem * (per + 1);
    return u < big ? u / (per + 1) : rem + (u - big) / per;
}

}  // namespace w12
