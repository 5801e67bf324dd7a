// gemm_common.cuh -- output stores, the balanced stream-K partition and the
// stream-K fix-up shared by the batched GEMM kernels.
#pragma once

#include <cuda_bf16.h>

#include "device_common.cuh"
#include "w12_internal.h"

namespace w12 {

// Barrier over the threads taking part in the epilogue: the whole CTA, or
// the first nthreads of it (named barrier 1) when a producer warp is apart.
__device__ __forceinline__ void epi_sync(int nthreads) {
    if (nthreads == int(blockDim.x))
        __syncthreads();
    else
        asm volatile("bar.sync 1, %0;" ::"r"(nthreads) : "memory");
}

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

// Stream-K fix-up of the batched kernels.  Column tile nb of a product
// covers the global units [first, first + steps) (the product's units start
// at ubase); U units are spread over the grid as above.  Every CTA that
// covered a piece of the tile stored the piece's partial sums (all m < M,
// n < N) in the slot of the piece's first unit,
//   partial[((u - ubase) * M + m) * cpt + c],
// and adds the piece's unit count to counters[nb].  The CTA that brings the
// count to `steps` sums the pieces' slots in unit order (the same bits on
// every call), writes y, and sets the counter back to zero.  Slots need no
// clearing: only slots that were written are read.
__device__ __forceinline__ void streamk_fixup_raw(uint32_t *counters, const float *partial, int first,
                                                  int ubase, int steps, int U, int M, int N, void *y,
                                                  int y_dtype, int cpt, int nb, int count, int *s_last,
                                                  int tid, int nthreads) {
    __threadfence();
    epi_sync(nthreads);
    if (tid == 0) {
        const uint32_t old = atomicAdd(&counters[nb], uint32_t(count));
        *s_last = (int(old) + count == steps);
    }
    epi_sync(nthreads);
    if (*s_last) {
        __threadfence();
        const int G = int(gridDim.x), per = U / G, rem = U % G;
        const int c_first = sk_cta_of(first, per, rem);
        const int q4 = cpt / 4, total = M * q4;  // float4 groups of a slot
        const size_t slot_floats = size_t(M) * size_t(cpt);
        constexpr int kB = 4;  // groups per thread in flight
        for (int o0 = tid; o0 < total; o0 += kB * nthreads) {
            float4 acc[kB];
            for (int c = c_first;; ++c) {
                const int us = max(first, sk_unit_begin(c, per, rem));
                if (us >= first + steps) break;
                const float *slot = partial + size_t(us - ubase) * slot_floats;
                float4 v[kB];
#pragma unroll
                for (int j = 0; j < kB; ++j) {
                    const int o = o0 + j * nthreads;
                    v[j] = make_float4(0.f, 0.f, 0.f, 0.f);
                    if (o < total)
                        v[j] = __ldcg(reinterpret_cast<const float4 *>(slot + size_t(o / q4) * cpt) + o % q4);
                }
#pragma unroll
                for (int j = 0; j < kB; ++j) {
                    if (c == c_first) {
                        acc[j] = v[j];
                    } else {
                        acc[j].x += v[j].x;
                        acc[j].y += v[j].y;
                        acc[j].z += v[j].z;
                        acc[j].w += v[j].w;
                    }
                }
            }
#pragma unroll
            for (int j = 0; j < kB; ++j) {
                const int o = o0 + j * nthreads;
                if (o >= total) break;
                const int m = o / q4, n0 = nb * cpt + 4 * (o % q4);
                const float r[4] = {acc[j].x, acc[j].y, acc[j].z, acc[j].w};
#pragma unroll
                for (int e = 0; e < 4; ++e)
                    if (n0 + e < N) store_out(y, y_dtype, N, m, n0 + e, r[e]);
            }
        }
        if (tid == 0) counters[nb] = 0u;
    }
    epi_sync(nthreads);
}

}  // namespace w12
