// gemm_common.cuh -- tile scheduling and the split-K epilogue shared by the
// W12 GEMM kernels.
//
// Work is cut into tiles (column block nb, k split kc), tile t = kc*NB + nb.
// CTA c owns the contiguous range of tiles [t0, t1) (balanced to within one
// tile).  With one split a tile writes y directly.  With several, it writes
// fp32 partials[kc][m][n], bumps the arrival counter of its column block,
// and the CTA that arrives last sums the splits in kc order (so results are
// the same bits on every run), writes y and sets the counter back to zero.
#pragma once

#include <cuda_bf16.h>

#include "device_common.cuh"
#include "w12_internal.h"

namespace w12 {

__device__ __forceinline__ void tile_range(int64_t T, int64_t &t0, int64_t &t1) {
    const int64_t G = gridDim.x, c = blockIdx.x;
    const int64_t per = T / G, rem = T % G;
    t0 = c * per + (c < rem ? c : rem);
    t1 = t0 + per + (c < rem ? 1 : 0);
}

__device__ __forceinline__ void store_y(const GemmArgs &a, int64_t m, int64_t n, float v) {
    if (a.y_dtype == W12_F32) {
        static_cast<float *>(a.y)[m * a.N + n] = v;
    } else {
        static_cast<__nv_bfloat16 *>(a.y)[m * a.N + n] = __float2bfloat16_rn(v);
    }
}

// Store one finished output of split kc: straight to y, or to the partials.
__device__ __forceinline__ void emit(const GemmArgs &a, int64_t kc, int64_t m, int64_t n, float v) {
    if (a.nks == 1)
        store_y(a, m, n, v);
    else
        a.partial[(kc * a.M + m) * a.N + n] = v;
}

// Called by every thread of the CTA after its tile's outputs are emitted.
__device__ __forceinline__ void finish_tile(const GemmArgs &a, int64_t nb, int *s_last) {
    if (a.nks == 1) return;
    __threadfence();
    __syncthreads();
    if (threadIdx.x == 0) *s_last = (atomicAdd(&a.counters[nb], 1u) == uint32_t(a.nks - 1));
    __syncthreads();
    if (*s_last) {
        __threadfence();
        const int64_t cpt = a.cols_per_tile;
        for (int64_t o = threadIdx.x; o < cpt * a.M; o += blockDim.x) {
            const int64_t m = o / cpt, n = nb * cpt + o % cpt;
            if (n >= a.N) continue;
            float s = 0.f;
            for (int kc = 0; kc < a.nks; ++kc) s += __ldcg(&a.partial[(kc * a.M + m) * a.N + n]);
            store_y(a, m, n, s);
        }
        if (threadIdx.x == 0) a.counters[nb] = 0u;
    }
}

}  // namespace w12
