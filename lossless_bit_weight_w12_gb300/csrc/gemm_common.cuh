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

// Barrier over the threads taking part in the epilogue: the whole CTA, or
// the first nthreads of it (named barrier 1) when a producer warp is apart.
__device__ __forceinline__ void epi_sync(int nthreads) {
    if (nthreads == int(blockDim.x))
        __syncthreads();
    else
        asm volatile("bar.sync 1, %0;" ::"r"(nthreads) : "memory");
}

// Called by every epilogue thread (tid < nthreads) after its tile's outputs
// are emitted.
__device__ __forceinline__ void finish_tile(const GemmArgs &a, int64_t nb, int *s_last, int tid,
                                            int nthreads) {
    if (a.nks == 1) return;
    __threadfence();
    epi_sync(nthreads);
    if (tid == 0) *s_last = (atomicAdd(&a.counters[nb], 1u) == uint32_t(a.nks - 1));
    epi_sync(nthreads);
    if (*s_last) {
        __threadfence();
        const int64_t cpt = a.cols_per_tile;
        for (int64_t o = tid; o < cpt * a.M; o += nthreads) {
            const int64_t m = o / cpt, n = nb * cpt + o % cpt;
            if (n >= a.N) continue;
            float s = 0.f;
            for (int kc = 0; kc < a.nks; ++kc) s += __ldcg(&a.partial[(kc * a.M + m) * a.N + n]);
            store_y(a, m, n, s);
        }
        if (tid == 0) a.counters[nb] = 0u;
    }
    epi_sync(nthreads);  // s_last is reused by the next tile
}

// Store one output of a batched GEMV (y row-major [M][N], fp32 or bf16).
__device__ __forceinline__ void store_out(void *y, int y_dtype, int64_t N, int64_t m, int64_t n, float v) {
    if (y_dtype == W12_F32)
        static_cast<float *>(y)[m * N + n] = v;
    else
        static_cast<__nv_bfloat16 *>(y)[m * N + n] = __float2bfloat16_rn(v);
}

// Stream-K fix-up on explicit buffers (the batched GEMV): same protocol as
// streamk_fixup below; slots are partial[((nb * steps + ks) * M + m) * cpt + c].
__device__ __forceinline__ void streamk_fixup_raw(uint32_t *counters, float *partial, int64_t steps,
                                                  int M, int64_t N, void *y, int y_dtype, int64_t cpt,
                                                  int64_t nb, int64_t count, int *s_last, int tid,
                                                  int nthreads) {
    __threadfence();
    epi_sync(nthreads);
    if (tid == 0) {
        const uint32_t old = atomicAdd(&counters[nb], uint32_t(count));
        *s_last = (int64_t(old) + count == steps);
    }
    epi_sync(nthreads);
    if (*s_last) {
        __threadfence();
        for (int64_t o = tid; o < cpt * M; o += nthreads) {
            const int64_t m = o / cpt, c = o % cpt, n = nb * cpt + c;
            float s = 0.f;
            for (int64_t ks = 0; ks < steps; ++ks) {
                float *slot = &partial[((nb * steps + ks) * M + m) * cpt + c];
                s += __ldcg(slot);
                *slot = 0.f;
            }
            if (n < N) store_out(y, y_dtype, N, m, n, s);
        }
        if (tid == 0) counters[nb] = 0u;
    }
    epi_sync(nthreads);
}

// Stream-K fix-up of column tile nb after a CTA covered `count` of its
// `steps` stages and stored its partial sums in slot (nb, first stage).  The
// CTA that completes the tile sums the slots in stage order (deterministic),
// writes y, and zeroes the slots and the counter for the next call.
__device__ __forceinline__ void streamk_fixup(const GemmArgs &a, int64_t nb, int64_t count,
                                              int *s_last, int tid, int nthreads) {
    __threadfence();
    epi_sync(nthreads);
    if (tid == 0) {
        const uint32_t old = atomicAdd(&a.counters[nb], uint32_t(count));
        *s_last = (int64_t(old) + count == a.steps);
    }
    epi_sync(nthreads);
    if (*s_last) {
        __threadfence();
        const int64_t cpt = a.cols_per_tile;
        for (int64_t o = tid; o < cpt * a.M; o += nthreads) {
            const int64_t m = o / cpt, c = o % cpt, n = nb * cpt + c;
            float s = 0.f;
            for (int64_t ks = 0; ks < a.steps; ++ks) {
                float *slot = &a.partial[((nb * a.steps + ks) * a.M + m) * cpt + c];
                s += __ldcg(slot);
                *slot = 0.f;
            }
            if (n < a.N) store_y(a, m, n, s);
        }
        if (tid == 0) a.counters[nb] = 0u;
    }
    epi_sync(nthreads);
}

}  // namespace w12
