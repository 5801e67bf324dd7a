// kernels_verify.cu -- greedy draft-block verification on logits.
//
// Each (row, split) work item scans a contiguous slice of one logits row with
// 16-byte loads, keeping the largest packed key (order_key(value) << 32 |
// ~index: NaN above all numbers, -0 == +0, lowest index on ties), reduces it
// over the CTA and stores it in the workspace.  The CTA that finishes last
// (arrival counter, no spin-wait) folds the splits per row and runs the
// acceptance rule.  HBM-bound: one pass over R*T*V logits.
#include <cuda_runtime.h>

#include "verify_common.cuh"
#include "w12_internal.h"

namespace w12 {

namespace {

constexpr int kThreads = 256;

__device__ __forceinline__ unsigned long long kmax(unsigned long long a, unsigned long long b) {
    return a > b ? a : b;
}

template <int DT>
__device__ __forceinline__ float logit_at(const void *p, int64_t i) {
    if (DT == W12_F32) return static_cast<const float *>(p)[i];
    return bf16_bits_to_float(static_cast<const uint16_t *>(p)[i]);
}

template <int DT>
__global__ void __launch_bounds__(kThreads) verify_kernel(const VerifyArgs a, int vec_ok) {
    __shared__ unsigned long long s_red[kThreads / 32];
    __shared__ int s_last;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int64_t items = a.rows * a.splits;
    for (int64_t it = blockIdx.x; it < items; it += gridDim.x) {
        const int64_t row = it / a.splits, sp = it % a.splits;
        const int64_t c0 = sp * a.chunk;
        const int64_t c1 = min(a.V, c0 + a.chunk);
        const int64_t base = row * a.V;
        unsigned long long best = 0ull;
        if (vec_ok) {
            constexpr int VEC = (DT == W12_F32) ? 4 : 8;
            for (int64_t i = c0 + int64_t(threadIdx.x) * VEC; i < c1; i += int64_t(kThreads) * VEC) {
                const uint4 v = ldg_stream(static_cast<const char *>(a.logits) +
                                           (base + i) * (DT == W12_F32 ? 4 : 2));
                const uint32_t w[4] = {v.x, v.y, v.z, v.w};
                if (DT == W12_F32) {
#pragma unroll
                    for (int q = 0; q < 4; ++q)
                        best = kmax(best, pack_key(__uint_as_float(w[q]), uint32_t(i + q)));
                } else {
#pragma unroll
                    for (int q = 0; q < 4; ++q) {
                        best = kmax(best, pack_key(bf16_bits_to_float(w[q] & 0xFFFFu), uint32_t(i + 2 * q)));
                        best = kmax(best, pack_key(bf16_bits_to_float(w[q] >> 16), uint32_t(i + 2 * q + 1)));
                    }
                }
            }
        } else {
            for (int64_t i = c0 + threadIdx.x; i < c1; i += kThreads)
                best = kmax(best, pack_key(logit_at<DT>(a.logits, base + i), uint32_t(i)));
        }
#pragma unroll
        for (int off = 16; off >= 1; off >>= 1) best = kmax(best, __shfl_xor_sync(0xFFFFFFFFu, best, off));
        if (lane == 0) s_red[warp] = best;
        __syncthreads();
        if (threadIdx.x == 0) {
            unsigned long long b = s_red[0];
            for (int w2 = 1; w2 < kThreads / 32; ++w2) b = kmax(b, s_red[w2]);
            a.partial[sp * a.rows + row] = b;
        }
        __syncthreads();
    }
    __threadfence();
    __syncthreads();
    if (threadIdx.x == 0) s_last = (atomicAdd(a.counter, 1u) == gridDim.x - 1);
    __syncthreads();
    if (s_last) {
        __threadfence();
        verify_from_keys(a.partial, a.splits, a.rows, a.R, a.T, a.draft, a.accept_len, a.next_tok,
                         a.gbuf);
        if (threadIdx.x == 0) *a.counter = 0u;
    }
}

}  // namespace

int launch_verify(const VerifyArgs &a, int grid, void *stream) {
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    const int esize = a.dtype == W12_F32 ? 4 : 2;
    const int vec = 16 / esize;
    const int vec_ok = ((a.V * esize) % 16 == 0) && (a.chunk % vec == 0) &&
                       ((reinterpret_cast<uintptr_t>(a.logits) & 15u) == 0);
    if (a.dtype == W12_F32)
        verify_kernel<W12_F32><<<unsigned(grid), kThreads, 0, s>>>(a, vec_ok);
    else
        verify_kernel<W12_BF16><<<unsigned(grid), kThreads, 0, s>>>(a, vec_ok);
    return cudaGetLastError() == cudaSuccess ? W12_OK : W12_ERR_CUDA;
}

}  // namespace w12
