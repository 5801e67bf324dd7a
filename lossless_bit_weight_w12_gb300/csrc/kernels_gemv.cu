// kernels_gemv.cu -- W12 GEMV for M <= 4: CUDA-core FFMA, warp-shuffle reduce.
//
// At M = 1 a skinny decode step is a pure weight stream (SpecPilot summary,
// airadar.tv English edition, first paragraph: a single request reads all
// target weights per step), so the kernel is built around HBM: each lane
// streams 16-byte vectors of the three planes (32 consecutive k of one
// column, L1 bypassed), rebuilds them in registers (rebuild32: ~2.5 integer
// ops per weight), and feeds packed fp32x2 FMAs (Blackwell FFMA2, 0.5 issue
// slots per weight).  A warp covers 1024 k of CPW columns per step; the lane
// partial sums are combined by a transposing shuffle reduction (log2(32)
// shuffles in total for all CPW*MT values instead of 5 per value).
//
// Layout of one tile: 8 warps x CPW columns, k range [kc*kchunk, +kchunk).
#include <cuda_runtime.h>

#include "gemm_common.cuh"

namespace w12 {

namespace {

constexpr int kThreads = 256;

__device__ __forceinline__ float2 unpack_bf16x2(uint32_t p) {
    return make_float2(__uint_as_float(p << 16), __uint_as_float(p & 0xFFFF0000u));
}

__device__ __forceinline__ uint32_t word_of(const uint4 &v, int c) {
    return c == 0 ? v.x : c == 1 ? v.y : c == 2 ? v.z : v.w;
}

// Sum NV values across the warp.  Afterwards the lanes whose low (5 - log2 NV)
// bits are zero hold the totals: lane L holds value L >> (5 - log2 NV).
template <int NV>
__device__ __forceinline__ void transpose_reduce(float (&v)[NV], int lane) {
    constexpr unsigned kFull = 0xFFFFFFFFu;
    int nv = NV;
#pragma unroll
    for (int off = 16; off >= 1; off >>= 1) {
        if (nv > 1) {
            const int half = nv / 2;
            const bool upper = (lane & off) != 0;
#pragma unroll
            for (int i = 0; i < NV / 2; ++i) {
                if (i < half) {
                    const float send = upper ? v[i] : v[i + half];
                    const float keep = upper ? v[i + half] : v[i];
                    v[i] = keep + __shfl_xor_sync(kFull, send, off);
                }
            }
            nv = half;
        } else {
            v[0] += __shfl_xor_sync(kFull, v[0], off);
        }
    }
}

template <int NV>
struct Log2 {
    static constexpr int value = NV <= 1 ? 0 : 1 + Log2<NV / 2>::value;
};
template <>
struct Log2<1> {
    static constexpr int value = 0;
};

template <int CPW, int MT>
__global__ void __launch_bounds__(kThreads, 2) gemv_kernel(const GemmArgs a) {
    __shared__ int s_last;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    int64_t t0, t1;
    tile_range(a.T, t0, t1);
    for (int64_t t = t0; t < t1; ++t) {
        const int64_t kc = t / a.NB, nb = t % a.NB;
        const int64_t kbeg = kc * a.kchunk;
        const int64_t kend = min(a.K, kbeg + a.kchunk);
        const int64_t col0 = nb * a.cols_per_tile + int64_t(warp) * CPW;

        float2 acc[CPW][MT];
#pragma unroll
        for (int j = 0; j < CPW; ++j)
#pragma unroll
            for (int m = 0; m < MT; ++m) acc[j][m] = make_float2(0.f, 0.f);

        for (int64_t k0 = kbeg; k0 < kend; k0 += 1024) {
            const int64_t kl = k0 + int64_t(lane) * 32;
            if (kl < kend) {
                // issue every load of the step before any arithmetic
                uint4 h[CPW], l[CPW], e[CPW];
                uint32_t m0[CPW], m1[CPW];
#pragma unroll
                for (int j = 0; j < CPW; ++j) {
                    const int64_t n = col0 + j;
                    if (n < a.N) {
                        const int64_t wo = n * a.KW + (kl >> 3);
                        h[j] = ldg_stream(a.H + wo);
                        l[j] = ldg_stream(a.L + wo);
                        e[j] = ldg_stream(a.E + wo);
                        const int64_t g = n * a.KG + (kl >> 7);
                        m0[j] = ldg_u32(a.meta + g);
                        m1[j] = ldg_u32(a.meta + g + 1);
                    }
                }
                uint4 xv[MT][4];
#pragma unroll
                for (int m = 0; m < MT; ++m) {
#pragma unroll
                    for (int q = 0; q < 4; ++q) {
                        xv[m][q] = (m < a.M) ? ldg_v4(a.x + int64_t(m) * a.K + kl + 8 * q)
                                             : make_uint4(0u, 0u, 0u, 0u);
                    }
                }
                // MT == 1: widen x once per step and reuse it for all CPW columns;
                // MT > 1: widen at the point of use to keep register pressure down.
                float2 xf[MT == 1 ? 16 : 1];
                if (MT == 1) {
#pragma unroll
                    for (int i = 0; i < 16; ++i) xf[MT == 1 ? i : 0] = unpack_bf16x2(word_of(xv[0][i >> 2], i & 3));
                }
#pragma unroll
                for (int j = 0; j < CPW; ++j) {
                    if (col0 + j < a.N) {
                        uint32_t w[16];
                        rebuild32(h[j], l[j], e[j], (m0[j] & 0xFFu) * 0x00800080u, w);
                        if ((m0[j] >> 8) != (m1[j] >> 8))
                            patch_escapes(w, m0[j], m1[j], uint32_t(kl & 127), a.esc, a.n_esc,
                                          a.err);
#pragma unroll
                        for (int i = 0; i < 16; ++i) {
                            const float2 wf = unpack_bf16x2(w[i]);
#pragma unroll
                            for (int m = 0; m < MT; ++m) {
                                const float2 xi = (MT == 1) ? xf[MT == 1 ? i : 0]
                                                            : unpack_bf16x2(word_of(xv[m][i >> 2], i & 3));
                                acc[j][m] = __ffma2_rn(wf, xi, acc[j][m]);
                            }
                        }
                    }
                }
            }
        }

        constexpr int NV = CPW * MT;
        float v[NV];
#pragma unroll
        for (int j = 0; j < CPW; ++j)
#pragma unroll
            for (int m = 0; m < MT; ++m) v[j * MT + m] = acc[j][m].x + acc[j][m].y;
        transpose_reduce<NV>(v, lane);
        constexpr int kShift = 5 - Log2<NV>::value;
        if ((lane & ((1 << kShift) - 1)) == 0) {
            const int vi = lane >> kShift;
            const int j = vi / MT, m = vi % MT;
            const int64_t n = col0 + j;
            if (n < a.N && m < a.M) emit(a, kc, m, n, v[0]);
        }
        finish_tile(a, nb, &s_last);
    }
}

template <int CPW, int MT>
int launch_t(const GemmPlan &p, const GemmArgs &a, cudaStream_t s) {
    gemv_kernel<CPW, MT><<<unsigned(p.grid), kThreads, 0, s>>>(a);
    return cudaGetLastError() == cudaSuccess ? W12_OK : W12_ERR_CUDA;
}

template <int CPW, int MT>
int occ_t(int *blocks) {
    return cudaOccupancyMaxActiveBlocksPerMultiprocessor(blocks, gemv_kernel<CPW, MT>, kThreads, 0) ==
                   cudaSuccess
               ? W12_OK
               : W12_ERR_CUDA;
}

}  // namespace

// variant -> (columns per warp, tokens); the set the planner chooses from.
#define W12_GEMV_VARIANTS(X) X(0, 1, 1) X(1, 2, 1) X(2, 4, 1) X(3, 1, 2) X(4, 2, 2) X(5, 1, 4)

int launch_gemv(const GemmPlan &p, const GemmArgs &a, void *stream) {
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    switch (p.variant) {
#define X(id, cpw, mt) \
    case id:           \
        return launch_t<cpw, mt>(p, a, s);
        W12_GEMV_VARIANTS(X)
#undef X
    }
    return W12_ERR_ARG;
}

int gemv_occupancy(int variant, int *blocks) {
    switch (variant) {
#define X(id, cpw, mt) \
    case id:           \
        return occ_t<cpw, mt>(blocks);
        W12_GEMV_VARIANTS(X)
#undef X
    }
    return W12_ERR_ARG;
}

}  // namespace w12
