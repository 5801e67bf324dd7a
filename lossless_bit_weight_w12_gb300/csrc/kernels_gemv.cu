// kernels_gemv.cu -- W12 GEMV for M <= 4: cp.async-pipelined weight stream,
// mixed bf16 x bf16 -> fp32 FMA on the CUDA cores, warp-shuffle reduction.
//
// At M = 1 a skinny decode step is a pure weight stream (SpecPilot summary,
// airadar.tv English edition, first paragraph: a single request reads all the
// target's weights every step), so the kernel is built around HBM:
//  - stream-K: the work is cut into units of one stage (16 columns x 1024 k)
//    and every CTA takes the same number of consecutive units; a column tile
//    cut by a CTA boundary is finished by a deterministic partial-sum fix-up;
//  - each warp owns 2 of a unit's columns and lane l the 32 weights
//    k = 32l .. 32l+31: the lane streams its own 16-byte vectors of the three
//    planes (and its two meta words) with cp.async into private,
//    lane-interleaved shared-memory slots kStages units ahead, so every load
//    is coalesced (a warp reads 512 contiguous bytes per plane and column),
//    the reads back are conflict-free, and a thread only ever waits for its
//    own copies (cp.async.wait_group: no barrier, no spin);
//  - the lane rebuilds its 32 bf16 weights in registers (rebuild32, ~1.75 ALU
//    ops per weight), patches escapes, and multiplies with fma.rn.f32.bf16
//    straight from the bf16 halves of weights and activations;
//  - per tile the lane partial sums are combined by a transposing shuffle
//    reduction.
#include <cuda_runtime.h>

#include "async_common.cuh"
#include "gemm_common.cuh"

namespace w12 {

namespace {

constexpr int kWarps = 8;
constexpr int kThreads = kWarps * 32;
constexpr int kCW = 2;                         // columns per warp
constexpr int kCols = kWarps * kCW;            // columns per unit / tile
constexpr int kStageK = 1024;                  // k per unit
constexpr int kRows = 3 * kCW + 1;             // per warp and slot: 6 plane rows + 1 meta row
constexpr int kRowBytes = 32 * 16;             // one 16-byte chunk per lane

template <int MT>
struct GemvCfg {
    static constexpr int kStages = MT == 1 ? 4 : 3;
    static constexpr int kMinBlocks = MT == 4 ? 1 : 2;
    static constexpr int kSmem = kWarps * kStages * kRows * kRowBytes;
};

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
    static constexpr int value = 1 + Log2<NV / 2>::value;
};
template <>
struct Log2<1> {
    static constexpr int value = 0;
};

template <int MT>
__global__ void __launch_bounds__(kThreads, GemvCfg<MT>::kMinBlocks) gemv_kernel(const GemmArgs a) {
    constexpr int S = GemvCfg<MT>::kStages;
    extern __shared__ __align__(128) unsigned char smem[];
    __shared__ int s_last;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const uint32_t my = smem_addr(smem) + uint32_t(warp * S * kRows * kRowBytes + lane * 16);
    const uint64_t pol = l2_evict_first_policy();
    int64_t u0, u1;
    tile_range(a.T, u0, u1);

    // Unit u covers column tile u / steps and k = (u % steps) * kStageK.  The
    // three positions the loop needs (copy issue S-1 units ahead, activation
    // prefetch one unit ahead, compute) are advanced by increments: no
    // division inside the loop.
    struct Pos {
        int64_t nb, ks;
        __device__ void next(int64_t steps) {
            if (++ks == steps) {
                ks = 0;
                ++nb;
            }
        }
    };
    const int64_t steps = a.steps;
    Pos pc{u0 / steps, u0 % steps};  // compute position

    // Start the copies of the unit at p into slot s (this lane's chunks only).
    auto issue = [&](const Pos &p, int s) {
        const int64_t kl = p.ks * kStageK + 32 * lane;
        if (kl >= a.K) return;
        const uint32_t slot = my + uint32_t(s * kRows * kRowBytes);
#pragma unroll
        for (int j = 0; j < kCW; ++j) {
            const int64_t n = p.nb * kCols + warp * kCW + j;
            if (n < a.N) {
                const int64_t wo = n * a.KW + (kl >> 3);
                cp_async16_stream(slot + (3 * j + 0) * kRowBytes, a.H + wo, pol);
                cp_async16_stream(slot + (3 * j + 1) * kRowBytes, a.L + wo, pol);
                cp_async16_stream(slot + (3 * j + 2) * kRowBytes, a.E + wo, pol);
                const int64_t g = n * a.KG + (kl >> 7);
                cp_async4(slot + 6 * kRowBytes + 8 * j, a.meta + g);
                cp_async4(slot + 6 * kRowBytes + 8 * j + 4, a.meta + g + 1);
            }
        }
    };
    // This lane's 32 activations of the unit at p for every token (zeros past K or M).
    auto load_x = [&](const Pos &p, uint4 (&xv)[MT][4]) {
        const int64_t kl = p.ks * kStageK + 32 * lane;
#pragma unroll
        for (int m = 0; m < MT; ++m)
#pragma unroll
            for (int q = 0; q < 4; ++q)
                xv[m][q] = (kl < a.K && m < a.M) ? ldg_v4(a.x + int64_t(m) * a.K + kl + 8 * q)
                                                 : make_uint4(0u, 0u, 0u, 0u);
    };

    Pos pi = pc;  // copy-issue position
#pragma unroll
    for (int i = 0; i < S - 1; ++i) {
        if (u0 + i < u1) issue(pi, i);
        pi.next(steps);
        cp_async_commit();
    }
    uint4 xnext[MT][4];
    Pos px = pc;  // activation prefetch position
    if (u0 < u1) load_x(px, xnext);
    px.next(steps);

    uint32_t it = 0, slot_i = S - 1, slot_c = 0;
    for (int64_t u = u0; u < u1;) {
        const int64_t nb = pc.nb, first = nb * steps;
        const int64_t ua = u, ub = min(u1, first + steps);
        const int64_t col0 = nb * kCols;

        float acc[kCW][MT][2];
#pragma unroll
        for (int j = 0; j < kCW; ++j)
#pragma unroll
            for (int m = 0; m < MT; ++m) acc[j][m][0] = acc[j][m][1] = 0.f;

        for (; u < ub; ++u, ++it) {
            if (u + S - 1 < u1) issue(pi, int(slot_i));
            pi.next(steps);
            slot_i = (slot_i + 1 == uint32_t(S)) ? 0u : slot_i + 1;
            cp_async_commit();
            cp_async_wait<S - 1>();  // this lane's copies of unit u have landed
            uint4 xv[MT][4];
#pragma unroll
            for (int m = 0; m < MT; ++m)
#pragma unroll
                for (int q = 0; q < 4; ++q) xv[m][q] = xnext[m][q];
            if (u + 1 < u1) load_x(px, xnext);
            px.next(steps);

            const int64_t kl = pc.ks * kStageK + 32 * lane;
            pc.next(steps);
            if (kl < a.K) {
                const uint32_t slot = my + slot_c * uint32_t(kRows * kRowBytes);
#pragma unroll
                for (int j = 0; j < kCW; ++j) {
                    if (col0 + warp * kCW + j < a.N) {
                        const uint4 h = lds128(slot + (3 * j + 0) * kRowBytes);
                        const uint4 l = lds128(slot + (3 * j + 1) * kRowBytes);
                        const uint4 e = lds128(slot + (3 * j + 2) * kRowBytes);
                        const uint32_t m0 = lds32(slot + 6 * kRowBytes + 8 * j);
                        const uint32_t m1 = lds32(slot + 6 * kRowBytes + 8 * j + 4);
                        uint32_t w[16];
                        rebuild32(h, l, e, base4(m0), w);
                        if ((m0 >> 8) != (m1 >> 8))
                            patch_escapes(w, m0, m1, uint32_t(32 * (lane & 3)), a.esc, a.n_esc, a.err);
#pragma unroll
                        for (int i = 0; i < 16; ++i) {
#pragma unroll
                            for (int m = 0; m < MT; ++m)
                                fma_bf16x2(acc[j][m][0], acc[j][m][1], w[i], word_of(xv[m][i >> 2], i & 3));
                        }
                    }
                }
            }
            slot_c = (slot_c + 1 == uint32_t(S)) ? 0u : slot_c + 1;
        }

        constexpr int NV = kCW * MT;
        float v[NV];
#pragma unroll
        for (int j = 0; j < kCW; ++j)
#pragma unroll
            for (int m = 0; m < MT; ++m) v[j * MT + m] = acc[j][m][0] + acc[j][m][1];
        transpose_reduce<NV>(v, lane);
        constexpr int kShift = 5 - Log2<NV>::value;
        const bool whole = (ua == first) && (ub == first + a.steps);
        if ((lane & ((1 << kShift) - 1)) == 0) {
            const int vi = lane >> kShift;
            const int j = vi / MT, m = vi % MT;
            const int c = warp * kCW + j;
            if (col0 + c < a.N && m < a.M) {
                if (whole)
                    store_y(a, m, col0 + c, v[0]);
                else
                    a.partial[(ua * a.M + m) * kCols + c] = v[0];
            }
        }
        if (!whole) streamk_fixup(a, nb, ub - ua, &s_last, threadIdx.x, kThreads);
    }
    cp_async_wait<0>();
}

template <int MT>
int prepare_t() {
    return cudaFuncSetAttribute(gemv_kernel<MT>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                GemvCfg<MT>::kSmem) == cudaSuccess
               ? W12_OK
               : W12_ERR_CUDA;
}

// The dynamic shared-memory limit is raised once per device, by occ_t(),
// which the planner always runs before the first launch on a device.
template <int MT>
int launch_t(const GemmPlan &p, const GemmArgs &a, cudaStream_t s) {
    gemv_kernel<MT><<<unsigned(p.grid), kThreads, GemvCfg<MT>::kSmem, s>>>(a);
    return cudaGetLastError() == cudaSuccess ? W12_OK : W12_ERR_CUDA;
}

template <int MT>
int occ_t(int *blocks) {
    if (prepare_t<MT>() != W12_OK) return W12_ERR_CUDA;
    return cudaOccupancyMaxActiveBlocksPerMultiprocessor(blocks, gemv_kernel<MT>, kThreads,
                                                         GemvCfg<MT>::kSmem) == cudaSuccess
               ? W12_OK
               : W12_ERR_CUDA;
}

}  // namespace

// variant = log2(MT): tokens 1, 2, 4.
int launch_gemv(const GemmPlan &p, const GemmArgs &a, void *stream) {
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    switch (p.variant) {
        case 0: return launch_t<1>(p, a, s);
        case 1: return launch_t<2>(p, a, s);
        case 2: return launch_t<4>(p, a, s);
    }
    return W12_ERR_ARG;
}

int gemv_occupancy(int variant, int *blocks) {
    switch (variant) {
        case 0: return occ_t<1>(blocks);
        case 1: return occ_t<2>(blocks);
        case 2: return occ_t<4>(blocks);
    }
    return W12_ERR_ARG;
}

int gemv_cols_per_tile() { return kCols; }
int gemv_stage_k() { return kStageK; }

}  // namespace w12
