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
    static constexpr int kMinBlocks = MT == 1 ? 2 : 1;
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

// Unit cursor over the concatenated units of the batch: GEMM gi, column
// tile nb, k step ks.  Advanced by increments (no division in the loop);
// all index arithmetic in the loop is 32-bit.
struct Cur {
    int gi, nb, ks;
};

__device__ __forceinline__ void cur_next(const GemvBatch &b, Cur &c) {
    if (++c.ks == b.g[c.gi].steps) {
        c.ks = 0;
        if (++c.nb == b.g[c.gi].NB) {
            c.nb = 0;
            ++c.gi;
        }
    }
}

__device__ __forceinline__ Cur cur_at(const GemvBatch &b, int u) {
    Cur c{0, 0, 0};
    while (c.gi + 1 < b.count && u >= b.g[c.gi + 1].ubase) ++c.gi;
    const int local = u - b.g[c.gi].ubase;
    c.nb = local / b.g[c.gi].steps;
    c.ks = local % b.g[c.gi].steps;
    return c;
}

template <int MT>
__global__ void __launch_bounds__(kThreads, GemvCfg<MT>::kMinBlocks) gemv_kernel(const GemvBatch b) {
    constexpr int S = GemvCfg<MT>::kStages;
    extern __shared__ __align__(128) unsigned char smem[];
    __shared__ int s_last;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const uint32_t my = smem_addr(smem) + uint32_t(warp * S * kRows * kRowBytes + lane * 16);
    const uint64_t pol = l2_evict_first_policy();
    int u0, u1;
    {
        const int G = int(gridDim.x), c = int(blockIdx.x);
        const int per = b.U / G, rem = b.U % G;
        u0 = c * per + (c < rem ? c : rem);
        u1 = u0 + per + (c < rem ? 1 : 0);
    }
    if (u0 >= u1) return;
    const int M = b.M;

    // Start the copies of the unit at c into slot s.  Planes: this lane's
    // 16-byte chunks.  Meta: when K % 1024 == 0 a column's 9 words (groups
    // g0..g0+8, g0 a multiple of 8) lie in one aligned 48-byte window (inside
    // the meta section and its padding), copied as three 16-byte chunks by
    // three lanes into the warp-shared meta row; otherwise every lane copies
    // the two words of its own group for each column into its private chunk.
    auto issue = [&](const Cur &c, int s) {
        const GemvOne &g = b.g[c.gi];
        const int kst = c.ks * kStageK;
        const int kl = kst + 32 * lane;
        const uint32_t slot = my + uint32_t(s * kRows * kRowBytes);
        const bool fast_meta = (g.KG & 7) == 0;
        if (kl < g.K) {
#pragma unroll
            for (int j = 0; j < kCW; ++j) {
                const int n = c.nb * kCols + warp * kCW + j;
                if (n < g.N) {
                    const uint32_t wo = uint32_t(n) * uint32_t(g.KW) + uint32_t(kl >> 3);
                    cp_async16_stream(slot + (3 * j + 0) * kRowBytes, g.H + wo, pol);
                    cp_async16_stream(slot + (3 * j + 1) * kRowBytes, g.L + wo, pol);
                    cp_async16_stream(slot + (3 * j + 2) * kRowBytes, g.E + wo, pol);
                    if (!fast_meta) {
                        const uint32_t gg = uint32_t(n) * uint32_t(g.KG) + uint32_t(kl >> 7);
                        cp_async4(slot + 6 * kRowBytes + 8 * j, g.meta + gg);
                        cp_async4(slot + 6 * kRowBytes + 8 * j + 4, g.meta + gg + 1);
                    }
                }
            }
        }
        if (fast_meta && lane < 3 * kCW) {
            const int j = lane / 3, q = lane % 3;
            const int n = c.nb * kCols + warp * kCW + j;
            if (n < g.N)
                cp_async16(slot - uint32_t(lane * 16) + 6 * kRowBytes + j * 64 + q * 16,
                           g.meta + (uint32_t(n) * uint32_t(g.KG) + uint32_t(kst >> 7) + 4u * q));
        }
    };
    // This lane's 32 activations of the unit at c for every token (zeros past K or M).
    auto load_x = [&](const Cur &c, uint4 (&xv)[MT][4]) {
        const GemvOne &g = b.g[c.gi];
        const int kl = c.ks * kStageK + 32 * lane;
#pragma unroll
        for (int m = 0; m < MT; ++m)
#pragma unroll
            for (int q = 0; q < 4; ++q)
                xv[m][q] = (kl < g.K && m < M)
                               ? ldg_v4(g.x + (uint32_t(m) * uint32_t(g.K) + uint32_t(kl + 8 * q)))
                               : make_uint4(0u, 0u, 0u, 0u);
    };

    const Cur c0 = cur_at(b, u0);
    Cur ci = c0;  // copy-issue cursor
#pragma unroll
    for (int i = 0; i < S - 1; ++i) {
        if (u0 + i < u1) {
            issue(ci, i);
            cur_next(b, ci);
        }
        cp_async_commit();
    }
    Cur cc = c0;  // compute cursor
    uint32_t slot_i = S - 1, slot_c = 0;
    for (int u = u0; u < u1;) {
        const int gi = cc.gi;
        const GemvOne &g = b.g[gi];
        const int nb = cc.nb, first = g.ubase + nb * g.steps;
        const int ua = u, ub = min(u1, first + g.steps);
        const int col0 = nb * kCols;

        float acc[kCW][MT][2];
#pragma unroll
        for (int j = 0; j < kCW; ++j)
#pragma unroll
            for (int m = 0; m < MT; ++m) acc[j][m][0] = acc[j][m][1] = 0.f;

        for (; u < ub; ++u) {
            if (u + S - 1 < u1) {
                issue(ci, int(slot_i));
                cur_next(b, ci);
            }
            slot_i = (slot_i + 1 == uint32_t(S)) ? 0u : slot_i + 1;
            cp_async_commit();
            cp_async_wait<S - 1>();  // this lane's copies of unit u have landed ...
            __syncwarp();            // ... and so have the meta words other lanes copied
            uint4 xv[MT][4];
            load_x(cc, xv);          // L1-resident: every warp of the CTA reads the same slice
            const int kl = cc.ks * kStageK + 32 * lane;
            cur_next(b, cc);
            if (kl < g.K) {
                const uint32_t slot = my + slot_c * uint32_t(kRows * kRowBytes);
#pragma unroll
                for (int j = 0; j < kCW; ++j) {
                    if (col0 + warp * kCW + j < g.N) {
                        const uint4 h = lds128(slot + (3 * j + 0) * kRowBytes);
                        const uint4 l = lds128(slot + (3 * j + 1) * kRowBytes);
                        const uint4 e = lds128(slot + (3 * j + 2) * kRowBytes);
                        uint32_t m0, m1;
                        if ((g.KG & 7) == 0) {  // warp-shared 48-byte windows, g0 % 8 == 0
                            const uint32_t at = slot - uint32_t(lane * 16) + 6 * kRowBytes + j * 64 +
                                                uint32_t(lane >> 2) * 4u;
                            m0 = lds32(at);
                            m1 = lds32(at + 4);
                        } else {
                            m0 = lds32(slot + 6 * kRowBytes + 8 * j);
                            m1 = lds32(slot + 6 * kRowBytes + 8 * j + 4);
                        }
                        uint32_t w[16];
                        rebuild32(h, l, e, base4(m0), w);
                        if ((m0 >> 8) != (m1 >> 8))
                            patch_escapes(w, m0, m1, uint32_t(32 * (lane & 3)), g.esc, g.n_esc, b.err);
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
        const bool whole = (ua == first) && (ub == first + g.steps);
        if ((lane & ((1 << kShift) - 1)) == 0) {
            const int vi = lane >> kShift;
            const int j = vi / MT, m = vi % MT;
            const int c = warp * kCW + j;
            if (col0 + c < g.N && m < M) {
                if (whole)
                    store_out(g.y, b.y_dtype, g.N, m, col0 + c, v[0]);
                else
                    g.partial[(uint32_t(ua - g.ubase) * uint32_t(M) + uint32_t(m)) * kCols + c] = v[0];
            }
        }
        if (!whole)
            streamk_fixup_raw(g.counters, g.partial, first, g.ubase, g.steps, b.U, M, g.N, g.y, b.y_dtype, kCols,
                              nb, ub - ua, &s_last, threadIdx.x, kThreads);
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
int launch_t(const GemvBatch &b, int grid, cudaStream_t s) {
    gemv_kernel<MT><<<unsigned(grid), kThreads, GemvCfg<MT>::kSmem, s>>>(b);
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
int launch_gemv_batch(const GemvBatch &b, int variant, int grid, void *stream) {
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    switch (variant) {
        case 0: return launch_t<1>(b, grid, s);
        case 1: return launch_t<2>(b, grid, s);
        case 2: return launch_t<4>(b, grid, s);
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
