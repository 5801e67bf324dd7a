// kernels_mma.cu -- W12 decode-GEMM on tensor cores for 2 <= M <= 128.
//
// Swap-AB: the weight tile is operand A (16 output columns n x 16 k per
// mma.m16n8k16), the tokens are operand B (n = 8 tokens per mma), so a draft
// block of M tokens (SpecPilot repository page, "项目介绍": the W12 GEMM
// serves batch 1-32) fills the 8-wide side and the weight side stays 16 rows.
// Each lane streams 16-byte vectors of the three planes for two output
// columns (rows g and g+8 of the fragment) and rebuilds them straight into
// the A-fragment registers: lane t of a quad owns k = 32t .. 32t+31 of the
// group, and A/B agree on that k order, so no shuffle or shared-memory round
// trip is needed for the weights.  The tokens' slice of x is staged once per
// tile in shared memory (16-byte chunks XOR-swizzled so the B-fragment loads
// are conflict-free) and read with one 16-byte load per two mma k-steps.
//
// CTA = 8 warps x 16 columns = 128 columns; k range [kc*kchunk, +kchunk),
// x staged xchunk k at a time.  With FUSED the tile outputs are not stored
// as y: each CTA keeps a running (value, lowest index) maximum per token and
// the last CTA to finish runs the greedy acceptance on those maxima.
#include <cuda_runtime.h>

#include "gemm_common.cuh"
#include "verify_common.cuh"

namespace w12 {

namespace {

constexpr int kThreads = 256;
constexpr int kColsPerTile = 128;

__device__ __forceinline__ void mma_bf16(float (&c)[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                         uint32_t a3, uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
        "{%8,%9}, {%0,%1,%2,%3};"
        : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// Byte offset of 16-byte chunk c of token row r in the x tile (row pitch in
// bytes = 2 * kchunk).  Flips the two low chunk bits by bit 3 of c and the
// row parity, which makes each quarter-warp's 16-byte B loads hit 8 distinct
// bank groups.
__device__ __forceinline__ uint32_t x_chunk_offset(int r, int c, int pitch) {
    const int cs = c ^ (((c >> 3) & 1) << 1) ^ (r & 1);
    return uint32_t(r * pitch + cs * 16);
}

struct AFrag {
    uint4 h[2], l[2], e[2];
    uint32_t m0[2], m1[2];
};

__device__ __forceinline__ void load_a(const GemmArgs &a, int64_t nrow0, int64_t k, int t, AFrag &f) {
#pragma unroll
    for (int r = 0; r < 2; ++r) {
        const int64_t n = nrow0 + 8 * r;
        if (n < a.N) {
            const int64_t wo = n * a.KW + ((k + 32 * t) >> 3);
            f.h[r] = ldg_stream(a.H + wo);
            f.l[r] = ldg_stream(a.L + wo);
            f.e[r] = ldg_stream(a.E + wo);
            const int64_t g = n * a.KG + (k >> 7);
            f.m0[r] = ldg_u32(a.meta + g);
            f.m1[r] = ldg_u32(a.meta + g + 1);
        } else {
            f.h[r] = f.l[r] = f.e[r] = make_uint4(0u, 0u, 0u, 0u);
            f.m0[r] = f.m1[r] = 0u;
        }
    }
}

// Best (value, lowest index) key per token over this tile's columns, folded
// into the CTA's shared running maximum (the lm_head argmax epilogue).
template <int NT>
__device__ __forceinline__ void tile_argmax(const GemmArgs &a, const float (&acc)[NT][4],
                                            int64_t nrow0, int t, unsigned long long *s_best) {
#pragma unroll
    for (int j = 0; j < NT; ++j) {
#pragma unroll
        for (int q = 0; q < 2; ++q) {
            const int m = 8 * j + 2 * t + q;
            unsigned long long best = 0ull;
            if (nrow0 < a.N) best = pack_key(acc[j][q], uint32_t(nrow0));
            if (nrow0 + 8 < a.N) {
                const unsigned long long k2 = pack_key(acc[j][q + 2], uint32_t(nrow0 + 8));
                best = k2 > best ? k2 : best;
            }
            // lanes with the same t (same tokens) differ in lane bits 2..4
#pragma unroll
            for (int off = 4; off <= 16; off <<= 1) {
                const unsigned long long o = __shfl_xor_sync(0xFFFFFFFFu, best, off);
                best = o > best ? o : best;
            }
            if ((threadIdx.x & 28) == 0 && m < a.M && best != 0ull) atomicMax(&s_best[m], best);
        }
    }
}

template <int NT, bool FUSED>
__global__ void __launch_bounds__(kThreads, NT >= 8 ? 1 : 2) mma_kernel(const GemmArgs a) {
    extern __shared__ __align__(16) unsigned char xs[];
    __shared__ int s_last;
    __shared__ unsigned long long s_best[FUSED ? NT * 8 : 1];
    constexpr int MP = NT * 8;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int g = lane >> 2, t = lane & 3;
    const int pitch = int(a.xchunk) * 2;
    if (FUSED) {
        for (int m = threadIdx.x; m < MP; m += kThreads) s_best[m] = 0ull;
    }
    int64_t t0, t1;
    tile_range(a.T, t0, t1);
    for (int64_t tile = t0; tile < t1; ++tile) {
        const int64_t kc = tile / a.NB, nb = tile % a.NB;
        const int64_t kbeg = kc * a.kchunk;
        const int64_t kend = min(a.K, kbeg + a.kchunk);
        const int64_t nrow0 = nb * kColsPerTile + warp * 16 + g;

        float acc[NT][4];
#pragma unroll
        for (int j = 0; j < NT; ++j) acc[j][0] = acc[j][1] = acc[j][2] = acc[j][3] = 0.f;

        AFrag cur, nxt;
        load_a(a, nrow0, kbeg, t, cur);
        for (int64_t xb = kbeg; xb < kend; xb += a.xchunk) {
            const int64_t xe = min(kend, xb + a.xchunk);
            const int nchunks = int(xe - xb) / 8;
            // stage x[0..MP) x [xb, xe) (token rows >= M are zero)
            __syncthreads();
            for (int i = threadIdx.x; i < MP * nchunks; i += kThreads) {
                const int r = i / nchunks, c = i % nchunks;
                uint4 v = make_uint4(0u, 0u, 0u, 0u);
                if (r < a.M) v = ldg_v4(a.x + int64_t(r) * a.K + xb + 8 * c);
                *reinterpret_cast<uint4 *>(xs + x_chunk_offset(r, c, pitch)) = v;
            }
            __syncthreads();
            for (int64_t k = xb; k < xe; k += 128) {
                if (k + 128 < kend) load_a(a, nrow0, k + 128, t, nxt);
                uint32_t wa[16], wb[16];
                rebuild32(cur.h[0], cur.l[0], cur.e[0], base4(cur.m0[0]), wa);
                rebuild32(cur.h[1], cur.l[1], cur.e[1], base4(cur.m0[1]), wb);
                if ((cur.m0[0] >> 8) != (cur.m1[0] >> 8))
                    patch_escapes(wa, cur.m0[0], cur.m1[0], uint32_t(32 * t), a.esc, a.n_esc, a.err);
                if ((cur.m0[1] >> 8) != (cur.m1[1] >> 8))
                    patch_escapes(wb, cur.m0[1], cur.m1[1], uint32_t(32 * t), a.esc, a.n_esc, a.err);
                const int cbase = int(k - xb) / 8 + 4 * t;
#pragma unroll
                for (int sp = 0; sp < 4; ++sp) {
#pragma unroll
                    for (int j = 0; j < NT; ++j) {
                        const uint4 b = *reinterpret_cast<const uint4 *>(
                            xs + x_chunk_offset(8 * j + g, cbase + sp, pitch));
                        mma_bf16(acc[j], wa[4 * sp], wb[4 * sp], wa[4 * sp + 1], wb[4 * sp + 1],
                                 b.x, b.y);
                        mma_bf16(acc[j], wa[4 * sp + 2], wb[4 * sp + 2], wa[4 * sp + 3],
                                 wb[4 * sp + 3], b.z, b.w);
                    }
                }
                cur = nxt;
            }
        }

        // C fragment: acc[j][0..1] = (row g, tokens 8j+2t, +1), [2..3] = row g+8.
        if (FUSED) {
            if (a.logits_out) {
#pragma unroll
                for (int j = 0; j < NT; ++j)
#pragma unroll
                    for (int q = 0; q < 4; ++q) {
                        const int64_t n = nrow0 + 8 * (q >> 1);
                        const int m = 8 * j + 2 * t + (q & 1);
                        if (n < a.N && m < a.M) a.logits_out[int64_t(m) * a.N + n] = acc[j][q];
                    }
            }
            tile_argmax<NT>(a, acc, nrow0, t, s_best);
        } else {
#pragma unroll
            for (int j = 0; j < NT; ++j) {
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    const int64_t n = nrow0 + 8 * (q >> 1);
                    const int m = 8 * j + 2 * t + (q & 1);
                    if (n < a.N && m < a.M) emit(a, kc, m, n, acc[j][q]);
                }
            }
            finish_tile(a, nb, &s_last, threadIdx.x, kThreads);
        }
    }
    if (FUSED) {
        // publish this CTA's per-token best; the last CTA to finish verifies
        __syncthreads();
        for (int m = threadIdx.x; m < a.M; m += kThreads)
            a.row_best[int64_t(blockIdx.x) * a.M + m] = s_best[m];
        __threadfence();
        __syncthreads();
        if (threadIdx.x == 0) s_last = (atomicAdd(a.counters, 1u) == gridDim.x - 1);
        __syncthreads();
        if (s_last) {
            __threadfence();
            verify_from_keys(a.row_best, int64_t(gridDim.x), a.M, a.vR, a.vT, a.draft,
                             a.accept_len, a.next_tok, a.gbuf);
            if (threadIdx.x == 0) a.counters[0] = 0u;
        }
    }
}

constexpr int kMaxXSmem = 64 * 1024;  // the planner keeps MP * xchunk * 2 within this

// The dynamic shared-memory limit is raised once per device, by occ_t(),
// which the planner always runs before the first launch on a device.
template <int NT, bool FUSED>
int launch_t(const GemmPlan &p, const GemmArgs &a, cudaStream_t s) {
    const size_t smem = size_t(NT) * 8 * size_t(a.xchunk) * 2;
    if (smem > size_t(kMaxXSmem)) return W12_ERR_ARG;
    mma_kernel<NT, FUSED><<<unsigned(p.grid), kThreads, smem, s>>>(a);
    return cudaGetLastError() == cudaSuccess ? W12_OK : W12_ERR_CUDA;
}

template <int NT>
int occ_t(int *blocks, size_t smem) {
    if (cudaFuncSetAttribute(mma_kernel<NT, false>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             kMaxXSmem) != cudaSuccess ||
        cudaFuncSetAttribute(mma_kernel<NT, true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             kMaxXSmem) != cudaSuccess)
        return W12_ERR_CUDA;
    return cudaOccupancyMaxActiveBlocksPerMultiprocessor(blocks, mma_kernel<NT, false>, kThreads,
                                                         smem) == cudaSuccess
               ? W12_OK
               : W12_ERR_CUDA;
}


}  // namespace

// variant v: NT = 1 << v, i.e. tokens padded to 8, 16, 32, 64 or 128.
int launch_mma(const GemmPlan &p, const GemmArgs &a, void *stream) {
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    const bool fused = a.row_best != nullptr;
    switch (p.variant) {
        case 0: return fused ? launch_t<1, true>(p, a, s) : launch_t<1, false>(p, a, s);
        case 1: return fused ? launch_t<2, true>(p, a, s) : launch_t<2, false>(p, a, s);
        case 2: return fused ? launch_t<4, true>(p, a, s) : launch_t<4, false>(p, a, s);
        case 3: return fused ? launch_t<8, true>(p, a, s) : launch_t<8, false>(p, a, s);
        case 4: return fused ? launch_t<16, true>(p, a, s) : launch_t<16, false>(p, a, s);
    }
    return W12_ERR_ARG;
}

int mma_occupancy(int variant, size_t smem, int *blocks) {
    switch (variant) {
        case 0: return occ_t<1>(blocks, smem);
        case 1: return occ_t<2>(blocks, smem);
        case 2: return occ_t<4>(blocks, smem);
        case 3: return occ_t<8>(blocks, smem);
        case 4: return occ_t<16>(blocks, smem);
    }
    return W12_ERR_ARG;
}

}  // namespace w12
