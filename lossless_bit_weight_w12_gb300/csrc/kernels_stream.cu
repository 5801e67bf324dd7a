// kernels_stream.cu -- W12 decode-GEMM for skinny M (1 <= M <= 128) on
// mma.sync tensor tiles, fed by the Tensor Memory Accelerator.
//
// A decode or verification step reads every weight once (SpecPilot summary,
// airadar.tv English edition, first paragraph), so this kernel is a weight
// stream first: one warp of each CTA only issues copies, eight warps only
// rebuild and multiply, and the two meet in a ring of shared-memory stages.
//
//  - Work: units of one 128-k group of a 128-column tile, over every product
//    of the batch (stream-K): CTA c takes a balanced contiguous range of
//    units, so the busiest CTA does at most one group more than the
//    average.  A tile cut by a CTA boundary is finished by a deterministic
//    fix-up (partial sums added in CTA order by the CTA that completes it).
//  - Producer warp: per unit, one bulk copy of the unit block (format v2:
//    the H, L, E planes of 128 columns x 128 k and their meta words, one
//    contiguous 25 KB block of the blob) and one 3-D tensor copy of x
//    (every token's 128 activations of the group, 128-byte swizzle, rows
//    past M zero-filled), both completing on the stage's "full" barrier.
//    At the start of every tile piece it prefetches the piece's escape
//    entries (one contiguous range of the escape list) into L1, so the rare
//    patch-up does not wait on HBM.
//  - Compute warps (swap-AB, mma.m16n8k16: weights are operand A, tokens
//    operand B): warp w owns columns 16w .. 16w + 15 of the tile; lane
//    (g, t) rebuilds columns 16w + g and 16w + g + 8 for k = 32t .. 32t + 31
//    of the group straight into A-fragment registers ("reconstructing bit by
//    bit in GEMM registers", same page, "Reasons" bullet 2), patches escapes
//    and reads the matching B fragments from the swizzled x box.  A and B
//    agree on that k order, so no shuffle is needed.  After its last read of
//    a stage each warp arrives on the stage's "empty" barrier.
//  - Shared-memory reads are conflict-free: plane rows are 64 bytes (the
//    two columns of a quarter-warp fill one 128-byte line, their chunks
//    permuted alike by the format's swizzle); in the x box a token's row
//    pair (2 r, 2 r + 1) under the 128-byte swizzle sends the 8 lanes of a
//    quarter-warp to 8 different 16-byte bank groups.
// Every mbarrier wait is bounded (async_common.cuh): after a timeout the
// error word says W12_ERR_TIMEOUT and all roles run to the end without
// waiting, so the CTA still reaches its named barriers and exits.
#include <cuda.h>
#include <cuda_runtime.h>

#include <mutex>
#include <unordered_map>

#include "async_common.cuh"
#include "gemm_common.cuh"
#include "stream_common.h"
#include "stream_device.cuh"
#include "verify_common.cuh"

namespace w12 {

namespace {

constexpr int kCW = 8;                    // compute warps
constexpr int kCT = kCW * 32;             // compute threads
constexpr int kST = kCT + 32;             // + one producer warp
constexpr int kMaxM = W12_MAX_M;

// Stage layout (bytes from the stage start, stages 1024-byte aligned):
// x box (MP tokens x 2 halves x 128 bytes), then the unit block (H, L, E
// planes, meta words).
template <int NT>
struct SCfg {
    static constexpr int MP = 8 * NT;
    static constexpr int kX = MP * 256;
    static constexpr int kH = kX, kL = kX + kPlaneBlock, kE = kX + 2 * kPlaneBlock;
    static constexpr int kMeta = kX + kMetaAt;
    static constexpr int kStage = (kX + kUnitBytes + 1023) / 1024 * 1024;
};

// Ring depth for NT and CTAs per SM: as many stages as fit in the 227 KB a
// CTA may use (or half of it for two CTAs per SM), at most 8.
// With two CTAs per SM the barriers and scalars (full[S], empty[S], the wait
// state, s_last, s_best) live in the dynamic region after the ring, and the
// kernel has no static shared memory: its dynamic region then starts at the
// CTA's 1024-byte aligned shared base (checked), with no alignment slack
// (measured faster: the M = 1 GEMV layer 79.9 -> 79.0 us, mma.sync at
// M = 16 84.8 -> 83.9).  With one CTA per SM they stay static shared
// memory in front of a 1024-aligned ring (the other layout was slower
// there: mma.sync at M = 128 230 -> 244 us).
constexpr int kSmemPerSm = 227 * 1024;
template <int NT, int MINB>
struct SRing {
    static constexpr bool kBarAfter = MINB == 2;
    static constexpr int kAvail = kSmemPerSm / MINB - 1024 - 2048;  // alignment slack or barriers
    static constexpr int kFit = kAvail / SCfg<NT>::kStage;
    static constexpr int S = kFit > 8 ? 8 : kFit;
    static constexpr size_t kBarOff = size_t(S) * SCfg<NT>::kStage;
    static constexpr size_t kBarBytes = size_t(2 * S) * 8 + 16 + 8 + size_t(kMaxM) * 8;
    static constexpr size_t kDynSmem = kBarAfter ? kBarOff + kBarBytes : kBarOff + 1024;
};

__device__ __forceinline__ void mma_bf16(float (&c)[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                         uint32_t a3, uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
        "{%8,%9}, {%0,%1,%2,%3};"
        : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// Best (value, lowest index) key per token over the columns a warp holds in
// its C fragments, folded into the CTA's running maximum s_best (shared).
template <int NT>
__device__ __forceinline__ void frag_argmax(const float (&acc)[NT][4], int na, int nbb, int N, int M, int t,
                                            int lane, unsigned long long *s_best) {
#pragma unroll
    for (int j = 0; j < NT; ++j) {
#pragma unroll
        for (int q = 0; q < 2; ++q) {
            const int m = 8 * j + 2 * t + q;
            unsigned long long best = 0ull;
            if (na < N) best = pack_key(acc[j][q], uint32_t(na));
            if (nbb < N) {
                const unsigned long long k2 = pack_key(acc[j][q + 2], uint32_t(nbb));
                best = k2 > best ? k2 : best;
            }
            // lanes with the same t hold the same tokens; they differ in lane bits 2..4
#pragma unroll
            for (int off = 4; off <= 16; off <<= 1) {
                const unsigned long long o = __shfl_xor_sync(0xFFFFFFFFu, best, off);
                best = o > best ? o : best;
            }
            if ((lane & 28) == 0 && m < M && best != 0ull) atomicMax(&s_best[m], best);
        }
    }
}

// MT = 0: mma.sync consumers (tokens padded to 8 NT).  MT = 1, 2, 4: the
// CUDA-core GEMV consumers for M <= MT (NT = 1): lane (g, t) multiplies its
// rebuilt weights of rows g and g + 8, k = 32t .. 32t + 31, with each
// token's activations (fma.rn.f32.bf16 on the bf16 halves: no unpacking),
// and the four lanes of a row are summed with two warp shuffles at the end
// of a tile piece.
template <int NT, int MINB, bool FUSED, int MT = 0>
__global__ void __launch_bounds__(kST, MINB) stream_kernel(const __grid_constant__ StreamBatch b) {
    static_assert(MT == 0 || (NT == 1 && !FUSED), "the GEMV consumers serve plain products, M <= 4");
    using C = SCfg<NT>;
    constexpr int S = SRing<NT, MINB>::S;
    using Ring = SRing<NT, MINB>;
    extern __shared__ unsigned char smem_dyn[];
    uint64_t *full, *empty;
    WaitCtl *ctl;
    int *lastp;
    unsigned long long *s_best;
    uint32_t base;
    if constexpr (Ring::kBarAfter) {
        if (smem_addr(smem_dyn) & 1023u) {  // the stages need a 1024-byte aligned start
            if (threadIdx.x == 0) record_error(b.err, W12_ERR_DEVICE);
            return;
        }
        full = reinterpret_cast<uint64_t *>(smem_dyn + Ring::kBarOff);
        empty = full + S;
        ctl = reinterpret_cast<WaitCtl *>(empty + S);
        lastp = reinterpret_cast<int *>(empty + S + 2);
        s_best = reinterpret_cast<unsigned long long *>(empty + S + 3);
        base = smem_addr(smem_dyn);
    } else {
        __shared__ __align__(8) uint64_t full_s[S], empty_s[S];
        __shared__ WaitCtl ctl_s;
        __shared__ int last_s;
        __shared__ unsigned long long best_s[FUSED ? kMaxM : 1];
        full = full_s;
        empty = empty_s;
        ctl = &ctl_s;
        lastp = &last_s;
        s_best = best_s;
        base = (smem_addr(smem_dyn) + 1023u) & ~1023u;
    }
    WaitCtl &s_ctl = *ctl;
    int &s_last = *lastp;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    int u0, u1;
    {
        const int G = int(gridDim.x), c = int(blockIdx.x);
        const int per = b.U / G, rem = b.U % G;
        u0 = sk_unit_begin(c, per, rem);
        u1 = u0 + per + (c < rem ? 1 : 0);
    }
    if (threadIdx.x == 0) {
        for (int s = 0; s < S; ++s) {
            mbar_init(&full[s], 1);  // the producer's expect_tx arrival (+ bytes)
            mbar_init(&empty[s], kCW);
        }
        wait_ctl_init(&s_ctl, b);
        mbar_fence_init();
    }
    if (FUSED)
        for (int m = threadIdx.x; m < kMaxM; m += kST) s_best[m] = 0ull;
    __syncthreads();
    if (threadIdx.x == 0) pdl_launch();
    if (!FUSED && u0 >= u1) return;

    if (warp == kCW) {
        if (u0 >= u1) return;
        stream_producer<S, false>(b, base, C::kStage, C::kX, C::MP, full, empty, &s_ctl, u0, u1, lane);
        return;
    }
    pdl_wait();  // nothing below touches global memory the previous kernel may write before this

    // ---------------------------------------------------------------- compute
    const int g8 = lane >> 2, t = lane & 3;
    const int ra = 16 * warp + g8;  // tile column of fragment row g8
    // this lane's 16 bytes (logical chunk t) of plane row ra, and of row
    // ra + 8 (same swizzle, 512 bytes on)
    const uint32_t pa = uint32_t(ra * 64 + 16 * (t ^ ((ra >> 1) & 3)));
    const uint32_t pb = pa + 8u * 64u;
    const uint32_t ma = uint32_t(4 * ra), mb = ma + 32u;  // meta words ra, ra + 8
    // x box: token r, half h at row 2r + h (128 bytes), 16-byte chunk c
    // stored at c ^ (row & 7).  Lane t reads half t >> 1, chunks
    // 4 (t & 1) + sp, sp = 0..3; token 8j + g8 adds j * 2048 bytes.
    const int xr = 2 * g8 + (t >> 1);
    const uint32_t xb0 = uint32_t(xr * 128) + (uint32_t((4 * (t & 1)) ^ (xr & 7)) << 4);
    const int M = b.M;
    SCur c = s_at(b, u0);
    int s = 0;
    uint32_t ph = 0;
    for (int u = u0; u < u1;) {
        const StreamOne &g = b.g[c.gi];
        const int nb = c.nb, first = g.ubase + nb * g.KG;
        const int ua = u, ub = min(u1, first + g.KG);
        const int na = nb * kTileN + ra, nbb = na + 8;
        const bool va = na < g.N, vb = nbb < g.N;

        float acc[NT][4];
#pragma unroll
        for (int j = 0; j < NT; ++j) acc[j][0] = acc[j][1] = acc[j][2] = acc[j][3] = 0.f;
        float fa[MT > 0 ? MT : 1][2][2], fb[MT > 0 ? MT : 1][2][2];  // [token][lo/hi][chain]
#pragma unroll
        for (int m = 0; m < (MT > 0 ? MT : 1); ++m)
#pragma unroll
            for (int q = 0; q < 2; ++q) fa[m][q][0] = fa[m][q][1] = fb[m][q][0] = fb[m][q][1] = 0.f;

        for (; u < ub; ++u) {
            mbar_wait(&full[s], ph, &s_ctl, b.err);
            const uint32_t st = base + uint32_t(s) * C::kStage;
            const uint4 ha = lds128(st + C::kH + pa), la = lds128(st + C::kL + pa), ea = lds128(st + C::kE + pa);
            const uint4 hb = lds128(st + C::kH + pb), lb = lds128(st + C::kL + pb), eb = lds128(st + C::kE + pb);
            const uint2 mA = make_uint2(lds32(st + C::kMeta + ma), lds32(st + C::kMeta + ma + 4u));
            const uint2 mB = make_uint2(lds32(st + C::kMeta + mb), lds32(st + C::kMeta + mb + 4u));
            uint32_t wa[16], wb[16];
            rebuild32(ha, la, ea, base4(mA.x), wa);
            rebuild32(hb, lb, eb, base4(mB.x), wb);
            if (va && (mA.x >> 8) != (mA.y >> 8))
                patch_escapes(wa, mA.x, mA.y, uint32_t(32 * t), g.esc, g.n_esc, b.err);
            if (vb && (mB.x >> 8) != (mB.y >> 8))
                patch_escapes(wb, mB.x, mB.y, uint32_t(32 * t), g.esc, g.n_esc, b.err);
            if (MT == 0) {
#pragma unroll
                for (int sp = 0; sp < 4; ++sp) {
#pragma unroll
                    for (int j = 0; j < NT; ++j) {
                        const uint4 bx = lds128(st + uint32_t(j * 2048) + (xb0 ^ uint32_t(sp << 4)));
                        mma_bf16(acc[j], wa[4 * sp], wb[4 * sp], wa[4 * sp + 1], wb[4 * sp + 1], bx.x, bx.y);
                        mma_bf16(acc[j], wa[4 * sp + 2], wb[4 * sp + 2], wa[4 * sp + 3], wb[4 * sp + 3], bx.z,
                                 bx.w);
                    }
                }
            } else {
#pragma unroll
                for (int m = 0; m < (MT > 0 ? MT : 1); ++m) {
                    if (m >= M) break;
                    // token m, half t >> 1 at x-box row 2m + (t >> 1)
                    const int xrm = 2 * m + (t >> 1);
                    const uint32_t xm = uint32_t(xrm * 128);
#pragma unroll
                    for (int sp = 0; sp < 4; ++sp) {
                        const uint4 bx =
                            lds128(st + xm + (uint32_t((4 * (t & 1) + sp) ^ (xrm & 7)) << 4));
                        const uint32_t xv[4] = {bx.x, bx.y, bx.z, bx.w};
#pragma unroll
                        for (int q = 0; q < 4; ++q) {
                            fma_bf16x2(fa[m][0][q & 1], fa[m][1][q & 1], wa[4 * sp + q], xv[q]);
                            fma_bf16x2(fb[m][0][q & 1], fb[m][1][q & 1], wb[4 * sp + q], xv[q]);
                        }
                    }
                }
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(&empty[s]);
            if (++s == S) {
                s = 0;
                ph ^= 1u;
            }
        }

        if (MT > 0) {
            // GEMV: fold the lane's chains, then the four lanes t of each row
            // (lanes g8 * 4 + t); lane t == 0 ends with the row sums, which
            // are placed where the mma epilogue expects token 0 (acc[0][0] for
            // row g8, acc[0][2] for row g8 + 8) and tokens 1.. in a side array.
#pragma unroll
            for (int m = 0; m < (MT > 0 ? MT : 1); ++m) {
                float va2 = (fa[m][0][0] + fa[m][1][0]) + (fa[m][0][1] + fa[m][1][1]);
                float vb2 = (fb[m][0][0] + fb[m][1][0]) + (fb[m][0][1] + fb[m][1][1]);
                va2 += __shfl_xor_sync(0xFFFFFFFFu, va2, 1);
                vb2 += __shfl_xor_sync(0xFFFFFFFFu, vb2, 1);
                va2 += __shfl_xor_sync(0xFFFFFFFFu, va2, 2);
                vb2 += __shfl_xor_sync(0xFFFFFFFFu, vb2, 2);
                fa[m][0][0] = va2;
                fb[m][0][0] = vb2;
            }
            if (ua == first && ub == first + g.KG) {
                if (t == 0) {
#pragma unroll
                    for (int m = 0; m < (MT > 0 ? MT : 1); ++m) {
                        if (m >= M) break;
                        if (na < g.N) store_out(g.y, b.y_dtype, g.N, m, na, fa[m][0][0]);
                        if (nbb < g.N) store_out(g.y, b.y_dtype, g.N, m, nbb, fb[m][0][0]);
                    }
                }
            } else {
                const int slot = ua == u0 ? 0 : 1;
                float *P = b.partial + (size_t(blockIdx.x) * 2 + slot) * size_t(M) * kTileN;
                if (t == 0) {
#pragma unroll
                    for (int m = 0; m < (MT > 0 ? MT : 1); ++m) {
                        if (m >= M) break;
                        P[m * kTileN + ra] = fa[m][0][0];
                        P[m * kTileN + ra + 8] = fb[m][0][0];
                    }
                }
                stream_fixup<false>(b, g, first, nb, ub - ua, &s_last, threadIdx.x, kCT, s_best);
            }
            s_next_tile(b, c);
            continue;
        }

        // C fragment: acc[j][0..1] = (row g8, tokens 8j + 2t, +1), [2..3] = row g8 + 8.
        if (ua == first && ub == first + g.KG) {
            if (!FUSED || g.y) {
#pragma unroll
                for (int j = 0; j < NT; ++j)
#pragma unroll
                    for (int q = 0; q < 4; ++q) {
                        const int n = q < 2 ? na : nbb;
                        const int m = 8 * j + 2 * t + (q & 1);
                        if (n < g.N && m < M) store_out(g.y, b.y_dtype, g.N, m, n, acc[j][q]);
                    }
            }
            if (FUSED) frag_argmax<NT>(acc, na, nbb, g.N, M, t, lane, s_best);
        } else {
            const int slot = ua == u0 ? 0 : 1;
            float *P = b.partial + (size_t(blockIdx.x) * 2 + slot) * size_t(M) * kTileN;
#pragma unroll
            for (int j = 0; j < NT; ++j)
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    const int m = 8 * j + 2 * t + (q & 1);
                    if (m < M) P[m * kTileN + (q < 2 ? ra : ra + 8)] = acc[j][q];
                }
            stream_fixup<FUSED>(b, g, first, nb, ub - ua, &s_last, threadIdx.x, kCT, s_best);
        }
        s_next_tile(b, c);
    }

    if (FUSED) {
        // publish this CTA's per-token best; the last CTA to arrive folds
        // them and runs the acceptance rule
        const int tid = threadIdx.x;
        named_sync(kCT);
        for (int m = tid; m < M; m += kCT) b.row_best[size_t(blockIdx.x) * M + m] = s_best[m];
        __threadfence();
        named_sync(kCT);
        if (tid == 0) s_last = (atomicAdd(b.done, 1u) == gridDim.x - 1);
        named_sync(kCT);
        if (s_last) {
            __threadfence();
            verify_from_keys(b.row_best, int64_t(gridDim.x), M, b.vR, b.vT, b.draft, b.accept_len, b.next_tok,
                             b.gbuf, tid, kCT);
            if (tid == 0) *b.done = 0u;
        }
    }
}

// ------------------------------------------------------------------ host side

using EncodeTiledFn = CUresult (*)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *, const cuuint64_t *,
                                   const cuuint64_t *, const cuuint32_t *, const cuuint32_t *,
                                   CUtensorMapInterleave, CUtensorMapSwizzle, CUtensorMapL2promotion,
                                   CUtensorMapFloatOOBfill);

// The driver's tensor-map encoder, looked up once through the runtime (the
// library does not link libcuda directly).
EncodeTiledFn encoder() {
    static const EncodeTiledFn fn = [] {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q = cudaDriverEntryPointSymbolNotFound;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) !=
                cudaSuccess ||
            q != cudaDriverEntryPointSuccess)
            return static_cast<EncodeTiledFn>(nullptr);
        return reinterpret_cast<EncodeTiledFn>(p);
    }();
    return fn;
}

// x [M][K] bf16 as [M][K/64][64]; box 64 x 2 x MP (one group, every token),
// 128-byte swizzle, tokens past M read as zeros (the mma.sync kernel).
int x_map(CUtensorMap *m, const uint16_t *x, int64_t K, int M, int MP) {
    const cuuint64_t dims[3] = {64, cuuint64_t(K / 64), cuuint64_t(M)};
    const cuuint64_t strides[2] = {128, cuuint64_t(K * 2)};
    const cuuint32_t box[3] = {64, 2, cuuint32_t(MP)};
    const cuuint32_t es[3] = {1, 1, 1};
    return encoder()(m, CU_TENSOR_MAP_DATA_TYPE_UINT16, 3, const_cast<uint16_t *>(x), dims, strides, box, es,
                     CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_128B,
                     CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS
               ? W12_OK
               : W12_ERR_CUDA;
}

// x [M][K] bf16 as a 2-D array; box 64 k x MP tokens, 128-byte swizzle,
// tokens past M read as zeros (the tcgen05 kernel's B operand).
int x_map_tc(CUtensorMap *m, const uint16_t *x, int64_t K, int M, int MP) {
    const cuuint64_t dims[2] = {cuuint64_t(K), cuuint64_t(M)};
    const cuuint64_t strides[1] = {cuuint64_t(K * 2)};
    const cuuint32_t box[2] = {64, cuuint32_t(MP)};
    const cuuint32_t es[2] = {1, 1};
    return encoder()(m, CU_TENSOR_MAP_DATA_TYPE_UINT16, 2, const_cast<uint16_t *>(x), dims, strides, box, es,
                     CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_128B,
                     CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS
               ? W12_OK
               : W12_ERR_CUDA;
}

template <int NT, int MINB, bool FUSED = false, int MT = 0>
int launch_t(const StreamBatch &b, int grid, cudaStream_t s) {
    return launch_pdl(stream_kernel<NT, MINB, FUSED, MT>, grid, kST, SRing<NT, MINB>::kDynSmem, s, b);
}

template <int NT, int MINB, bool FUSED = false, int MT = 0>
int occ_t(int *blocks) {
    const size_t smem = SRing<NT, MINB>::kDynSmem;
    if (cudaFuncSetAttribute(stream_kernel<NT, MINB, FUSED, MT>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             int(smem)) != cudaSuccess)
        return W12_ERR_CUDA;
    return cudaOccupancyMaxActiveBlocksPerMultiprocessor(blocks, stream_kernel<NT, MINB, FUSED, MT>, kST, smem) ==
                   cudaSuccess
               ? W12_OK
               : W12_ERR_CUDA;
}

}  // namespace

// v = 2 * log2(NT) + (ctas_per_sm - 1); two CTAs per SM only where the
// ring still holds three stages (NT <= 4).
int stream_occupancy(int v, int *blocks) {
    switch (v) {
        case 0: return occ_t<1, 1>(blocks);
        case 1: return occ_t<1, 2>(blocks);
        case 2: return occ_t<2, 1>(blocks);
        case 3: return occ_t<2, 2>(blocks);
        case 4: return occ_t<4, 1>(blocks);
        case 5: return occ_t<4, 2>(blocks);
        case 6: return occ_t<8, 1>(blocks);
        case 8: return occ_t<16, 1>(blocks);
    }
    return W12_ERR_ARG;
}

namespace {

// Tensor maps depend only on the address and the shape they describe, so
// they are encoded once and reused (a batched call of six products would
// otherwise spend tens of microseconds of host time in the encoder).
struct MapKey {
    uintptr_t ptr;
    int64_t a, b, c;
    bool operator==(const MapKey &o) const { return ptr == o.ptr && a == o.a && b == o.b && c == o.c; }
};
struct MapKeyHash {
    size_t operator()(const MapKey &k) const {
        uint64_t h = k.ptr * 0x9E3779B97F4A7C15ull;
        h ^= uint64_t(k.a) + 0x632BE59BD9B4E019ull + (h << 6) + (h >> 2);
        h ^= uint64_t(k.b) + 0x8CB92BA72F3D8DD7ull + (h << 6) + (h >> 2);
        h ^= uint64_t(k.c) + 0x7F4A7C159E3779B9ull + (h << 6) + (h >> 2);
        return size_t(h);
    }
};
std::mutex g_map_mu;
std::unordered_map<MapKey, CUtensorMap, MapKeyHash> g_maps;
constexpr size_t kMaxCachedMaps = 4096;

template <class Make>
int cached_map(CUtensorMap *out, const MapKey &key, Make make) {
    {
        std::lock_guard<std::mutex> lock(g_map_mu);
        auto it = g_maps.find(key);
        if (it != g_maps.end()) {
            *out = it->second;
            return W12_OK;
        }
    }
    const int st = make(out);
    if (st != W12_OK) return st;
    std::lock_guard<std::mutex> lock(g_map_mu);
    if (g_maps.size() >= kMaxCachedMaps) g_maps.clear();
    g_maps.emplace(key, *out);
    return W12_OK;
}

}  // namespace

int stream_make_maps(StreamOne &g, const w12_desc &d, const uint16_t *x, int M, int MP, bool tc) {
    if (!encoder()) return W12_ERR_CUDA;
    const int64_t K = d.K;
    if (tc)
        return cached_map(&g.tx, MapKey{reinterpret_cast<uintptr_t>(x), K, M, -MP},
                          [&](CUtensorMap *m) { return x_map_tc(m, x, K, M, MP); });
    return cached_map(&g.tx, MapKey{reinterpret_cast<uintptr_t>(x), K, M, MP},
                      [&](CUtensorMap *m) { return x_map(m, x, K, M, MP); });
}

// The CUDA-core GEMV consumers: variant v = log2(MT) (M = 1, 2, 4), two
// CTAs per SM.
int stream_gemv_occupancy(int v, int *blocks) {
    switch (v) {
        case 0: return occ_t<1, 2, false, 1>(blocks);
        case 1: return occ_t<1, 2, false, 2>(blocks);
        case 2: return occ_t<1, 2, false, 4>(blocks);
    }
    return W12_ERR_ARG;
}

int launch_stream_gemv(const StreamBatch &b, int v, int grid, void *stream) {
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    switch (v) {
        case 0: return launch_t<1, 2, false, 1>(b, grid, s);
        case 1: return launch_t<1, 2, false, 2>(b, grid, s);
        case 2: return launch_t<1, 2, false, 4>(b, grid, s);
    }
    return W12_ERR_ARG;
}

int stream_fused_occupancy(int v, int *blocks) {
    switch (v) {
        case 0: return occ_t<1, 1, true>(blocks);
        case 1: return occ_t<1, 2, true>(blocks);
        case 2: return occ_t<2, 1, true>(blocks);
        case 3: return occ_t<2, 2, true>(blocks);
        case 4: return occ_t<4, 1, true>(blocks);
        case 5: return occ_t<4, 2, true>(blocks);
        case 6: return occ_t<8, 1, true>(blocks);
        case 8: return occ_t<16, 1, true>(blocks);
    }
    return W12_ERR_ARG;
}

int launch_stream_fused(const StreamBatch &b, int v, int grid, void *stream) {
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    switch (v) {
        case 0: return launch_t<1, 1, true>(b, grid, s);
        case 1: return launch_t<1, 2, true>(b, grid, s);
        case 2: return launch_t<2, 1, true>(b, grid, s);
        case 3: return launch_t<2, 2, true>(b, grid, s);
        case 4: return launch_t<4, 1, true>(b, grid, s);
        case 5: return launch_t<4, 2, true>(b, grid, s);
        case 6: return launch_t<8, 1, true>(b, grid, s);
        case 8: return launch_t<16, 1, true>(b, grid, s);
    }
    return W12_ERR_ARG;
}

// The dynamic shared-memory limit is raised by stream_occupancy() (or
// stream_fused_occupancy()), which the planner runs once per device and
// variant before the first launch.
int launch_stream_batch(const StreamBatch &b, int v, int grid, void *stream) {
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    switch (v) {
        case 0: return launch_t<1, 1>(b, grid, s);
        case 1: return launch_t<1, 2>(b, grid, s);
        case 2: return launch_t<2, 1>(b, grid, s);
        case 3: return launch_t<2, 2>(b, grid, s);
        case 4: return launch_t<4, 1>(b, grid, s);
        case 5: return launch_t<4, 2>(b, grid, s);
        case 6: return launch_t<8, 1>(b, grid, s);
        case 8: return launch_t<16, 1>(b, grid, s);
    }
    return W12_ERR_ARG;
}

}  // namespace w12
