// kernels_tc.cu -- W12 decode-GEMM on the 5th-generation tensor cores
// (tcgen05, fp32 accumulator in tensor memory) for larger M.
//
// Swap-AB as in the mma.sync path: D[128 columns n][MP tokens] =
// W^T[n][k] . x[token][k], one UMMA of M = 128, N = MP (tokens padded to
// 16/32/64/128), K = 16 per instruction.  Work is cut into the same
// stream-K units as the mma.sync kernel (128 columns x 1024 k; the partial
// sums and the fix-up are shared) and every unit into stages of 64 k (one
// 128-byte swizzle atom).  Three roles per CTA:
//  - 8 decoder warps, two threads per output column (32 k each).  Each
//    thread streams its plane vectors and meta words a few stages ahead
//    with per-thread asynchronous copies into a private shared-memory ring,
//    rebuilds the bf16 weights in registers ("reconstructing bit by bit in
//    GEMM registers", SpecPilot summary, airadar.tv English edition,
//    "Reasons" bullet 2) and stores them as the stage's A tile: 128 rows x
//    128 bytes, K-major, 128-byte swizzle (16-byte chunk c of row r at
//    c ^ (r & 7)).  At the end of a column tile they read the accumulator
//    back with tcgen05.ld and write y (or stream-K partial sums);
//  - one producer warp copies the tokens' 64-k slice of x into the stage's
//    B tile (same layout) with asynchronous copies that arrive on the
//    stage's barrier when they land;
//  - one MMA warp: allocates the tensor memory, and one elected thread
//    issues the four tcgen05.mma of every stage once A and B are in place
//    and commits them to the stage's "empty" barrier (the stage may then be
//    refilled) and, at the end of a tile, to the accumulator barrier.  Two
//    accumulators alternate, so the next tile's products overlap the
//    epilogue of the previous one.
// Every mbarrier wait is bounded.  After a timeout all roles run on without
// waiting (so every thread still reaches every CTA barrier), the error word
// says W12_ERR_TIMEOUT, and the MMA thread waits (bounded) for its own
// products before the tensor memory is freed.
#include <cuda_runtime.h>

#include "async_common.cuh"
#include "gemm_common.cuh"

namespace w12 {

namespace {

constexpr int kDecWarps = 8;
constexpr int kDecThreads = kDecWarps * 32;
constexpr int kProdWarp = kDecWarps;      // x producer
constexpr int kMmaWarp = kDecWarps + 1;   // tensor-memory owner and MMA issuer
constexpr int kThreads = (kDecWarps + 2) * 32;
constexpr int kBK = 64;                   // k per stage (one 128-byte swizzle atom)
constexpr int kTile = kMmaCols;           // output columns per tile (UMMA M = 128)
constexpr int kUnit = kMmaUnitK;          // k per stream-K unit

// Ring depths: the plane prefetch ring keeps kRaw - 1 stages of weights in
// flight per thread (14 KB per stage and CTA), which is what hides the HBM
// latency; the A/B ring only decouples the decoders from the tensor core.
// Both are sized to fill the 227 KB of shared memory.
template <int MP>
struct TcCfg {
    static constexpr int kStages = MP >= 64 ? 3 : 4;  // A/B stage ring
    static constexpr int kRaw = MP >= 128 ? 8 : 10;   // plane prefetch ring
};

template <int MP>
struct TcSmem {
    static constexpr int kStages = TcCfg<MP>::kStages, kRaw = TcCfg<MP>::kRaw;
    uint8_t a[kStages][kTile * 128];      // 16 KB per stage, 1 KB aligned
    uint8_t b[kStages][MP * 128];
    uint4 raw[kRaw][3][kDecThreads];      // H, L, E vectors, lane-interleaved
    uint32_t rmeta[kRaw][2][kDecThreads]; // meta[g], meta[g + 1]
    uint64_t full[kStages], xfull[kStages], empty[kStages];
    uint64_t acc_done[2], tmem_free[2], fin;
    uint32_t tmem_addr;
    int last;
    int abort;
};

__host__ __device__ constexpr int tmem_cols(int mp) { return 2 * mp < 32 ? 32 : 2 * mp; }

__device__ __forceinline__ uint64_t desc_sw128(uint32_t addr) {
    uint64_t d = 0;
    d |= uint64_t((addr & 0x3FFFFu) >> 4);  // start address
    d |= uint64_t(16u >> 4) << 16;          // leading byte offset (not used with this swizzle)
    d |= uint64_t(1024u >> 4) << 32;        // stride byte offset: 8 rows x 128 B
    d |= uint64_t(1) << 46;                 // descriptor version
    d |= uint64_t(2) << 61;                 // 128-byte swizzle
    return d;
}

// D fp32, A and B bf16, both K-major, N = MP, M = 128.
template <int MP>
__device__ __forceinline__ uint32_t idesc_bf16() {
    return (1u << 4) | (1u << 7) | (1u << 10) | (uint32_t(MP >> 3) << 17) | (uint32_t(kTile >> 4) << 24);
}

__device__ __forceinline__ void mma_issue(uint32_t tmem, uint64_t ad, uint64_t bd, uint32_t idesc, uint32_t acc) {
    asm volatile(
        "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
        " tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}\n" ::"r"(tmem),
        "l"(ad), "l"(bd), "r"(idesc), "r"(acc)
        : "memory");
}

__device__ __forceinline__ void mma_commit(uint64_t *bar) {
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
                     smem_addr(bar))
                 : "memory");
}

__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void fence_async_smem() { asm volatile("fence.proxy.async.shared::cta;" ::: "memory"); }

// Arrive on `bar` once all of this thread's earlier cp.async copies landed.
__device__ __forceinline__ void cp_async_arrive_noinc(uint64_t *bar) {
    asm volatile("cp.async.mbarrier.arrive.noinc.shared::cta.b64 [%0];" ::"r"(smem_addr(bar)) : "memory");
}

__device__ __forceinline__ void tmem_ld16(uint32_t taddr, uint32_t (&r)[16]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
          "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
        : "r"(taddr));
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}

// Unit cursor over the batch: product gi, column tile nb, unit ks of the tile.
struct TcCur {
    int gi, nb, ks;
};

__device__ __forceinline__ void tc_next(const GemvBatch &b, TcCur &c) {
    if (++c.ks == b.g[c.gi].steps) {
        c.ks = 0;
        if (++c.nb == b.g[c.gi].NB) {
            c.nb = 0;
            ++c.gi;
        }
    }
}

__device__ __forceinline__ TcCur tc_at(const GemvBatch &b, int u) {
    TcCur c{0, 0, 0};
    while (c.gi + 1 < b.count && u >= b.g[c.gi + 1].ubase) ++c.gi;
    const int local = u - b.g[c.gi].ubase;
    c.nb = local / b.g[c.gi].steps;
    c.ks = local % b.g[c.gi].steps;
    return c;
}

// Flat walk over the stages of units [u, u1).
struct TcWalk {
    int u, u1, kb, kend;
    TcCur c;
    __device__ __forceinline__ void start(const GemvBatch &b) {
        if (u < u1) {
            kb = c.ks * kUnit;
            kend = min(b.g[c.gi].K, kb + kUnit);
        }
    }
    __device__ __forceinline__ void init(const GemvBatch &b, int u0, int u1_) {
        u = u0;
        u1 = u1_;
        c = TcCur{0, 0, 0};
        if (u < u1) c = tc_at(b, u);
        start(b);
    }
    __device__ __forceinline__ bool valid() const { return u < u1; }
    __device__ __forceinline__ void next(const GemvBatch &b) {
        kb += kBK;
        if (kb >= kend) {
            ++u;
            tc_next(b, c);
            start(b);
        }
    }
};

template <int MP>
__global__ void __launch_bounds__(kThreads, 1) tc_kernel(const __grid_constant__ GemvBatch b) {
    extern __shared__ __align__(1024) unsigned char smem_raw[];
    // the swizzle pattern repeats every 1 KB: align the stage tiles to it
    TcSmem<MP> &sm = *reinterpret_cast<TcSmem<MP> *>(
        smem_raw + ((1024u - (smem_addr(smem_raw) & 1023u)) & 1023u));
    constexpr int kStages = TcCfg<MP>::kStages, kRaw = TcCfg<MP>::kRaw;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int M = b.M;
    int u0, u1;
    {
        const int G = int(gridDim.x), c = int(blockIdx.x);
        const int per = b.U / G, rem = b.U % G;
        u0 = c * per + (c < rem ? c : rem);
        u1 = u0 + per + (c < rem ? 1 : 0);
    }
    if (tid == 0) {
        for (int s = 0; s < kStages; ++s) {
            mbar_init(&sm.full[s], kDecThreads);
            mbar_init(&sm.xfull[s], 32);
            mbar_init(&sm.empty[s], 1);
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(&sm.acc_done[i], 1);
            mbar_init(&sm.tmem_free[i], kDecThreads);
        }
        mbar_init(&sm.fin, 1);
        sm.abort = 0;
        mbar_fence_init();
    }
    if (warp == kMmaWarp) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                         smem_addr(&sm.tmem_addr)),
                     "r"(tmem_cols(MP))
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = sm.tmem_addr;

    if (warp == kMmaWarp) {
        // ---------------- MMA issuer ----------------
        if (lane == 0) {
            const uint32_t idesc = idesc_bf16<MP>();
            TcCur cc{0, 0, 0};
            if (u0 < u1) cc = tc_at(b, u0);
            uint32_t it = 0, seg = 0;
            bool ok = true;
            for (int u = u0; u < u1 && ok;) {
                const GemvOne &g = b.g[cc.gi];
                const int first = g.ubase + cc.nb * g.steps;
                const int ub = min(u1, first + g.steps);
                const uint32_t buf = seg & 1u;
                if (seg >= 2 && !mbar_wait(&sm.tmem_free[buf], ((seg >> 1) - 1) & 1u, &sm.abort, b.err)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const uint32_t dcol = tmem + buf * uint32_t(MP);
                uint32_t accumulate = 0;
                for (; u < ub && ok; ++u) {
                    const int kst = cc.ks * kUnit, kend = min(g.K, kst + kUnit);
                    tc_next(b, cc);
                    for (int kb = kst; kb < kend; kb += kBK, ++it) {
                        const uint32_t s = it % kStages, par = (it / kStages) & 1u;
                        if (!mbar_wait(&sm.full[s], par, &sm.abort, b.err) ||
                            !mbar_wait(&sm.xfull[s], par, &sm.abort, b.err)) {
                            ok = false;
                            break;
                        }
                        tc_fence_after();
                        fence_async_smem();
                        const uint32_t abase = smem_addr(&sm.a[s][0]), bbase = smem_addr(&sm.b[s][0]);
#pragma unroll
                        for (int k16 = 0; k16 < kBK / 16; ++k16) {
                            mma_issue(dcol, desc_sw128(abase + 32 * k16), desc_sw128(bbase + 32 * k16), idesc,
                                      accumulate);
                            accumulate = 1;
                        }
                        mma_commit(&sm.empty[s]);
                    }
                }
                if (ok) mma_commit(&sm.acc_done[buf]);
                ++seg;
            }
            // every product issued has completed before the memory is freed
            mma_commit(&sm.fin);
            volatile int no_abort = 0;
            mbar_wait(&sm.fin, 0, &no_abort, b.err);
        }
    } else if (warp == kProdWarp) {
        // ---------------- x producer ----------------
        TcWalk wk;
        wk.init(b, u0, u1);
        for (uint32_t it = 0; wk.valid(); ++it, wk.next(b)) {
            const GemvOne &g = b.g[wk.c.gi];
            const uint32_t s = it % kStages;
            if (it >= uint32_t(kStages)) mbar_wait(&sm.empty[s], ((it / kStages) - 1) & 1u, &sm.abort, b.err);
            const uint32_t bs = smem_addr(&sm.b[s][0]);
            for (int i = lane; i < M * 8; i += 32) {
                const int r = i >> 3, c = i & 7;
                cp_async16(bs + uint32_t(r * 128 + ((c ^ (r & 7)) * 16)),
                           g.x + (uint32_t(r) * uint32_t(g.K) + uint32_t(wk.kb + 8 * c)));
            }
            cp_async_arrive_noinc(&sm.xfull[s]);
        }
        cp_async_wait<0>();
    } else {
        // ---------------- decoders ----------------
        const int row = tid >> 1, half = tid & 1;  // column within the tile, 32-k half of the stage
        const uint64_t pol = l2_evict_first_policy();
        TcWalk pf;  // prefetch walk, kRaw - 1 stages ahead of the consumer
        pf.init(b, u0, u1);
        auto prefetch = [&](uint32_t slot) {
            if (pf.valid()) {
                const GemvOne &g = b.g[pf.c.gi];
                const int n = pf.c.nb * kTile + row;
                if (n < g.N) {
                    const uint32_t wo = uint32_t(n) * uint32_t(g.KW) + uint32_t((pf.kb + 32 * half) >> 3);
                    cp_async16_stream(smem_addr(&sm.raw[slot][0][tid]), g.H + wo, pol);
                    cp_async16_stream(smem_addr(&sm.raw[slot][1][tid]), g.L + wo, pol);
                    cp_async16_stream(smem_addr(&sm.raw[slot][2][tid]), g.E + wo, pol);
                    const uint32_t gg = uint32_t(n) * uint32_t(g.KG) + uint32_t(pf.kb >> 7);
                    cp_async4(smem_addr(&sm.rmeta[slot][0][tid]), g.meta + gg);
                    cp_async4(smem_addr(&sm.rmeta[slot][1][tid]), g.meta + gg + 1);
                }
                pf.next(b);
            }
            cp_async_commit();
        };
#pragma unroll
        for (int p = 0; p < kRaw - 1; ++p) prefetch(uint32_t(p));

        uint32_t it = 0, seg = 0;
        TcCur cc{0, 0, 0};
        if (u0 < u1) cc = tc_at(b, u0);
        for (int u = u0; u < u1;) {
            const GemvOne &g = b.g[cc.gi];
            const int nb = cc.nb, first = g.ubase + nb * g.steps;
            const int ua = u, ub = min(u1, first + g.steps);
            const bool col_ok = nb * kTile + row < g.N;
            for (; u < ub; ++u) {
                const int kst = cc.ks * kUnit, kend = min(g.K, kst + kUnit);
                tc_next(b, cc);
                for (int kb = kst; kb < kend; kb += kBK, ++it) {
                    prefetch((it + kRaw - 1) % kRaw);
                    cp_async_wait<kRaw - 1>();  // this stage's planes have landed
                    const uint32_t rs = it % kRaw;
                    uint32_t w[16];
                    if (col_ok) {
                        const uint4 h = lds128(smem_addr(&sm.raw[rs][0][tid]));
                        const uint4 l = lds128(smem_addr(&sm.raw[rs][1][tid]));
                        const uint4 e = lds128(smem_addr(&sm.raw[rs][2][tid]));
                        const uint32_t m0 = lds32(smem_addr(&sm.rmeta[rs][0][tid]));
                        const uint32_t m1 = lds32(smem_addr(&sm.rmeta[rs][1][tid]));
                        rebuild32(h, l, e, base4(m0), w);
                        if ((m0 >> 8) != (m1 >> 8))
                            patch_escapes(w, m0, m1, uint32_t((kb + 32 * half) & 127), g.esc, g.n_esc, b.err);
                    } else {
#pragma unroll
                        for (int i = 0; i < 16; ++i) w[i] = 0u;
                    }
                    const uint32_t s = it % kStages;
                    if (it >= uint32_t(kStages))  // the products that last read this stage are done
                        mbar_wait(&sm.empty[s], ((it / kStages) - 1) & 1u, &sm.abort, b.err);
                    uint8_t *arow = &sm.a[s][row * 128];
#pragma unroll
                    for (int q = 0; q < 4; ++q) {
                        const int c = 4 * half + q;
                        *reinterpret_cast<uint4 *>(arow + ((c ^ (row & 7)) * 16)) =
                            make_uint4(w[4 * q], w[4 * q + 1], w[4 * q + 2], w[4 * q + 3]);
                    }
                    fence_async_smem();  // generic-proxy stores -> tensor-core reads
                    mbar_arrive(&sm.full[s]);
                }
            }
            // Tile done: warps w and w + 4 read TMEM lanes 32 (w % 4) .. + 31 (output
            // columns), the first and second half of the token columns.
            const uint32_t buf = seg & 1u;
            mbar_wait(&sm.acc_done[buf], (seg >> 1) & 1u, &sm.abort, b.err);
            tc_fence_after();
            {
                const int quarter = warp & 3, colhalf = warp >> 2;
                const int nrow = nb * kTile + 32 * quarter + lane;
                const bool whole = (ua == first) && (ub == first + g.steps);
                constexpr int kCols = MP / 2 < 16 ? 16 : MP / 2;
                const int c_begin = MP / 2 < 16 ? 0 : colhalf * (MP / 2);
                __syncwarp();  // tcgen05.ld is warp-collective
                if (MP / 2 >= 16 || colhalf == 0) {
#pragma unroll
                    for (int c0 = 0; c0 < kCols; c0 += 16) {
                        uint32_t r[16];
                        tmem_ld16(tmem + (uint32_t(32 * quarter) << 16) + buf * uint32_t(MP) +
                                      uint32_t(c_begin + c0),
                                  r);
                        const int m0 = c_begin + c0;  // tokens m0 .. m0 + 15, column nrow
                        const int mc = min(16, M - m0);
                        if (nrow < g.N && mc > 0) {
                            if (!whole) {
                                float *pp = g.partial +
                                            (uint32_t(ua - g.ubase) * uint32_t(M) + uint32_t(m0)) * kTile +
                                            uint32_t(nrow - nb * kTile);
#pragma unroll
                                for (int j = 0; j < 16; ++j)
                                    if (j < mc) pp[j * kTile] = __uint_as_float(r[j]);
                            } else if (b.y_dtype == W12_F32) {
                                float *yp = static_cast<float *>(g.y) + size_t(m0) * size_t(g.N) + nrow;
#pragma unroll
                                for (int j = 0; j < 16; ++j, yp += g.N)
                                    if (j < mc) *yp = __uint_as_float(r[j]);
                            } else {
                                __nv_bfloat16 *yp =
                                    static_cast<__nv_bfloat16 *>(g.y) + size_t(m0) * size_t(g.N) + nrow;
#pragma unroll
                                for (int j = 0; j < 16; ++j, yp += g.N)
                                    if (j < mc) *yp = __float2bfloat16_rn(__uint_as_float(r[j]));
                            }
                        }
                    }
                }
                tc_fence_before();
                mbar_arrive(&sm.tmem_free[buf]);  // this accumulator may be overwritten
                ++seg;
                if (!whole)
                    streamk_fixup_raw(g.counters, g.partial, first, g.ubase, g.steps, b.U, M, g.N, g.y, b.y_dtype, kTile,
                              nb, ub - ua, &sm.last, tid, kDecThreads);
            }
        }
        cp_async_wait<0>();
    }
    tc_fence_before();
    __syncthreads();
    if (warp == kMmaWarp) {
        __syncwarp();
        tc_fence_after();
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(tmem_cols(MP))
                     : "memory");
    }
}

template <int MP>
constexpr size_t tc_smem() {
    return sizeof(TcSmem<MP>) + 1024;  // + slack for the 1 KB alignment
}

// The dynamic shared-memory limit is raised once per device by occ_tc_t(),
// which the planner always runs before the first launch on a device.
template <int MP>
int launch_tc_t(const GemvBatch &b, int grid, cudaStream_t s) {
    tc_kernel<MP><<<unsigned(grid), kThreads, tc_smem<MP>(), s>>>(b);
    return cudaGetLastError() == cudaSuccess ? W12_OK : W12_ERR_CUDA;
}

template <int MP>
int occ_tc_t(int *blocks) {
    if (cudaFuncSetAttribute(tc_kernel<MP>, cudaFuncAttributeMaxDynamicSharedMemorySize, int(tc_smem<MP>())) !=
        cudaSuccess)
        return W12_ERR_CUDA;
    return cudaOccupancyMaxActiveBlocksPerMultiprocessor(blocks, tc_kernel<MP>, kThreads, tc_smem<MP>()) ==
                   cudaSuccess
               ? W12_OK
               : W12_ERR_CUDA;
}

}  // namespace

// variant v: MP = 16 << v tokens (16, 32, 64, 128)
int launch_tc_batch(const GemvBatch &b, int variant, int grid, void *stream) {
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    switch (variant) {
        case 0: return launch_tc_t<16>(b, grid, s);
        case 1: return launch_tc_t<32>(b, grid, s);
        case 2: return launch_tc_t<64>(b, grid, s);
        case 3: return launch_tc_t<128>(b, grid, s);
    }
    return W12_ERR_ARG;
}

int tc_occupancy(int variant, int *blocks) {
    switch (variant) {
        case 0: return occ_tc_t<16>(blocks);
        case 1: return occ_tc_t<32>(blocks);
        case 2: return occ_tc_t<64>(blocks);
        case 3: return occ_tc_t<128>(blocks);
    }
    return W12_ERR_ARG;
}

}  // namespace w12
