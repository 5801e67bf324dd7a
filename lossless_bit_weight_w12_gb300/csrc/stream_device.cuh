// stream_device.cuh -- device pieces shared by the TMA-fed stream-K
// decode-GEMM kernels (kernels_stream.cu: mma.sync; kernels_tc.cu: tcgen05):
// tensor-copy and barrier primitives, the unit cursor and the stream-K
// fix-up.
#pragma once

#include <cuda.h>

#include <cstdint>

#include "async_common.cuh"
#include "gemm_common.cuh"
#include "stream_common.h"

namespace w12 {

constexpr int kTileN = 128;               // columns per tile
constexpr int kPlaneBytes = kTileN * 64;  // one plane box: 128 columns x 128 k
constexpr int kMetaBytes = kTileN * 8;    // meta[g], meta[g + 1] per column
constexpr int kEscPrefetchLines = 64;     // escape lines prefetched per tile piece (8 KB)

__device__ __forceinline__ uint2 lds64(uint32_t addr) {
    uint2 r;
    asm volatile("ld.shared.v2.u32 {%0,%1}, [%2];" : "=r"(r.x), "=r"(r.y) : "r"(addr));
    return r;
}

__device__ __forceinline__ void tma_2d(uint32_t dst, const CUtensorMap *map, int c0, int c1, uint64_t *bar,
                                       uint64_t policy) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.L2::cache_hint"
        " [%0], [%1, {%2, %3}], [%4], %5;" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(smem_addr(bar)), "l"(policy)
        : "memory");
}

__device__ __forceinline__ void tma_3d(uint32_t dst, const CUtensorMap *map, int c0, int c1, int c2,
                                       uint64_t *bar) {
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%2, %3, %4}], [%5];" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(c2), "r"(smem_addr(bar))
        : "memory");
}

__device__ __forceinline__ void tma_2d_keep(uint32_t dst, const CUtensorMap *map, int c0, int c1, uint64_t *bar) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%2, %3}], [%4];" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(smem_addr(bar))
        : "memory");
}

// Arrive on `bar` once every earlier cp.async of this thread has landed
// (counts as one of the barrier's expected arrivals).
__device__ __forceinline__ void cp_async_mbar_arrive_noinc(uint64_t *bar) {
    asm volatile("cp.async.mbarrier.arrive.noinc.shared::cta.b64 [%0];" ::"r"(smem_addr(bar)) : "memory");
}

__device__ __forceinline__ void prefetch_l1(const void *p) {
    asm volatile("prefetch.global.L1 [%0];" ::"l"(p));
}

// Bounded wait that ignores the abort flag (used only to let copies that
// are already in flight land before the CTA exits after a timeout).
__device__ __forceinline__ void mbar_drain(uint64_t *bar, uint32_t parity) {
    const uint64_t t0 = global_timer_ns();
    while (!mbar_try_wait(bar, parity)) {
        if (global_timer_ns() - t0 > kWaitLimitNs) return;
        __nanosleep(64);
    }
}

// Unit cursor: product gi, column tile nb, group kg.
struct SCur {
    int gi, nb, kg;
};

__device__ __forceinline__ SCur s_at(const StreamBatch &b, int u) {
    SCur c{0, 0, 0};
    while (c.gi + 1 < b.count && u >= b.g[c.gi + 1].ubase) ++c.gi;
    const int local = u - b.g[c.gi].ubase;
    c.nb = local / b.g[c.gi].KG;
    c.kg = local % b.g[c.gi].KG;
    return c;
}

__device__ __forceinline__ void s_next_tile(const StreamBatch &b, SCur &c) {
    c.kg = 0;
    if (++c.nb == b.g[c.gi].NB) {
        c.nb = 0;
        ++c.gi;
    }
}

__device__ __forceinline__ void s_next(const StreamBatch &b, SCur &c) {
    if (++c.kg == b.g[c.gi].KG) s_next_tile(b, c);
}

// Stream-K fix-up.  A tile (one product, 128 columns) covers the units
// [first, first + KG); CTA c's piece of it is stored in partial slot
// (c, 0) if the piece starts at c's first unit, else (c, 1) (only a CTA's
// first and last pieces can be split).  Each piece adds its unit count to
// counters[nb]; the CTA that completes the count sums the pieces' slots in
// CTA order (the same bits on every call), writes y and resets the counter.
template <bool FUSED>
__device__ __forceinline__ void stream_fixup(const StreamBatch &b, const StreamOne &g, int first, int nb,
                                             int count, int *s_last, int tid, int nthreads,
                                             unsigned long long *s_best) {
    __threadfence();
    named_sync(nthreads);
    if (tid == 0) {
        const uint32_t old = atomicAdd(&g.counters[nb], uint32_t(count));
        *s_last = (int(old) + count == g.KG);
    }
    named_sync(nthreads);
    if (*s_last) {
        __threadfence();
        const int G = int(gridDim.x), per = b.U / G, rem = b.U % G;
        const int c_first = sk_cta_of(first, per, rem), c_last = sk_cta_of(first + g.KG - 1, per, rem);
        const int M = b.M;
        const size_t slot_floats = size_t(M) * kTileN;
        for (int o = tid; o < M * (kTileN / 4); o += nthreads) {
            const int m = o / (kTileN / 4), c4 = o % (kTileN / 4);
            float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
            for (int c = c_first; c <= c_last; ++c) {
                const int slot = sk_unit_begin(c, per, rem) >= first ? 0 : 1;
                const float4 v = __ldcg(reinterpret_cast<const float4 *>(
                    b.partial + (size_t(c) * 2 + slot) * slot_floats + size_t(m) * kTileN) + c4);
                if (c == c_first) {
                    acc = v;
                } else {
                    acc.x += v.x;
                    acc.y += v.y;
                    acc.z += v.z;
                    acc.w += v.w;
                }
            }
            const int n0 = nb * kTileN + 4 * c4;
            const float r[4] = {acc.x, acc.y, acc.z, acc.w};
            unsigned long long best = 0ull;
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                if (n0 + e >= g.N) continue;
                if (!FUSED || g.y) store_out(g.y, b.y_dtype, g.N, m, n0 + e, r[e]);
                if (FUSED) {
                    const unsigned long long k = pack_key(r[e], uint32_t(n0 + e));
                    best = k > best ? k : best;
                }
            }
            if (FUSED && best != 0ull) atomicMax(&s_best[m], best);
        }
        if (tid == 0) g.counters[nb] = 0u;
    }
    named_sync(nthreads);  // s_last is reused by the next piece
}


// The producer warp of a stream kernel: for every unit of [u0, u1), once
// the stage's previous contents are released (empty[s]), start the copies
// of the unit into ring stage s and arm full[s]:
//  - the H, L, E plane boxes (2-D tensor copies, evict-first in L2) at
//    x_bytes, x_bytes + 8 KB, x_bytes + 16 KB of the stage;
//  - x at the stage start: one 3-D box (every token, both 64-k halves,
//    mma.sync layout), or (TC) two 2-D boxes of 64 k x MP tokens, the
//    second at MP * 128 bytes (the canonical K-major tcgen05 operand);
//  - meta[g], meta[g + 1] of each of the tile's columns (4-byte cp.async by
//    the 32 lanes, which then arrive on full[s] as they land), at
//    x_bytes + 24 KB.
// At the start of every tile piece the piece's escape entries (a contiguous
// range of the escape list) are prefetched into L1.  full[s] expects 33
// arrivals (32 lanes + the expect_tx) and the tensor bytes.
template <int S, bool TC>
__device__ __forceinline__ void stream_producer(const StreamBatch &b, uint32_t base, int stage_bytes,
                                                int x_bytes, int mp, uint64_t *full, uint64_t *empty,
                                                int *abort, int u0, int u1, int lane) {
    const uint64_t pol = l2_evict_first_policy();
    const uint32_t kH = uint32_t(x_bytes), kL = kH + kPlaneBytes, kE = kL + kPlaneBytes, kMeta = kE + kPlaneBytes;
    const uint32_t tx = uint32_t(x_bytes + 3 * kPlaneBytes);
    SCur c = s_at(b, u0);
    int s = 0, issued = 0;
    uint32_t ph = 0;
    for (int u = u0; u < u1; ++u) {
        const StreamOne &g = b.g[c.gi];
        if (issued >= S && !mbar_wait(&empty[s], ph ^ 1u, abort, b.err)) break;
        if (u == u0 || c.kg == 0) {
            // escape entries of this tile piece: groups [kga, kgb) of
            // columns n0 .. nl, one contiguous range of the list
            const int first = g.ubase + c.nb * g.KG;
            const int kgb = min(u1, first + g.KG) - first;
            const int n0 = c.nb * kTileN, nl = min(g.N, n0 + kTileN) - 1;
            uint32_t lo = 0, hi = 0;
            if (lane == 0) {
                lo = ldg_u32(g.meta + (uint32_t(n0) * uint32_t(g.KG) + uint32_t(c.kg))) >> 8;
                hi = ldg_u32(g.meta + (uint32_t(nl) * uint32_t(g.KG) + uint32_t(kgb))) >> 8;
            }
            lo = __shfl_sync(0xFFFFFFFFu, lo, 0);
            hi = min(__shfl_sync(0xFFFFFFFFu, hi, 0), g.n_esc);
            if (lo < hi) {
                const uintptr_t a0 = reinterpret_cast<uintptr_t>(g.esc + lo) & ~uintptr_t(127);
                const uintptr_t a1 = reinterpret_cast<uintptr_t>(g.esc + hi);
                for (int q = lane; q < kEscPrefetchLines; q += 32) {
                    const uintptr_t a = a0 + uintptr_t(q) * 128u;
                    if (a < a1) prefetch_l1(reinterpret_cast<const void *>(a));
                }
            }
        }
        const uint32_t st = base + uint32_t(s) * uint32_t(stage_bytes);
#pragma unroll
        for (int q = 0; q < kTileN / 32; ++q) {
            const int row = lane + 32 * q, n = c.nb * kTileN + row;
            if (n < g.N) {
                const uint32_t gi = uint32_t(n) * uint32_t(g.KG) + uint32_t(c.kg);
                cp_async4(st + kMeta + uint32_t(row) * 8u, g.meta + gi);
                cp_async4(st + kMeta + uint32_t(row) * 8u + 4u, g.meta + gi + 1);
            }
        }
        cp_async_mbar_arrive_noinc(&full[s]);
        if (lane == 0) {
            mbar_expect_tx(&full[s], tx);
            tma_2d(st + kH, &g.th, c.kg * 16, c.nb * kTileN, &full[s], pol);
            tma_2d(st + kL, &g.tl, c.kg * 16, c.nb * kTileN, &full[s], pol);
            tma_2d(st + kE, &g.te, c.kg * 16, c.nb * kTileN, &full[s], pol);
            if (TC) {
                tma_2d_keep(st, &g.tx, 128 * c.kg, 0, &full[s]);
                tma_2d_keep(st + uint32_t(mp) * 128u, &g.tx, 128 * c.kg + 64, 0, &full[s]);
            } else {
                tma_3d(st, &g.tx, 0, 2 * c.kg, 0, &full[s]);
            }
        }
        s_next(b, c);
        ++issued;
        if (++s == S) {
            s = 0;
            ph ^= 1u;
        }
    }
    cp_async_wait<0>();
    if (*reinterpret_cast<volatile int *>(abort)) {
        // let the tensor copies already issued land before the CTA exits
        for (int k = 0; k < S && k < issued; ++k) {
            if (--s < 0) {
                s = S - 1;
                ph ^= 1u;
            }
            mbar_drain(&full[s], ph);
        }
    }
}

}  // namespace w12
