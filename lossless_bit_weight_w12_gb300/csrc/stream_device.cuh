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

constexpr int kTileN = kTileCols;         // columns per tile
constexpr int kEscPrefetchLines = 64;     // escape lines prefetched per tile piece (8 KB)

// Bulk global -> shared copy (TMA engine) to a shared-memory address;
// completion counted in bytes on `bar`.  dst, src 16-byte aligned, bytes a
// multiple of 16.
__device__ __forceinline__ void bulk_copy(uint32_t dst, const void *src, uint32_t bytes, uint64_t *bar,
                                          uint64_t policy) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint"
        " [%0], [%1], %2, [%3], %4;" ::"r"(dst),
        "l"(src), "r"(bytes), "r"(smem_addr(bar)), "l"(policy)
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


__device__ __forceinline__ void prefetch_l1(const void *p) {
    asm volatile("prefetch.global.L1 [%0];" ::"l"(p));
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
        const int total = M * (kTileN / 4);
        // four outputs per thread and round trip, summed in CTA order (the
        // same bits on every call)
        for (int o0 = tid; o0 < total; o0 += 4 * nthreads) {
            float4 acc[4];
#pragma unroll
            for (int k = 0; k < 4; ++k) acc[k] = make_float4(0.f, 0.f, 0.f, 0.f);
            for (int c = c_first; c <= c_last; ++c) {
                const int slot = sk_unit_begin(c, per, rem) >= first ? 0 : 1;
                const float4 *P = reinterpret_cast<const float4 *>(b.partial + (size_t(c) * 2 + slot) * slot_floats);
                float4 v[4];
#pragma unroll
                for (int k = 0; k < 4; ++k) {
                    const int o = o0 + k * nthreads;
                    v[k] = o < total ? __ldcg(P + o) : make_float4(0.f, 0.f, 0.f, 0.f);  // [m][c4] = o
                }
#pragma unroll
                for (int k = 0; k < 4; ++k) {
                    if (c == c_first) {
                        acc[k] = v[k];
                    } else {
                        acc[k].x += v[k].x;
                        acc[k].y += v[k].y;
                        acc[k].z += v[k].z;
                        acc[k].w += v[k].w;
                    }
                }
            }
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                const int o = o0 + k * nthreads;
                if (o >= total) break;
                const int m = o / (kTileN / 4), c4 = o % (kTileN / 4);
                const int n0 = nb * kTileN + 4 * c4;
                const float r[4] = {acc[k].x, acc[k].y, acc[k].z, acc[k].w};
                unsigned long long best = 0ull;
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    if (n0 + e >= g.N) continue;
                    if (!FUSED || g.y) store_out(g.y, b.y_dtype, g.N, m, n0 + e, r[e]);
                    if (FUSED) {
                        const unsigned long long key = pack_key(r[e], uint32_t(n0 + e));
                        best = key > best ? key : best;
                    }
                }
                if (FUSED && best != 0ull) atomicMax(&s_best[m], best);
            }
        }
        if (tid == 0) g.counters[nb] = 0u;
    }
    named_sync(nthreads);  // s_last is reused by the next piece
}


// The unit block of cursor c (format v2: unit t * KG + kg of the product).
__device__ __forceinline__ const uint8_t *unit_block(const StreamOne &g, const SCur &c) {
    return g.units + size_t(uint32_t(c.nb) * uint32_t(g.KG) + uint32_t(c.kg)) * kUnitBytes;
}

// At the start of a tile piece (units u .. of tile c.nb, ending at the
// tile's last group or at u1), prefetch the piece's escape entries into
// L1: escapes are listed by unit, so they are one contiguous range, from
// the first unit's first column to the end of the piece's last unit.
// At most kEscPrefetchLines lines.
__device__ __forceinline__ void prefetch_piece_escapes(const StreamOne &g, const SCur &c, const uint8_t *unit,
                                                       int u, int u1) {
    const int first = g.ubase + c.nb * g.KG;
    const int nunits = min(u1, first + g.KG) - u;
    const uint32_t lo = ldg_u32(reinterpret_cast<const uint32_t *>(unit + kMetaAt)) >> 8;
    const uint32_t hi = min(ldg_u32(reinterpret_cast<const uint32_t *>(unit + size_t(nunits - 1) * kUnitBytes +
                                                                       kMetaAt + 4 * kTileN)) >> 8,
                            g.n_esc);
    if (lo < hi) {
        const uintptr_t a0 = reinterpret_cast<uintptr_t>(g.esc + lo) & ~uintptr_t(127);
        const uintptr_t a1 = reinterpret_cast<uintptr_t>(g.esc + hi);
        for (int q = 0; q < kEscPrefetchLines; ++q) {
            const uintptr_t a = a0 + uintptr_t(q) * 128u;
            if (a >= a1) break;
            prefetch_l1(reinterpret_cast<const void *>(a));
        }
    }
}

// Programmatic dependent launch: a stream kernel lets the next kernel of
// the stream start as soon as this grid's CTAs free their SMs
// (pdl_launch), and waits for the previous grid to complete, with its
// memory visible, before it reads x or writes anything (pdl_wait).  Both
// are no-ops for launches without the programmatic-serialization attribute.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_launch() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

// The producer warp of a stream kernel: for every unit of [u0, u1), once
// the stage's previous contents are released (empty[s]), lane 0 starts the
// copies of the unit into ring stage s and arms full[s] (one arrival and the
// bytes):
//  - the unit block (planes and meta words, kUnitBytes, evict-first in L2)
//    with one bulk copy, at x_bytes;
//  - x at the stage start: one 3-D box (every token, both 64-k halves,
//    mma.sync layout), or (TC) two 2-D boxes of 64 k x MP tokens, the
//    second at MP * 128 bytes (the canonical K-major tcgen05 operand).
// Nothing is read before griddepcontrol.wait (the previous kernel of the
// stream may have written the blob or x), unless the launch asked for the
// early weight stream (b.early_weights): then the first ring's worth of
// unit blocks is requested before it, overlapping the previous kernel's
// tail, and x only after it.
// At the start of every tile piece it prefetches the piece's escape entries
// (a contiguous range of the escape list: escapes are listed by unit, and a
// piece is consecutive units) into L1.
// The test hook b.withhold_unit leaves one unit's stage unarmed: its
// consumers' bounded wait runs out (W12_ERR_TIMEOUT).
template <int S, bool TC>
__device__ __forceinline__ void stream_producer(const StreamBatch &b, uint32_t base, int stage_bytes,
                                                int x_bytes, int mp, uint64_t *full, uint64_t *empty,
                                                WaitCtl *ctl, int u0, int u1, int lane) {
    if (lane != 0) return;
    const uint64_t pol = l2_evict_first_policy();
    const uint32_t tx = uint32_t(x_bytes + kUnitBytes);
    auto issue_weights = [&](const SCur &c, int u, uint32_t st, uint64_t *bar) {
        if (u == b.withhold_unit) return;
        const StreamOne &g = b.g[c.gi];
        const uint8_t *unit = unit_block(g, c);
        if (u == u0 || c.kg == 0) prefetch_piece_escapes(g, c, unit, u, u1);
        mbar_expect_tx(bar, tx);
        bulk_copy(st + uint32_t(x_bytes), unit, kUnitBytes, bar, pol);
    };
    auto issue_x = [&](const SCur &c, int u, uint32_t st, uint64_t *bar) {
        if (u == b.withhold_unit) return;
        const StreamOne &g = b.g[c.gi];
        if (TC) {
            tma_2d_keep(st, &g.tx, 128 * c.kg, 0, bar);
            tma_2d_keep(st + uint32_t(mp) * 128u, &g.tx, 128 * c.kg + 64, 0, bar);
        } else {
            tma_3d(st, &g.tx, 0, 2 * c.kg, 0, bar);
        }
    };
    // the first ring's worth of weights (before or after the dependency),
    // then their x
    SCur c = s_at(b, u0);
    const int P = min(S, u1 - u0);
    SCur first_c[S];
    if (!b.early_weights) pdl_wait();
    for (int k = 0; k < P; ++k) {
        first_c[k] = c;
        issue_weights(c, u0 + k, base + uint32_t(k) * uint32_t(stage_bytes), &full[k]);
        s_next(b, c);
    }
    if (b.early_weights) pdl_wait();
    for (int k = 0; k < P; ++k)
        issue_x(first_c[k], u0 + k, base + uint32_t(k) * uint32_t(stage_bytes), &full[k]);
    int s = P == S ? 0 : P, issued = P;
    uint32_t ph = P == S ? 1u : 0u;
    for (int u = u0 + P; u < u1; ++u) {
        // a consumer that gave up arrives without waiting for its copy, and
        // sets the abort flag before that arrival: stop here, so that every
        // copy in flight is among the last ring's worth drained below
        if (!mbar_wait(&empty[s], ph ^ 1u, ctl, b.err) || aborted(ctl)) break;
        const uint32_t st = base + uint32_t(s) * uint32_t(stage_bytes);
        issue_weights(c, u, st, &full[s]);
        issue_x(c, u, st, &full[s]);
        s_next(b, c);
        ++issued;
        if (++s == S) {
            s = 0;
            ph ^= 1u;
        }
    }
    if (aborted(ctl)) {
        // let the copies already issued land before the CTA exits
        for (int k = 0; k < S && k < issued; ++k) {
            if (--s < 0) {
                s = S - 1;
                ph ^= 1u;
            }
            mbar_drain(&full[s], ph, ctl->limit_ns);
        }
    }
}

// Set up the CTA's wait state (one thread, before the CTA's first barrier).
__device__ __forceinline__ void wait_ctl_init(WaitCtl *ctl, const StreamBatch &b) {
    ctl->abort = 0;
    ctl->limit_ns = b.wait_ns ? b.wait_ns : kWaitLimitNs;
}

}  // namespace w12
