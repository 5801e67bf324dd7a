// kernels_encode.cu -- the W12 encoder on the GPU (same bytes as the host
// encoder in encode.cpp and as the format text in include/w12.h).
//
// Loading a model through the host encoder means scanning every weight on a
// few CPU cores; here the same three steps run on the device:
//  1. scan: one half-warp per group (128 k of one column): the base (the
//     window [b, b+14], b <= 240, holding the most exponents, the largest b
//     on a tie) and the escape count 128 - cover -- from the group's
//     exponent range when it fits one window, else from its histogram;
//  2. an exclusive scan of the escape counts in unit, then column order
//     (the order of the escape list), giving every group's first escape;
//  3. pack: one half-warp per (unit, column): lane q builds word q of the
//     H, L and E planes (pos 8q .. 8q+7) and stores it at its swizzled place;
//     escaped weights write their entries at first_escape + rank (ballot
//     prefix); meta words follow.
// Padding columns (past N) get base 0, no escapes and zero plane bytes; the
// pack kernel writes every byte of the unit blocks, and the gap before the
// escape list and the tail after it are zero-filled.  Both kernels keep the
// loads of the next three groups in flight while they process one.
#include <cuda_runtime.h>

#include "async_common.cuh"
#include "w12_internal.h"

namespace w12 {

namespace {

constexpr int kScanBlock = 1024;  // threads of a scan block

struct EncArgs {
    const uint16_t *w;  // [N][K] (NK) or [K][N] (KN)
    int64_t K, N, KG;
    int layout;
    int64_t U;          // unit blocks
    uint8_t *base;      // [U * 128]
    uint32_t *count;    // [U * 128], then exclusive scan in place -> begin
    uint32_t *block_sum;
    uint8_t *blob;
    uint64_t off_esc, n_esc;
};

// A group (128 k of one column) is handled by a half-warp: lane q = 0..15
// of the half holds the 8 weights pos 8q .. 8q+7.  hmask: the half's lanes.
__device__ __forceinline__ unsigned half_mask(int lane) { return lane < 16 ? 0x0000FFFFu : 0xFFFF0000u; }

__device__ __forceinline__ void load8(const EncArgs &a, int64_t n, int64_t kg, int q, uint16_t (&v)[8]) {
    const int64_t k0 = kg * kGroup + 8 * q;
    if (a.layout == W12_LAYOUT_NK) {
        const uint4 r = *reinterpret_cast<const uint4 *>(a.w + n * a.K + k0);  // 16-byte aligned: K % 128 == 0
        const uint32_t wq[4] = {r.x, r.y, r.z, r.w};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            v[2 * i] = uint16_t(wq[i]);
            v[2 * i + 1] = uint16_t(wq[i] >> 16);
        }
    } else {
#pragma unroll
        for (int i = 0; i < 8; ++i) v[i] = a.w[(k0 + i) * a.N + n];
    }
}

// Base and escape count of one group, computed by a half-warp.  When every
// exponent lies in [emin, emin + 14] and emin <= 240, the window of the
// largest base covering all 128 starts at emin: base emin, no escapes
// (the common case).  Otherwise the exponent histogram (hist: the half's
// 256 shared counters) gives cover(b) = #exp in [b, b+14] for every b <= 240,
// and the best cover wins, the largest b on a tie.
__device__ __forceinline__ void group_base_half(const uint16_t (&v)[8], int q, unsigned hmask, uint32_t *hist,
                                                uint32_t &b_out, uint32_t &esc_out) {
    uint32_t e[8], lo = 255u, hi = 0u;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        e[i] = (v[i] >> 7) & 0xFFu;
        lo = min(lo, e[i]);
        hi = max(hi, e[i]);
    }
    lo = __reduce_min_sync(hmask, lo);
    hi = __reduce_max_sync(hmask, hi);
    if (hi - lo <= 14u && lo <= uint32_t(kMaxBase)) {
        b_out = lo;
        esc_out = 0u;
        return;
    }
#pragma unroll
    for (int i = 0; i < 16; ++i) hist[q * 16 + i] = 0u;
    __syncwarp(hmask);
#pragma unroll
    for (int i = 0; i < 8; ++i) atomicAdd(&hist[e[i]], 1u);
    __syncwarp(hmask);
    // inclusive prefix of the histogram: lane q owns bins 16q .. 16q+15
    uint32_t p[16];
    uint32_t run = 0;
#pragma unroll
    for (int i = 0; i < 16; ++i) {
        run += hist[q * 16 + i];
        p[i] = run;
    }
    uint32_t excl = run;  // inclusive scan of the lane totals over the half, then shift
#pragma unroll
    for (int off = 1; off < 16; off <<= 1) {
        const uint32_t o = __shfl_up_sync(hmask, excl, off, 16);
        if (q >= off) excl += o;
    }
    excl -= run;
    __syncwarp(hmask);
#pragma unroll
    for (int i = 0; i < 16; ++i) hist[q * 16 + i] = p[i] + excl;  // hist[e] = #exp <= e
    __syncwarp(hmask);
    // maximise (cover << 8 | b): the best cover, the largest b on ties
    uint32_t best = 0;
#pragma unroll
    for (int i = 0; i < 16; ++i) {
        const int bb = q * 16 + i;
        if (bb <= kMaxBase) {
            const uint32_t top = hist[bb + 14];
            const uint32_t below = bb > 0 ? hist[bb - 1] : 0u;
            const uint32_t key = ((top - below) << 8) | uint32_t(bb);
            best = key > best ? key : best;
        }
    }
    best = __reduce_max_sync(hmask, best);
    b_out = best & 0xFFu;
    esc_out = uint32_t(kGroup) - (best >> 8);
    __syncwarp(hmask);  // the histogram is reused by the half's next group
}

// 1. bases and escape counts; one half-warp per (unit, column) slot.
__global__ void __launch_bounds__(256) enc_scan_kernel(const EncArgs a) {
    __shared__ uint32_t hist[16][256];
    const int lane = threadIdx.x & 31, q = lane & 15, half = threadIdx.x >> 4;
    const unsigned hmask = half_mask(lane);
    const int64_t slots = a.U * kTileCols;
    for (int64_t sl = int64_t(blockIdx.x) * 16 + half; sl < slots; sl += int64_t(gridDim.x) * 16) {
        const int64_t u = sl / kTileCols, c = sl % kTileCols;
        const int64_t n = (u / a.KG) * kTileCols + c, kg = u % a.KG;
        uint32_t b = 0, e = 0;
        if (n < a.N) {  // uniform across the half
            uint16_t v[8];
            load8(a, n, kg, q, v);
            group_base_half(v, q, hmask, hist[half], b, e);
        }
        if (q == 0) {
            a.base[sl] = uint8_t(b);
            a.count[sl] = e;
        }
    }
}

// 2a. exclusive scan of count[] inside blocks of kScanBlock; block totals out.
__global__ void __launch_bounds__(kScanBlock) enc_scan_blocks(uint32_t *count, int64_t n, uint32_t *block_sum) {
    __shared__ uint32_t warp_tot[kScanBlock / 32];
    const int64_t i = int64_t(blockIdx.x) * kScanBlock + threadIdx.x;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const uint32_t v = i < n ? count[i] : 0u;
    uint32_t x = v;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
        const uint32_t o = __shfl_up_sync(0xFFFFFFFFu, x, off);
        if (lane >= off) x += o;
    }
    if (lane == 31) warp_tot[warp] = x;
    __syncthreads();
    if (warp == 0) {
        uint32_t t = warp_tot[lane];
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
            const uint32_t o = __shfl_up_sync(0xFFFFFFFFu, t, off);
            if (lane >= off) t += o;
        }
        warp_tot[lane] = t;  // inclusive
    }
    __syncthreads();
    const uint32_t before = warp > 0 ? warp_tot[warp - 1] : 0u;
    if (i < n) count[i] = before + x - v;  // exclusive within the block
    if (threadIdx.x == kScanBlock - 1) block_sum[blockIdx.x] = warp_tot[kScanBlock / 32 - 1];
}

// 2b. exclusive scan of the block totals (one block, looping); the grand
// total lands in block_sum[nb].
__global__ void __launch_bounds__(kScanBlock) enc_scan_totals(uint32_t *block_sum, int64_t nb) {
    __shared__ uint32_t warp_tot[kScanBlock / 32];
    __shared__ uint32_t carry;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    if (threadIdx.x == 0) carry = 0u;
    __syncthreads();
    for (int64_t base = 0; base < nb; base += kScanBlock) {
        const int64_t i = base + threadIdx.x;
        const uint32_t v = i < nb ? block_sum[i] : 0u;
        uint32_t x = v;
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
            const uint32_t o = __shfl_up_sync(0xFFFFFFFFu, x, off);
            if (lane >= off) x += o;
        }
        if (lane == 31) warp_tot[warp] = x;
        __syncthreads();
        if (warp == 0) {
            uint32_t t = warp_tot[lane];
#pragma unroll
            for (int off = 1; off < 32; off <<= 1) {
                const uint32_t o = __shfl_up_sync(0xFFFFFFFFu, t, off);
                if (lane >= off) t += o;
            }
            warp_tot[lane] = t;
        }
        __syncthreads();
        const uint32_t before = (warp > 0 ? warp_tot[warp - 1] : 0u) + carry;
        if (i < nb) block_sum[i] = before + x - v;
        __syncthreads();
        if (threadIdx.x == 0) carry += warp_tot[kScanBlock / 32 - 1];
        __syncthreads();
    }
    if (threadIdx.x == 0) block_sum[nb] = carry;
}

// 2c. add the scanned block totals back.
__global__ void __launch_bounds__(kScanBlock) enc_scan_add(uint32_t *count, int64_t n, const uint32_t *block_sum) {
    const int64_t i = int64_t(blockIdx.x) * kScanBlock + threadIdx.x;
    if (i < n) count[i] += block_sum[blockIdx.x];
}

// 3. pack; one half-warp per (unit, column) slot, lane q one word of each
// plane (pos 8q .. 8q+7).
__global__ void __launch_bounds__(256) enc_pack_kernel(const EncArgs a) {
    constexpr int kPermH[8] = {4, 0, 5, 1, 6, 2, 7, 3};
    constexpr int kPermL[8] = {0, 5, 1, 6, 2, 7, 3, 4};
    constexpr int kPermE[8] = {0, 4, 1, 5, 2, 6, 3, 7};
    const int lane = threadIdx.x & 31, q = lane & 15, half = threadIdx.x >> 4;
    const unsigned hmask = half_mask(lane);
    const int64_t slots = a.U * kTileCols;
    uint16_t *esc = reinterpret_cast<uint16_t *>(a.blob + a.off_esc);
    for (int64_t sl = int64_t(blockIdx.x) * 16 + half; sl < slots; sl += int64_t(gridDim.x) * 16) {
        const int64_t u = sl / kTileCols;
        const int c = int(sl % kTileCols);
        const int64_t n = (u / a.KG) * kTileCols + c, kg = u % a.KG;
        const bool live = n < a.N;  // uniform across the half
        uint8_t *ub = a.blob + u * kUnitBytes;
        const uint32_t b = a.base[sl], begin = a.count[sl];
        if (q == 0) {
            *reinterpret_cast<uint32_t *>(ub + kMetaAt + 4 * c) = b | (begin << 8);
            if (c == kTileCols - 1) {
                const uint64_t next = u + 1 < a.U ? a.count[(u + 1) * kTileCols] : a.n_esc;
                uint32_t *tail = reinterpret_cast<uint32_t *>(ub + kMetaAt + 4 * kTileCols);
                tail[0] = uint32_t(next << 8);
                tail[1] = tail[2] = tail[3] = 0u;  // the unit block's last 12 bytes
            }
        }
        const uint32_t off = uint32_t(c * 64 + (((q >> 2) ^ ((c >> 1) & 3)) << 4) + (q & 3) * 4);
        uint32_t hw = 0, lw = 0, ew = 0, flags = 0;
        uint16_t v[8];
        if (live) {
            load8(a, n, kg, q, v);
#pragma unroll
            for (int s = 0; s < 8; ++s) {
                const int jh = kPermH[s], jl = kPermL[s], je = kPermE[s];
                const uint32_t smh = (uint32_t(v[jh] & 0x7Fu) << 1) | (uint32_t(v[jh ^ 1]) >> 15);
                const uint32_t sml = (uint32_t(v[jl] & 0x7Fu) << 1) | (uint32_t(v[jl ^ 1]) >> 15);
                const uint32_t ee = (v[je] >> 7) & 0xFFu;
                const bool in = ee >= b && ee <= b + 14;
                hw |= (smh >> 4) << (4 * s);
                lw |= (sml & 0xFu) << (4 * s);
                ew |= (in ? ee - b : 15u) << (4 * s);
            }
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                const uint32_t e = (v[i] >> 7) & 0xFFu;
                if (!(e >= b && e <= b + 14)) flags |= 1u << i;
            }
        }
        // every plane byte of the unit is written (zeros for padding columns)
        *reinterpret_cast<uint32_t *>(ub + off) = hw;
        *reinterpret_cast<uint32_t *>(ub + kPlaneBlock + off) = lw;
        *reinterpret_cast<uint32_t *>(ub + 2 * kPlaneBlock + off) = ew;
        // escape entries in pos order: rank = escapes of earlier lanes + earlier bits
        if (__any_sync(hmask, flags != 0u)) {
            const uint32_t cnt = __popc(flags);
            uint32_t before = cnt;
#pragma unroll
            for (int o = 1; o < 16; o <<= 1) {
                const uint32_t t = __shfl_up_sync(hmask, before, o, 16);
                if (q >= o) before += t;
            }
            before -= cnt;
            uint32_t at = begin + before;
            for (int i = 0; i < 8; ++i) {
                if (flags & (1u << i)) {
                    const uint32_t pos = uint32_t(8 * q + i), e = (v[i] >> 7) & 0xFFu;
                    if (at < a.n_esc) esc[at] = uint16_t(pos | (e << 7));
                    ++at;
                }
            }
        }
    }
}

// Launched in plain stream order after the pack kernel.  The next launch
// on the stream may be a GEMM with programmatic dependent launch, whose
// producers start copying the blob before they wait for the kernel before
// them; with this one in between, the blob is complete and visible first.
__global__ void enc_done_kernel() {}

// One wave of grid-stride blocks of 256 threads (16 slots per pass).
template <class F>
int grid_for(F kernel, int64_t slots) {
    int sms = 0, per = 0;
    if (device_sm_count(&sms) != W12_OK) return -1;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per, kernel, 256, 0) != cudaSuccess || per < 1) return -1;
    const int64_t g = (slots + 15) / 16;
    const int64_t cap = int64_t(sms) * per;
    return int(g < cap ? (g > 0 ? g : 1) : cap);
}

}  // namespace

size_t encode_device_ws(int64_t K, int64_t N) {
    const int64_t U = ((N + kTileCols - 1) / kTileCols) * (K / kGroup);
    const int64_t slots = U * kTileCols;
    const int64_t nb = (slots + kScanBlock - 1) / kScanBlock;
    return kWsHeader + round256(uint64_t(slots)) + round256(uint64_t(slots) * 4u) + round256(uint64_t(nb + 1) * 4u);
}

// Steps 1-2 into the workspace; *total_dev receives the escape count.
int launch_encode_scan(const uint16_t *w, int64_t K, int64_t N, int layout, void *ws, void *stream,
                       uint32_t **total_dev) {
    EncArgs a{};
    a.w = w;
    a.K = K;
    a.N = N;
    a.KG = K / kGroup;
    a.layout = layout;
    a.U = ((N + kTileCols - 1) / kTileCols) * a.KG;
    const int64_t slots = a.U * kTileCols;
    const int64_t nb = (slots + kScanBlock - 1) / kScanBlock;
    uint8_t *p = static_cast<uint8_t *>(ws) + kWsHeader;
    a.base = p;
    a.count = reinterpret_cast<uint32_t *>(p + round256(uint64_t(slots)));
    a.block_sum = reinterpret_cast<uint32_t *>(p + round256(uint64_t(slots)) + round256(uint64_t(slots) * 4u));
    *total_dev = a.block_sum + nb;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    const int grid = grid_for(enc_scan_kernel, slots);
    if (grid < 0) return W12_ERR_CUDA;
    enc_scan_kernel<<<unsigned(grid), 256, 0, s>>>(a);
    enc_scan_blocks<<<unsigned(nb), kScanBlock, 0, s>>>(a.count, slots, a.block_sum);
    enc_scan_totals<<<1, kScanBlock, 0, s>>>(a.block_sum, nb);
    enc_scan_add<<<unsigned(nb), kScanBlock, 0, s>>>(a.count, slots, a.block_sum);
    return cudaGetLastError() == cudaSuccess ? W12_OK : W12_ERR_CUDA;
}

// Step 3 (after launch_encode_scan on the same workspace).
int launch_encode_pack(const uint16_t *w, const w12_desc *d, int layout, void *blob, void *ws, void *stream) {
    EncArgs a{};
    a.w = w;
    a.K = d->K;
    a.N = d->N;
    a.KG = d->K / kGroup;
    a.layout = layout;
    a.U = int64_t(d->n_units);
    const int64_t slots = a.U * kTileCols;
    uint8_t *p = static_cast<uint8_t *>(ws) + kWsHeader;
    a.base = p;
    a.count = reinterpret_cast<uint32_t *>(p + round256(uint64_t(slots)));
    a.blob = static_cast<uint8_t *>(blob);
    a.off_esc = d->off_esc;
    a.n_esc = d->n_esc;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    // every byte of the unit blocks is written by the kernel; zero the rest:
    // the gap before the escape list and the tail after it
    uint8_t *bl = static_cast<uint8_t *>(blob);
    const uint64_t units_end = d->n_units * uint64_t(kUnitBytes), esc_end = d->off_esc + 2u * d->n_esc;
    if (d->off_esc > units_end && cudaMemsetAsync(bl + units_end, 0, d->off_esc - units_end, s) != cudaSuccess)
        return W12_ERR_CUDA;
    if (d->total_bytes > esc_end && cudaMemsetAsync(bl + esc_end, 0, d->total_bytes - esc_end, s) != cudaSuccess)
        return W12_ERR_CUDA;
    const int grid = grid_for(enc_pack_kernel, slots);
    if (grid < 0) return W12_ERR_CUDA;
    enc_pack_kernel<<<unsigned(grid), 256, 0, s>>>(a);
    enc_done_kernel<<<1, 32, 0, s>>>();
    return cudaGetLastError() == cudaSuccess ? W12_OK : W12_ERR_CUDA;
}

}  // namespace w12
