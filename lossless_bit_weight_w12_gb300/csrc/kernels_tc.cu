// kernels_tc.cu -- W12 decode-GEMM on the 5th-generation tensor cores
// (tcgen05) for token counts where the product is a real dense contraction
// (16 < M <= 128): the weights are rebuilt into tensor memory as the A
// operand, the fp32 accumulator lives in tensor memory, and the tokens come
// from shared memory.
//
// Work split as in the mma.sync stream kernel (stream_device.cuh): units
// of one 128-k group of a 128-column tile, stream-K over the whole batch.
// Two rings feed a unit: the unit block (planes and meta words) lands in a
// weight stage, and the unit's tokens -- two boxes of 64 k x MP tokens with
// the 128-byte swizzle, the canonical K-major layout of the UMMA B operand
// -- in a token slot.  A weight stage is free again once the decoders have
// read it, a token slot only once the UMMAs that read it have completed, so
// the two rings turn over at different rates; each has its own producer
// warp.  Unit i of a CTA uses weight stage i % SW and token slot i % SX.
//
// Roles (one CTA per SM, 20 warps):
//  - 16 decoder warps in two groups that take alternate units, so two
//    units are decoded at once.  Thread (w, l) of a group owns tile row
//    r = 32 (w % 4) + l (tensor-memory lane r) and half h = (w % 8) / 4 of
//    the group's 128 k.  Per unit it rebuilds its 64 weights in registers
//    ("reconstructing bit by bit in GEMM registers", SpecPilot summary,
//    airadar.tv English edition, "Reasons" bullet 2), stores them with
//    tcgen05.st into the A buffer of the unit's token slot (64 columns,
//    column j holding the bf16 pair k = 2j, 2j + 1) and patches the
//    escaped ones there, one column per escaping lane, warp-wide.  At the
//    end of a tile piece all 16 warps read the accumulator back (tcgen05.ld;
//    warp w takes a quarter w / 4 of the tokens) and write y or the
//    stream-K partial slot, then run the fix-up.
//  - 1 weight producer warp: one bulk copy per unit block into the weight
//    ring, and the L1 prefetch of each tile piece's escape entries.
//  - 1 token producer warp: the two x boxes of each unit into the token ring.
//  - 2 MMA warps, one per unit parity (the first also allocates and frees
//    the tensor memory): the first thread of each issues the 8 UMMAs of its
//    units (M = 128 columns, N = MP tokens, K = 16: D_t += A_tmem . B_smem)
//    into its own accumulator D_t once A is in place (the decoders signal
//    that only after they saw the unit's tokens land), and commits them to
//    the token slot's empty barrier and, after a piece's last unit, to the
//    accumulators' barrier.  The epilogue adds D_0 and D_1.
// Shared memory: the token ring (1024-byte aligned), the weight ring, then
// the barriers.  Tensor memory: the accumulators at columns 0 and MP, then
// one A buffer of 64 columns per token slot; 512 columns allocated.  The slot's commit
// releases both; decoders that see the slot full again know that the UMMAs
// which read its A buffer last have completed (the producer refilled the
// slot only after that commit).  A K = 16 UMMA of M = 128 takes 45 cycles
// at N <= 32 and 64 at N = 128 (measured), but on its issuing thread every
// mbarrier wait costs ~200 cycles and every commit ~45 while UMMAs are in
// flight; with two issuers one's wait overlaps the other's UMMAs, and the
// tensor core runs at the bare UMMA rate (measured: 44 cycles per UMMA
// with a wait and a commit per 8, against 78 with one issuer).
// Every mbarrier wait is bounded; after a timeout every role runs to its
// end without waiting and the error word says W12_ERR_TIMEOUT.  The
// producers stop issuing once the CTA has aborted and let their copies in
// flight land, and each MMA thread waits (bounded) for its own UMMAs before
// the tensor memory is freed.
#include <cuda.h>
#include <cuda_runtime.h>

#include "stream_device.cuh"
#include "verify_common.cuh"

namespace w12 {

namespace {

constexpr int kDW = 16;                  // decoder warps
constexpr int kDT = kDW * 32;
constexpr int kWProdWarp = kDW;          // weight producer
constexpr int kXProdWarp = kDW + 1;      // token producer
constexpr int kMmaWarp = kDW + 2;        // tensor-memory owner, UMMA issuer of the even units
constexpr int kMmaWarp1 = kDW + 3;       // UMMA issuer of the odd units
constexpr int kTT = (kDW + 4) * 32;      // 640 threads
constexpr uint32_t kTmemCols = 512;

template <int MP, bool FUSED = false>
struct TCfg {
    static constexpr int kX = MP * 256;                        // token slot: two boxes of MP rows x 128 bytes
    // token slots (and A buffers): 4, but 3 for the fused lm_head at MP = 128
    // (its per-token keys leave no room for a fourth 32 KB slot)
    static constexpr int SX = MP >= 128 ? (FUSED ? 3 : 4) : 4;
    static constexpr int kXRing = SX * kX;                     // at the (1024-aligned) start of the ring
    static constexpr int kW = kUnitBytes;                      // weight stage stride (16-byte aligned)
    // The barriers and scalars live after the rings, so the kernel has no
    // static shared memory and its dynamic region starts at the CTA's
    // shared base (1024-byte aligned: no alignment slack is reserved; the
    // kernel checks it): (3 SW + 5 SX + 3) mbarriers, the tensor-memory
    // address, the wait state, s_last, s_best.  kBarMax sizes them for the
    // deepest weight ring (8 stages) to choose SW.
    static constexpr int kBarMax = (3 * 8 + 5 * SX + 3) * 8 + 64 + (FUSED ? MP * 8 : 8);
    static constexpr int kFit = (227 * 1024 - kBarMax - kXRing) / kW;
    static constexpr int SW = kFit > 8 ? 8 : kFit;             // weight stages, after the token ring
    static constexpr int kBarOff = kXRing + SW * kW;
    static constexpr int kBar = (3 * SW + 5 * SX + 3) * 8 + 64 + (FUSED ? MP * 8 : 8);
    static constexpr size_t kDynSmem = size_t(kBarOff) + size_t(kBar);
    static_assert(kDynSmem <= 227 * 1024, "shared memory");
    // tensor-memory columns: accumulators [0, MP) and [MP, 2 MP), A buffer of
    // slot s at kA + 64 s
    static constexpr uint32_t kA = 2 * MP < 64 ? 64u : uint32_t(2 * MP);
    static_assert(kA + 64u * SX <= kTmemCols, "A buffers exceed the tensor memory");
    static_assert(SW >= 2, "weight ring too shallow");
};

// UMMA shared-memory descriptor of a K-major operand with the 128-byte
// swizzle: 8-row core groups 1024 bytes apart.
__device__ __forceinline__ uint64_t desc_sw128(uint32_t addr) {
    uint64_t d = 0;
    d |= uint64_t((addr & 0x3FFFFu) >> 4);  // start address
    d |= uint64_t(16u >> 4) << 16;          // leading byte offset (unused with this swizzle)
    d |= uint64_t(1024u >> 4) << 32;        // stride byte offset: 8 rows x 128 B
    d |= uint64_t(1) << 46;                 // descriptor version
    d |= uint64_t(2) << 61;                 // 128-byte swizzle
    return d;
}

// Instruction descriptor: D fp32, A and B bf16, K-major, N = MP, M = 128.
template <int MP>
__device__ __forceinline__ uint32_t idesc_bf16() {
    return (1u << 4) | (1u << 7) | (1u << 10) | (uint32_t(MP >> 3) << 17) | (uint32_t(128 >> 4) << 24);
}

// D[tmem_d] (+)= A[tmem_a] . B[desc]; A read from tensor memory.
__device__ __forceinline__ void umma_ts(uint32_t tmem_d, uint32_t tmem_a, uint64_t bdesc, uint32_t idesc,
                                        uint32_t accumulate) {
    asm volatile(
        "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
        " tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n}\n" ::"r"(tmem_d),
        "r"(tmem_a), "l"(bdesc), "r"(idesc), "r"(accumulate)
        : "memory");
}

__device__ __forceinline__ void umma_commit(uint64_t *bar) {
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
                     smem_addr(bar))
                 : "memory");
}

__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

// Store 32 consecutive 32-bit columns of this thread's lane (the caller
// waits: tcgen05.wait::st).
__device__ __forceinline__ void tmem_st32(uint32_t taddr, const uint32_t (&v)[32]) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,"
        "%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};" ::"r"(taddr),
        "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7]), "r"(v[8]),
        "r"(v[9]), "r"(v[10]), "r"(v[11]), "r"(v[12]), "r"(v[13]), "r"(v[14]), "r"(v[15]), "r"(v[16]),
        "r"(v[17]), "r"(v[18]), "r"(v[19]), "r"(v[20]), "r"(v[21]), "r"(v[22]), "r"(v[23]), "r"(v[24]),
        "r"(v[25]), "r"(v[26]), "r"(v[27]), "r"(v[28]), "r"(v[29]), "r"(v[30]), "r"(v[31])
        : "memory");
}

// One 32-bit column of this thread's lane: load (tmem_ld_wait() before the
// register is used) and store (tcgen05.wait::st before a later load).
__device__ __forceinline__ uint32_t tmem_ld1(uint32_t taddr) {
    uint32_t r;
    asm volatile("tcgen05.ld.sync.aligned.32x32b.x1.b32 {%0}, [%1];" : "=r"(r) : "r"(taddr));
    return r;
}

__device__ __forceinline__ void tmem_st1(uint32_t taddr, uint32_t v) {
    asm volatile("tcgen05.st.sync.aligned.32x32b.x1.b32 [%0], {%1};" ::"r"(taddr), "r"(v) : "memory");
}

__device__ __forceinline__ void tmem_st_wait() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }

// Load 4 consecutive 32-bit columns of this thread's lane (tmem_ld_wait()
// before the registers are used).
__device__ __forceinline__ void tmem_ld4(uint32_t taddr, uint32_t (&r)[4]) {
    asm volatile("tcgen05.ld.sync.aligned.32x32b.x4.b32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
                 : "r"(taddr));
}

__device__ __forceinline__ void tmem_ld_wait() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }

// The first escape entry of each lane's column, when it falls in the lane's
// 64 weights (already stored, word i at column ta + i: the weights at
// k = pos0 + 2i, pos0 + 2i + 1), patched in tensor memory: the lanes that
// have one are taken in turn, warp-wide; each turn loads the column that
// holds the escaped weight (the same column in every lane), replaces the
// weight's exponent in the owner lane and stores the column back.  Tensor
// memory does the indexing, so no register select over the 32 words.
__device__ __forceinline__ void patch_first_escapes_tmem(const EscPending &ep, uint32_t ta, uint32_t pos0,
                                                         int lane) {
    const uint32_t j = (ep.e0 & 0x7Fu) - pos0;
    uint32_t todo = __ballot_sync(0xFFFFFFFFu, ep.lo != ep.hi && j < 64u);
    tmem_st_wait();  // the tile's words are in place before any column is read back
    if (!todo) return;
    const uint32_t sh = (j & 1u) * 16u;
    const uint32_t keep = ~(0x7F80u << sh), put = (ep.e0 & 0x7F80u) << sh;
    do {
        const int src = __ffs(todo) - 1;
        todo &= todo - 1u;
        const uint32_t q = __shfl_sync(0xFFFFFFFFu, j >> 1, src);
        uint32_t x = tmem_ld1(ta + q);
        tmem_ld_wait();
        if (lane == src) x = (x & keep) | put;
        tmem_st1(ta + q, x);
        tmem_st_wait();  // a later turn may read the same column
    } while (todo);
}

// Both rings signal a landed fill on a barrier of the decoder group that
// owns the unit (full[2 s + (i & 1)] for unit i in slot s = i % S), so each
// group waits on its own barriers only and sees their phases one by one.
// The parity of unit i's fill on that barrier: the group's fills of slot s
// are every fill of it (S even) or every other one (S odd).  A barrier
// cannot run two phases ahead of its group: the fill after unit i's on the
// same barrier needs the group's own release of unit i first.
template <int S>
__device__ __forceinline__ uint32_t group_parity(int i) {
    const int k = i / S;
    return uint32_t((S & 1) ? (k >> 1) : k) & 1u;
}

// Weight producer (lane 0 of its warp): unit i of the CTA into weight stage
// i % SW, once the decoders have released the stage's previous unit.  It
// reads the blob only after the previous kernel of the stream completed,
// unless the launch asked for the early weight stream (b.early_weights: the
// blob is not written by that kernel).  The test hook b.withhold_unit
// leaves one unit's stage unarmed, so its decoders' bounded wait runs out.
template <int SW>
__device__ __forceinline__ void tc_weight_producer(const StreamBatch &b, uint32_t wbase, uint32_t stride,
                                                   uint64_t *full_w, uint64_t *empty_w, WaitCtl *ctl, int u0,
                                                   int u1) {
    if (!b.early_weights) pdl_wait();
    const uint64_t pol = l2_evict_first_policy();
    SCur c = s_at(b, u0);
    int issued = 0;
    for (int u = u0; u < u1; ++u) {
        const int i = u - u0, s = i % SW;
        // (a decoder that gave up sets the abort flag before it arrives
        // without waiting: stop, so the drain below covers every copy in flight)
        if (i >= SW && (!mbar_wait(&empty_w[s], uint32_t(i / SW - 1) & 1u, ctl, b.err) || aborted(ctl))) break;
        const StreamOne &g = b.g[c.gi];
        const uint8_t *unit = unit_block(g, c);
        if (u != b.withhold_unit) {
            if (u == u0 || c.kg == 0) prefetch_piece_escapes(g, c, unit, u, u1);
            uint64_t *bar = &full_w[2 * s + (i & 1)];
            mbar_expect_tx(bar, uint32_t(kUnitBytes));
            bulk_copy(wbase + uint32_t(s) * stride, unit, uint32_t(kUnitBytes), bar, pol);
        }
        s_next(b, c);
        ++issued;
    }
    if (aborted(ctl))  // let the copies in flight land
        for (int j = issued - 1; j >= 0 && j >= issued - SW; --j)
            mbar_drain(&full_w[2 * (j % SW) + (j & 1)], group_parity<SW>(j), ctl->limit_ns);
}

// Token producer (lane 0 of its warp): the two 64-k boxes of unit i's tokens
// into token slot i % SX, once the UMMAs that read the slot's previous unit
// have completed.  x may be written by the previous kernel of the stream.
template <int SX>
__device__ __forceinline__ void tc_x_producer(const StreamBatch &b, uint32_t xbase, int mp, uint64_t *full_x,
                                              uint64_t *empty_x, WaitCtl *ctl, int u0, int u1) {
    pdl_wait();
    const uint32_t kx = uint32_t(mp) * 256u;
    SCur c = s_at(b, u0);
    int issued = 0;
    for (int u = u0; u < u1; ++u) {
        const int i = u - u0, s = i % SX;
        if (i >= SX && (!mbar_wait(&empty_x[s], uint32_t(i / SX - 1) & 1u, ctl, b.err) || aborted(ctl))) break;
        const StreamOne &g = b.g[c.gi];
        const uint32_t dst = xbase + uint32_t(s) * kx;
        uint64_t *bar = &full_x[2 * s + (i & 1)];
        mbar_expect_tx(bar, kx);
        tma_2d_keep(dst, &g.tx, 128 * c.kg, 0, bar);
        tma_2d_keep(dst + uint32_t(mp) * 128u, &g.tx, 128 * c.kg + 64, 0, bar);
        s_next(b, c);
        ++issued;
    }
    if (aborted(ctl))
        for (int j = issued - 1; j >= 0 && j >= issued - SX; --j)
            mbar_drain(&full_x[2 * (j % SX) + (j & 1)], group_parity<SX>(j), ctl->limit_ns);
}

// FUSED: the lm_head + greedy verify epilogue (as in kernels_stream.cu):
// tile outputs fold into a per-CTA running (value, lowest index) maximum
// per token, split tiles are folded by the CTA that completes them, and the
// last CTA to arrive runs the acceptance rule over every CTA's keys.
template <int MP, bool FUSED>
__global__ void __launch_bounds__(kTT, 1) tc_kernel(const __grid_constant__ StreamBatch b) {
    using C = TCfg<MP, FUSED>;
    constexpr int SW = C::SW, SX = C::SX;
    extern __shared__ __align__(1024) unsigned char smem_dyn[];
    // the token ring needs a 1024-byte aligned start (128-byte swizzle of the
    // boxes and the UMMA descriptors); a misaligned region is reported, not used
    if (smem_addr(smem_dyn) & 1023u) {
        if (threadIdx.x == 0) record_error(b.err, W12_ERR_DEVICE);
        return;
    }
    unsigned char *bar_block = smem_dyn + C::kBarOff;
    uint64_t *full_w = reinterpret_cast<uint64_t *>(bar_block);
    uint64_t *empty_w = full_w + 2 * SW;
    uint64_t *full_x = empty_w + SW;
    uint64_t *empty_x = full_x + 2 * SX;
    uint64_t *a_full = empty_x + SX;
    uint64_t &acc_full = a_full[2 * SX];
    uint64_t &acc_empty = a_full[2 * SX + 1];
    uint64_t &fin = a_full[2 * SX + 2];
    uint32_t &s_tmem = *reinterpret_cast<uint32_t *>(a_full + 2 * SX + 3);
    WaitCtl &s_ctl = *reinterpret_cast<WaitCtl *>(a_full + 2 * SX + 4);
    int &s_last = *reinterpret_cast<int *>(a_full + 2 * SX + 6);
    unsigned long long *s_best = reinterpret_cast<unsigned long long *>(a_full + 2 * SX + 8);
    const uint32_t xbase = smem_addr(smem_dyn);  // token ring, then the weight ring
    const uint32_t wbase = xbase + uint32_t(C::kXRing);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    int u0, u1;
    {
        const int G = int(gridDim.x), c = int(blockIdx.x);
        const int per = b.U / G, rem = b.U % G;
        u0 = sk_unit_begin(c, per, rem);
        u1 = u0 + per + (c < rem ? 1 : 0);
    }
    if (threadIdx.x == 0) {
        for (int s = 0; s < 2 * SW; ++s) mbar_init(&full_w[s], 1);  // the producer's expect_tx arrival (+ bytes)
        for (int s = 0; s < 2 * SX; ++s) mbar_init(&full_x[s], 1);
        for (int s = 0; s < SW; ++s) mbar_init(&empty_w[s], kDW / 2);  // the decoder group of the unit
        for (int s = 0; s < SX; ++s) mbar_init(&empty_x[s], 1);         // the unit's UMMA commit
        for (int s = 0; s < 2 * SX; ++s) mbar_init(&a_full[s], kDW / 2);  // per decoder group, as full_x
        mbar_init(&acc_full, 2);  // both issuers' commits after a piece's last unit
        mbar_init(&acc_empty, kDW);
        mbar_init(&fin, 2);
        wait_ctl_init(&s_ctl, b);
        mbar_fence_init();
    }
    if (FUSED)
        for (int m = threadIdx.x; m < MP; m += kTT) s_best[m] = 0ull;
    if (warp == kMmaWarp) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_addr(&s_tmem)),
                     "r"(kTmemCols)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = s_tmem;
    if (threadIdx.x == 0) pdl_launch();

    if (warp == kWProdWarp) {
        if (lane == 0 && u0 < u1) tc_weight_producer<SW>(b, wbase, C::kW, full_w, empty_w, &s_ctl, u0, u1);
        return;
    }
    if (warp == kXProdWarp) {
        if (lane == 0 && u0 < u1) tc_x_producer<SX>(b, xbase, MP, full_x, empty_x, &s_ctl, u0, u1);
        return;
    }
    pdl_wait();  // nothing below touches global memory the previous kernel may write before this

    if (warp == kMmaWarp || warp == kMmaWarp1) {
        // ----------------------------------------------------------- UMMA issuers
        const int t = warp - kMmaWarp;  // units of parity t, accumulator t
        if (lane == 0) {
            const uint32_t idesc = idesc_bf16<MP>();
            const uint32_t dt = tmem + uint32_t(t * MP);
            SCur c = s_at(b, u0);
            int i = 0, piece = 0;
            for (int u = u0; u < u1;) {
                const StreamOne &g = b.g[c.gi];
                const int first = g.ubase + c.nb * g.KG;
                const int ub = min(u1, first + g.KG);
                // the epilogue of the previous piece has read the accumulators
                if (piece > 0) mbar_wait(&acc_empty, uint32_t(piece - 1) & 1u, &s_ctl, b.err);
                tc_fence_after();
                bool fresh = true;  // this issuer's next UMMA starts its sum of the piece
                const int iend = i + (ub - u);
                for (int iu = i + ((i & 1) != t); iu < iend; iu += 2) {  // this issuer's units
                    const int sx = iu % SX;
                    // The decoders that signal a_full waited for this
                    // slot's full barrier first (tokens landed), so the
                    // UMMAs may read it once a_full is observed.
                    mbar_wait(&a_full[2 * sx + t], group_parity<SX>(iu), &s_ctl, b.err);
                    tc_fence_after();
                    const uint64_t d0 = desc_sw128(xbase + uint32_t(sx) * uint32_t(C::kX));
                    const uint32_t ta = tmem + C::kA + 64u * uint32_t(sx);
#pragma unroll
                    for (int ks = 0; ks < 8; ++ks) {
                        // x box ks / 4 (k half), 16 k = 32 bytes per step inside the swizzle atom
                        const uint64_t dx = d0 + uint64_t(((ks >> 2) * MP * 128 + 32 * (ks & 3)) >> 4);
                        umma_ts(dt, ta + 8u * uint32_t(ks), dx, idesc, (fresh && ks == 0) ? 0u : 1u);
                    }
                    fresh = false;
                    umma_commit(&empty_x[sx]);  // frees the token slot and its A buffer
                }
                umma_commit(&acc_full);
                u = ub;
                i = iend;
                ++piece;
                s_next_tile(b, c);
            }
            // every UMMA issued has completed before the memory is freed
            umma_commit(&fin);
            mbar_drain(&fin, 0u, s_ctl.limit_ns);
            if (piece > 0) mbar_wait(&acc_empty, uint32_t(piece - 1) & 1u, &s_ctl, b.err);
        }
        __syncwarp();
        if (warp == kMmaWarp) {
            tc_fence_after();
            asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(kTmemCols)
                         : "memory");
        }
        return;
    }

    // ---------------------------------------------------------------- decoders
    const int r = 32 * (warp & 3) + lane;  // tile row = tensor-memory lane
    const int grp = warp >> 3;             // units of this parity
    const int h = (warp & 7) >> 2;         // k half of the group
    const int qt = warp >> 2;              // token quarter of the epilogue
    const uint32_t lane_off = uint32_t(32 * (warp & 3)) << 16;
    // plane row r, logical 16-byte chunks 2h and 2h + 1 (the format stores
    // chunk j of row r at j ^ ((r >> 1) & 3): a warp's 32 rows read 8
    // different bank groups per quarter-warp)
    const uint32_t sw = uint32_t((r >> 1) & 3);
    const uint32_t p0 = uint32_t(r * 64) + ((uint32_t(2 * h) ^ sw) << 4);
    const uint32_t p1 = uint32_t(r * 64) + ((uint32_t(2 * h + 1) ^ sw) << 4);
    const int M = b.M;
    SCur c = s_at(b, u0);
    int i = 0, piece = 0;
    for (int u = u0; u < u1;) {
        const StreamOne &g = b.g[c.gi];
        const int nb = c.nb, first = g.ubase + nb * g.KG;
        const int ua = u, ub = min(u1, first + g.KG);
        const int n = nb * kTileN + r;
        const bool valid = n < g.N;
        const int iend = i + (ub - u);
        for (int iu = i + ((i & 1) != grp); iu < iend; iu += 2) {  // this group's units of the piece
            const int s = iu % SW, sx = iu % SX;
            mbar_wait(&full_w[2 * s + grp], group_parity<SW>(iu), &s_ctl, b.err);
            const uint32_t st = wbase + uint32_t(s) * uint32_t(C::kW);
            const uint4 h0 = lds128(st + p0), h1 = lds128(st + p1);
            const uint4 l0 = lds128(st + kPlaneBlock + p0), l1 = lds128(st + kPlaneBlock + p1);
            const uint4 e0 = lds128(st + 2 * kPlaneBlock + p0), e1 = lds128(st + 2 * kPlaneBlock + p1);
            const uint2 mw = make_uint2(lds32(st + kMetaAt + 4u * uint32_t(r)),
                                        lds32(st + kMetaAt + 4u * uint32_t(r) + 4u));
            // the column's first escape entry (if any) is read while the
            // rebuild runs
            const EscPending ep = esc_begin(valid, mw.x, mw.y, g.esc, g.n_esc, b.err);
            __syncwarp();
            if (lane == 0) mbar_arrive(&empty_w[s]);  // planes and meta read
            uint32_t w[32];
            uint32_t(&wlo)[16] = *reinterpret_cast<uint32_t(*)[16]>(&w[0]);
            uint32_t(&whi)[16] = *reinterpret_cast<uint32_t(*)[16]>(&w[16]);
            const uint32_t b4 = base4(mw.x);
            rebuild32(h0, l0, e0, b4, wlo);
            rebuild32(h1, l1, e1, b4, whi);
            // the unit's tokens have landed, and with them the UMMAs that
            // read this slot's A buffer last have completed; the escape
            // entries are applied after that wait, which gives their loads
            // more time
            mbar_wait(&full_x[2 * sx + grp], group_parity<SX>(iu), &s_ctl, b.err);
            if (__any_sync(0xFFFFFFFFu, ep.hi - ep.lo > 1u)) {  // a column's further entries (rare)
                esc_apply_rest(ep, wlo, uint32_t(64 * h), g.esc);
                esc_apply_rest(ep, whi, uint32_t(64 * h + 32), g.esc);
            }
            tc_fence_after();
            const uint32_t ta = tmem + lane_off + C::kA + 64u * uint32_t(sx) + 32u * uint32_t(h);
            tmem_st32(ta, w);
            patch_first_escapes_tmem(ep, ta, uint32_t(64 * h), lane);
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&a_full[2 * sx + grp]);
        }
        u = ub;
        i = iend;

        // ---- epilogue: accumulator row r, tokens [h MP/4, (h + 1) MP/4):
        // D_0 + D_1, each only if its issuer had a unit in this piece
        mbar_wait(&acc_full, uint32_t(piece) & 1u, &s_ctl, b.err);
        tc_fence_after();
        const int cnt = ub - ua, ia = i - cnt;
        const bool has0 = cnt >= 2 || (ia & 1) == 0, has1 = cnt >= 2 || (ia & 1) == 1;
        constexpr int kHalf = MP / 4;
        float v[kHalf];
        // up to 8 tokens of each accumulator per round trip to tensor memory
        constexpr int kQ = kHalf >= 8 ? 8 : kHalf;
#pragma unroll
        for (int q0 = 0; q0 < kHalf; q0 += kQ) {
            uint32_t r0[kQ] = {}, r1[kQ] = {};
#pragma unroll
            for (int q = 0; q < kQ; q += 4) {
                uint32_t(&a)[4] = *reinterpret_cast<uint32_t(*)[4]>(&r0[q]);
                uint32_t(&bb)[4] = *reinterpret_cast<uint32_t(*)[4]>(&r1[q]);
                if (has0) tmem_ld4(tmem + lane_off + uint32_t(qt * kHalf + q0 + q), a);
                if (has1) tmem_ld4(tmem + lane_off + uint32_t(MP + qt * kHalf + q0 + q), bb);
            }
            tmem_ld_wait();
#pragma unroll
            for (int e = 0; e < kQ; ++e)
                v[q0 + e] = has0 && has1 ? __uint_as_float(r0[e]) + __uint_as_float(r1[e])
                                         : __uint_as_float(has0 ? r0[e] : r1[e]);
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&acc_empty);
        if (ua == first && ub == first + g.KG) {
            if (valid && (!FUSED || g.y)) {
#pragma unroll
                for (int e = 0; e < kHalf; ++e) {
                    const int m = qt * kHalf + e;
                    if (m < M) store_out(g.y, b.y_dtype, g.N, m, n, v[e]);
                }
            }
            if (FUSED) {
                // per token: the warp's 32 rows -> one key, then the CTA maximum
#pragma unroll
                for (int e = 0; e < kHalf; ++e) {
                    unsigned long long best = valid ? pack_key(v[e], uint32_t(n)) : 0ull;
#pragma unroll
                    for (int off = 16; off >= 1; off >>= 1) {
                        const unsigned long long o = __shfl_xor_sync(0xFFFFFFFFu, best, off);
                        best = o > best ? o : best;
                    }
                    const int m = qt * kHalf + e;
                    if (lane == 0 && m < M && best != 0ull) atomicMax(&s_best[m], best);
                }
            }
        } else {
            const int slot = ua == u0 ? 0 : 1;
            float *P = b.partial + (size_t(blockIdx.x) * 2 + slot) * size_t(M) * kTileN;
#pragma unroll
            for (int e = 0; e < kHalf; ++e) {
                const int m = qt * kHalf + e;
                if (m < M) P[m * kTileN + r] = v[e];
            }
            stream_fixup<FUSED>(b, g, first, nb, ub - ua, &s_last, threadIdx.x, kDT, s_best);
        }
        ++piece;
        s_next_tile(b, c);
    }

    if (FUSED) {
        // publish this CTA's per-token best; the last CTA to arrive folds
        // them and runs the acceptance rule
        const int tid = threadIdx.x;
        named_sync(kDT);
        for (int m = tid; m < M; m += kDT) b.row_best[size_t(blockIdx.x) * M + m] = s_best[m];
        __threadfence();
        named_sync(kDT);
        if (tid == 0) s_last = (atomicAdd(b.done, 1u) == gridDim.x - 1);
        named_sync(kDT);
        if (s_last) {
            __threadfence();
            verify_from_keys(b.row_best, int64_t(gridDim.x), M, b.vR, b.vT, b.draft, b.accept_len, b.next_tok,
                             b.gbuf, tid, kDT);
            if (tid == 0) *b.done = 0u;
        }
    }
}

template <int MP, bool FUSED = false>
int launch_tc_t(const StreamBatch &b, int grid, cudaStream_t s) {
    return launch_pdl(tc_kernel<MP, FUSED>, grid, kTT, TCfg<MP, FUSED>::kDynSmem, s, b);
}

template <int MP, bool FUSED = false>
int occ_tc_t(int *blocks) {
    if (cudaFuncSetAttribute(tc_kernel<MP, FUSED>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             int(TCfg<MP, FUSED>::kDynSmem)) != cudaSuccess)
        return W12_ERR_CUDA;
    return cudaOccupancyMaxActiveBlocksPerMultiprocessor(blocks, tc_kernel<MP, FUSED>, kTT, TCfg<MP, FUSED>::kDynSmem) ==
                   cudaSuccess
               ? W12_OK
               : W12_ERR_CUDA;
}

}  // namespace

// variant v: MP = 16 << v tokens (16, 32, 64, 128).  The dynamic
// shared-memory limit is raised by tc_occupancy(), which the planner runs
// once per device and variant before the first launch.
int launch_tc_batch(const StreamBatch &b, int variant, int grid, void *stream) {
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    switch (variant) {
        case 0: return launch_tc_t<16>(b, grid, s);
        case 1: return launch_tc_t<32>(b, grid, s);
        case 2: return launch_tc_t<64>(b, grid, s);
        case 3: return launch_tc_t<128>(b, grid, s);
    }
    return W12_ERR_ARG;
}

// The fused lm_head + verify variants (same v).
int launch_tc_fused(const StreamBatch &b, int variant, int grid, void *stream) {
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    switch (variant) {
        case 0: return launch_tc_t<16, true>(b, grid, s);
        case 1: return launch_tc_t<32, true>(b, grid, s);
        case 2: return launch_tc_t<64, true>(b, grid, s);
        case 3: return launch_tc_t<128, true>(b, grid, s);
    }
    return W12_ERR_ARG;
}

int tc_fused_occupancy(int variant, int *blocks) {
    switch (variant) {
        case 0: return occ_tc_t<16, true>(blocks);
        case 1: return occ_tc_t<32, true>(blocks);
        case 2: return occ_tc_t<64, true>(blocks);
        case 3: return occ_tc_t<128, true>(blocks);
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
