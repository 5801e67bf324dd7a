// kernels_tc.cu -- W12 decode-GEMM on the 5th-generation tensor cores
// (tcgen05) for token counts where the product is a real dense contraction
// (16 < M <= 128): the weights are rebuilt into tensor memory as the A
// operand, the fp32 accumulator lives in tensor memory, and the tokens come
// from shared memory.
//
// Work split: stream-K over units of one 128-k group of a 128-column tile,
// as in the mma.sync stream kernel (stream_device.cuh), but in PAIR order:
// the tiles of a product are taken two at a time (a phantom tile pads an odd
// count), and within a pair the units run (kg, tile 0), (kg, tile 1),
// (kg + 1, tile 0), ...  A "step" is the two units of one k-group of a pair:
// both multiply the same tokens, so one token box (two boxes of 64 k x MP
// tokens with the 128-byte swizzle, the canonical K-major layout of the UMMA
// B operand) serves two units, and the tile of a unit is its parity.  CTA c
// takes a balanced contiguous range of units (it may start or end in the
// middle of a step).
//
// Roles (one CTA per SM, 20 warps):
//  - 16 decoder warps in two groups; group j takes the units of parity j
//    (tile j of each pair), so two units are decoded at once.  Thread (w, l)
//    of a group owns tile row r = 32 (w % 4) + l (tensor-memory lane r) and
//    half h = (w % 8) / 4 of the group's 128 k.  Per unit it rebuilds its 64
//    weights in registers ("reconstructing bit by bit in GEMM registers",
//    SpecPilot summary, airadar.tv English edition, "Reasons" bullet 2),
//    patches escapes, and stores them with tcgen05.st into one of the
//    group's A buffers (64 columns, column c holding the bf16 pair k = 2c,
//    2c + 1).  At the end of a tile piece the group reads its accumulator
//    back (tcgen05.ld; warp w takes half (w % 8) / 4 of the tokens) and
//    writes y or the stream-K partial slot, then runs the fix-up.
//  - 1 weight producer warp: one bulk copy per unit block into the group's
//    weight ring, and the L1 prefetch of each tile piece's escape entries.
//  - 1 token producer warp: one token box per step into the token ring.
//  - 2 MMA warps, issuer j for the units of parity j (the first also
//    allocates and frees the tensor memory): the first thread of each
//    issues the 8 UMMAs of a unit (M = 128 columns, N = MP tokens, K = 16:
//    D_j += A_tmem . B_smem) once the step's tokens have landed and the
//    unit's A buffer is written, then commits them to the A buffer's empty
//    barrier, and after the step to the token slot's empty barrier (two
//    arrivals, one per issuer, so a slot turns over only when both tiles'
//    UMMAs have read it); after a piece's last unit it commits to the
//    accumulator's full barrier.
// The three rings are independent: a weight stage is free once the decoders
// have read it, an A buffer once its UMMAs have completed, a token slot once
// both issuers' UMMAs of the step have completed; so the decoders never wait
// for tokens, and the token ring prefetches as far ahead as it is deep.
// Tensor memory: D_0 at column 0, D_1 at MP, then the A buffers (NA per
// group); 512 columns allocated.  A K = 16 UMMA of M = 128 takes 45 cycles
// at N <= 32 and 64 at N = 128 (measured), but on its issuing thread every
// mbarrier wait costs ~200 cycles and every commit ~45 while UMMAs are in
// flight; with two issuers one's wait overlaps the other's UMMAs.
// Every mbarrier wait is bounded; after a timeout every role runs to its
// end without waiting and the error word says W12_ERR_TIMEOUT.  The
// producers let their copies in flight land and the MMA threads wait
// (bounded) for their UMMAs before the tensor memory is freed.
#include <cuda.h>
#include <cuda_runtime.h>

#include "stream_device.cuh"
#include "verify_common.cuh"

namespace w12 {

namespace {

constexpr int kDW = 16;                  // decoder warps
constexpr int kDT = kDW * 32;
constexpr int kGT = kDT / 2;             // threads of one decoder group
constexpr int kWProdWarp = kDW;          // weight producer
constexpr int kXProdWarp = kDW + 1;      // token producer
constexpr int kMmaWarp = kDW + 2;        // tensor-memory owner, UMMA issuer of tile 0
constexpr int kTT = (kDW + 4) * 32;      // 640 threads
constexpr uint32_t kTmemCols = 512;
// named barriers: 1 all decoders, 2 + j decoder group j, 4 decoders + the
// tensor-memory owner (end of the kernel)
constexpr uint32_t kBarGroup = 2, kBarEnd = 4;

template <int MP>
struct TCfg {
    static constexpr int kX = MP * 256;                        // token slot: two boxes of MP rows x 128 bytes
    static constexpr int SX = MP >= 128 ? 2 : MP >= 64 ? 4 : MP >= 32 ? 3 : 4;  // token slots
    static constexpr int kXRing = SX * kX;                     // at the (1024-aligned) start of the ring
    static constexpr int kW = (kUnitBytes + 127) / 128 * 128;  // weight stage stride
    static constexpr int kFit = (227 * 1024 - 1024 - 2048 - kXRing) / kW;
    static constexpr int SWG = (kFit > 8 ? 8 : kFit) / 2;      // weight stages per decoder group
    static constexpr size_t kDynSmem = size_t(kXRing) + size_t(2 * SWG) * kW + 1024;
    // tensor-memory columns: accumulators [0, MP) and [MP, 2 MP); A buffer a
    // of group j at kA + 64 (j NA + a)
    static constexpr uint32_t kA = 2 * MP < 64 ? 64u : uint32_t(2 * MP);
    static constexpr int NA = int((kTmemCols - kA) / 128u) > 4 ? 4 : int((kTmemCols - kA) / 128u);
    static_assert(kA + 128u * NA <= kTmemCols, "A buffers exceed the tensor memory");
    static_assert(SWG >= 2 && NA >= 2, "rings too shallow");
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

// Store 32 consecutive 32-bit columns of this thread's lane.
__device__ __forceinline__ void tmem_st32(uint32_t taddr, const uint32_t (&v)[32]) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,"
        "%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};" ::"r"(taddr),
        "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7]), "r"(v[8]),
        "r"(v[9]), "r"(v[10]), "r"(v[11]), "r"(v[12]), "r"(v[13]), "r"(v[14]), "r"(v[15]), "r"(v[16]),
        "r"(v[17]), "r"(v[18]), "r"(v[19]), "r"(v[20]), "r"(v[21]), "r"(v[22]), "r"(v[23]), "r"(v[24]),
        "r"(v[25]), "r"(v[26]), "r"(v[27]), "r"(v[28]), "r"(v[29]), "r"(v[30]), "r"(v[31])
        : "memory");
    asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}

// Load 8 consecutive 32-bit columns of this thread's lane (no wait).
__device__ __forceinline__ void tmem_ld8(uint32_t taddr, uint32_t (&r)[8]) {
    asm volatile("tcgen05.ld.sync.aligned.32x32b.x8.b32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
                   "=r"(r[7])
                 : "r"(taddr));
}

__device__ __forceinline__ void tmem_ld_wait() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }

__device__ __forceinline__ void named_sync_id(uint32_t id, uint32_t nthreads) {
    asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(nthreads) : "memory");
}

__device__ __forceinline__ void named_arrive_id(uint32_t id, uint32_t nthreads) {
    asm volatile("bar.arrive %0, %1;" ::"r"(id), "r"(nthreads) : "memory");
}

// A slot of a ring: index and the parity of its current fill.
struct Ring {
    int s;
    uint32_t ph;
    template <int S>
    __device__ __forceinline__ void next() {
        if (++s == S) {
            s = 0;
            ph ^= 1u;
        }
    }
};

// Cursor over the pair order of a batch: product gi, pair p, group kg,
// tile j of the pair (tile 2 p + j of the product).  Every product has an
// even number of units (KG x the tile count rounded up to even), so the
// parity of a unit index is its j.
struct PCur {
    int gi, p, kg, j;
};

__device__ __forceinline__ int pairs_of(const StreamOne &g) { return (g.NB + 1) >> 1; }

__device__ __forceinline__ PCur p_at(const StreamBatch &b, int u) {
    PCur c{0, 0, 0, 0};
    while (c.gi + 1 < b.count && u >= b.g[c.gi + 1].ubase) ++c.gi;
    const int local = u - b.g[c.gi].ubase, KG = b.g[c.gi].KG;
    c.p = local / (2 * KG);
    const int r = local - c.p * 2 * KG;
    c.kg = r >> 1;
    c.j = r & 1;
    return c;
}

// The next step (same j).
__device__ __forceinline__ void p_next_step(const StreamBatch &b, PCur &c) {
    if (++c.kg == b.g[c.gi].KG) {
        c.kg = 0;
        if (++c.p == pairs_of(b.g[c.gi])) {
            c.p = 0;
            ++c.gi;
        }
    }
}

__device__ __forceinline__ void p_next(const StreamBatch &b, PCur &c) {
    if (c.j == 0) {
        c.j = 1;
    } else {
        c.j = 0;
        p_next_step(b, c);
    }
}

__device__ __forceinline__ int pair_first(const StreamBatch &b, const PCur &c) {
    return b.g[c.gi].ubase + c.p * 2 * b.g[c.gi].KG;
}

// The units of tile j of the pair that starts at unit pf (KG groups) which
// lie in [lo, hi): their number.
__device__ __forceinline__ int tile_units_in(int pf, int KG, int j, int lo, int hi) {
    lo = max(lo, pf + j);
    hi = min(hi, pf + 2 * KG);
    if (hi <= lo) return 0;
    // units pf + j + 2 t for t = 0 .. KG - 1
    const int t0 = (lo - pf - j + 1) >> 1, t1 = (hi - pf - j + 1) >> 1;
    return t1 - t0;
}

// L1 prefetch of the escape entries of tile nb's groups [kg0, kg1) (one
// contiguous range of the escape list), at most kEscPrefetchLines lines.
__device__ __forceinline__ void prefetch_tile_escapes(const StreamOne &g, int nb, int kg0, int kg1) {
    const uint8_t *u0 = g.units + size_t(uint32_t(nb) * uint32_t(g.KG) + uint32_t(kg0)) * kUnitBytes;
    const uint8_t *u1 = g.units + size_t(uint32_t(nb) * uint32_t(g.KG) + uint32_t(kg1 - 1)) * kUnitBytes;
    const uint32_t lo = ldg_u32(reinterpret_cast<const uint32_t *>(u0 + kMetaAt)) >> 8;
    const uint32_t hi = min(ldg_u32(reinterpret_cast<const uint32_t *>(u1 + kMetaAt + 4 * kTileN)) >> 8, g.n_esc);
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

// Weight producer (lane 0 of its warp): unit u of the CTA into the next
// stage of group u & 1's weight ring, once the group has released the
// stage's previous unit.  A phantom tile's unit (the padding tile of an odd
// tile count) copies nothing: the producer only arrives on the stage.
template <int SWG>
__device__ __forceinline__ void tc_weight_producer(const StreamBatch &b, uint32_t wbase, uint32_t stride,
                                                   uint64_t (*full_w)[SWG], uint64_t (*empty_w)[SWG],
                                                   WaitCtl *ctl, int u0, int u1) {
    if (!b.early_weights) pdl_wait();
    const uint64_t pol = l2_evict_first_policy();
    Ring r[2] = {{0, 0u}, {0, 0u}};
    int issued[2] = {0, 0};
    PCur c = p_at(b, u0);
    for (int u = u0; u < u1; ++u, p_next(b, c)) {
        const int j = c.j;
        Ring &q = r[j];
        // (a decoder that gave up sets the abort flag before it arrives
        // without waiting: stop, so the drain below covers every copy in flight)
        if (issued[j] >= SWG && (!mbar_wait(&empty_w[j][q.s], q.ph ^ 1u, ctl, b.err) || aborted(ctl))) break;
        const StreamOne &g = b.g[c.gi];
        const int nb = 2 * c.p + j;
        uint64_t *bar = &full_w[j][q.s];
        if (u != b.withhold_unit) {
            if (nb >= g.NB) {
                mbar_arrive(bar);
            } else {
                const int pf = pair_first(b, c);
                if (c.kg == 0 || u - 2 < u0) {
                    // first unit of this tile in the CTA: prefetch the
                    // escapes of the tile's groups up to the CTA's last one
                    const int last = min(u1 - 1, pf + 2 * g.KG - 1);
                    const int lu = (last & 1) == j ? last : last - 1;
                    prefetch_tile_escapes(g, nb, c.kg, ((lu - pf) >> 1) + 1);
                }
                mbar_expect_tx(bar, uint32_t(kUnitBytes));
                bulk_copy(wbase + uint32_t(j * SWG + q.s) * stride,
                          g.units + size_t(uint32_t(nb) * uint32_t(g.KG) + uint32_t(c.kg)) * kUnitBytes,
                          uint32_t(kUnitBytes), bar, pol);
            }
        }
        ++issued[j];
        q.template next<SWG>();
    }
    if (aborted(ctl)) {  // let the copies in flight land
        for (int j = 0; j < 2; ++j) {
            Ring q = r[j];
            for (int k = 0; k < SWG && k < issued[j]; ++k) {
                if (--q.s < 0) {
                    q.s = SWG - 1;
                    q.ph ^= 1u;
                }
                mbar_drain(&full_w[j][q.s], q.ph, ctl->limit_ns);
            }
        }
    }
}

// Token producer (lane 0 of its warp): the token box of each of the CTA's
// steps into the next token slot, once both issuers' UMMAs that read the
// slot's previous step have completed.  x may be written by the previous
// kernel of the stream.
template <int SX>
__device__ __forceinline__ void tc_x_producer(const StreamBatch &b, uint32_t xbase, int mp, uint64_t *full_x,
                                              uint64_t *empty_x, WaitCtl *ctl, int u0, int u1) {
    pdl_wait();
    const uint32_t kx = uint32_t(mp) * 256u;
    const int nsteps = ((u1 - 1) >> 1) - (u0 >> 1) + 1;
    PCur c = p_at(b, u0);
    Ring q{0, 0u};
    int issued = 0;
    for (int t = 0; t < nsteps; ++t, p_next_step(b, c)) {
        if (t >= SX && (!mbar_wait(&empty_x[q.s], q.ph ^ 1u, ctl, b.err) || aborted(ctl))) break;
        const StreamOne &g = b.g[c.gi];
        const uint32_t dst = xbase + uint32_t(q.s) * kx;
        uint64_t *bar = &full_x[q.s];
        mbar_expect_tx(bar, kx);
        tma_2d_keep(dst, &g.tx, 128 * c.kg, 0, bar);
        tma_2d_keep(dst + uint32_t(mp) * 128u, &g.tx, 128 * c.kg + 64, 0, bar);
        ++issued;
        q.template next<SX>();
    }
    if (aborted(ctl))
        for (int k = 0; k < SX && k < issued; ++k) {
            if (--q.s < 0) {
                q.s = SX - 1;
                q.ph ^= 1u;
            }
            mbar_drain(&full_x[q.s], q.ph, ctl->limit_ns);
        }
}

// Stream-K fix-up of tile nb = 2 p + j of a pair that starts at unit pf,
// run by the kGT threads of decoder group j (named barrier kBarGroup + j).
// Each piece of the tile adds its unit count to counters[nb]; the group
// that completes the count sums the pieces' partial slots in CTA order (the
// same bits on every call), writes y and resets the counter.  CTA c keeps
// the piece of the pair that contains its first unit in slots 0 + j and
// its other (last) pair piece in slots 2 + j.
template <bool FUSED>
__device__ __forceinline__ void tc_fixup(const StreamBatch &b, const StreamOne &g, int pf, int nb, int j,
                                         int count, int *s_last, int gtid, unsigned long long *s_best) {
    __threadfence();
    named_sync_id(kBarGroup + j, kGT);
    if (gtid == 0) {
        const uint32_t old = atomicAdd(&g.counters[nb], uint32_t(count));
        *s_last = (int(old) + count == g.KG);
    }
    named_sync_id(kBarGroup + j, kGT);
    if (*s_last) {
        __threadfence();
        const int G = int(gridDim.x), per = b.U / G, rem = b.U % G;
        const int KG = g.KG;
        const int c_first = sk_cta_of(pf + j, per, rem), c_last = sk_cta_of(pf + 2 * (KG - 1) + j, per, rem);
        const int M = b.M;
        const size_t slot_floats = size_t(M) * kTileN;
        for (int o = gtid; o < M * (kTileN / 4); o += kGT) {
            const int m = o / (kTileN / 4), c4 = o % (kTileN / 4);
            float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
            bool started = false;
            for (int c = c_first; c <= c_last; ++c) {
                const int beg = sk_unit_begin(c, per, rem), end = sk_unit_begin(c + 1, per, rem);
                if (tile_units_in(pf, KG, j, beg, end) == 0) continue;
                const int slot = (beg >= pf ? 0 : 2) + j;
                const float4 v = __ldcg(reinterpret_cast<const float4 *>(
                    b.partial + (size_t(c) * 4 + slot) * slot_floats + size_t(m) * kTileN) + c4);
                if (!started) {
                    acc = v;
                    started = true;
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
        if (gtid == 0) g.counters[nb] = 0u;
    }
    named_sync_id(kBarGroup + j, kGT);  // s_last is reused by the next piece
}

// FUSED: the lm_head + greedy verify epilogue (as in kernels_stream.cu):
// tile outputs fold into a per-CTA running (value, lowest index) maximum
// per token, split tiles are folded by the CTA that completes them, and the
// last CTA to arrive runs the acceptance rule over every CTA's keys.
template <int MP, bool FUSED>
__global__ void __launch_bounds__(kTT, 1) tc_kernel(const __grid_constant__ StreamBatch b) {
    using C = TCfg<MP>;
    constexpr int SWG = C::SWG, SX = C::SX, NA = C::NA;
    extern __shared__ unsigned char smem_dyn[];
    __shared__ __align__(8) uint64_t full_w[2][SWG], empty_w[2][SWG], full_x[SX], empty_x[SX];
    __shared__ __align__(8) uint64_t a_full[2][NA], a_empty[2][NA], acc_full[2], acc_empty[2], fin;
    __shared__ uint32_t s_tmem;
    __shared__ WaitCtl s_ctl;
    __shared__ int s_last[2];
    __shared__ unsigned long long s_best[FUSED ? MP : 1];
    const uint32_t xbase = (smem_addr(smem_dyn) + 1023u) & ~1023u;  // token ring, then the weight rings
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
        for (int j = 0; j < 2; ++j) {
            for (int s = 0; s < SWG; ++s) {
                mbar_init(&full_w[j][s], 1);       // the producer's (expect_tx) arrival
                mbar_init(&empty_w[j][s], kDW / 2);  // the group's warps
            }
            for (int a = 0; a < NA; ++a) {
                mbar_init(&a_full[j][a], kDW / 2);  // the group's warps
                mbar_init(&a_empty[j][a], 1);       // the issuer's commit
            }
            mbar_init(&acc_full[j], 1);
            mbar_init(&acc_empty[j], kDW / 2);
        }
        for (int s = 0; s < SX; ++s) {
            mbar_init(&full_x[s], 1);
            mbar_init(&empty_x[s], 2);  // one commit per issuer and step
        }
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
        if (lane == 0 && u0 < u1) tc_weight_producer<SWG>(b, wbase, C::kW, full_w, empty_w, &s_ctl, u0, u1);
        return;
    }
    if (warp == kXProdWarp) {
        if (lane == 0 && u0 < u1) tc_x_producer<SX>(b, xbase, MP, full_x, empty_x, &s_ctl, u0, u1);
        return;
    }
    pdl_wait();  // nothing below touches global memory the previous kernel may write before this

    if (warp >= kMmaWarp) {
        // ----------------------------------------------------------- UMMA issuers
        const int j = warp - kMmaWarp;  // units of parity j, accumulator D_j
        if (lane == 0 && u0 < u1) {
            const uint32_t idesc = idesc_bf16<MP>();
            const uint32_t dt = tmem + uint32_t(j * MP);
            const int nsteps = ((u1 - 1) >> 1) - (u0 >> 1) + 1;
            PCur c = p_at(b, u0 & ~1);
            Ring xq{0, 0u}, aq{0, 0u};
            int pieces = 0;
            bool fresh = true;
            for (int t = 0; t < nsteps; ++t, p_next_step(b, c)) {
                const int u = ((u0 >> 1) + t) * 2 + j;
                // every issuer waits for every step's tokens, so each phase
                // of a slot's empty barrier gets exactly the step's two commits
                mbar_wait(&full_x[xq.s], xq.ph, &s_ctl, b.err);
                if (u >= u0 && u < u1) {
                    const StreamOne &g = b.g[c.gi];
                    const bool first = c.kg == 0 || u - 2 < u0;
                    const bool last = c.kg == g.KG - 1 || u + 2 >= u1;
                    if (first) {
                        // the epilogue of the previous piece has read D_j
                        if (pieces > 0) mbar_wait(&acc_empty[j], uint32_t(pieces - 1) & 1u, &s_ctl, b.err);
                        fresh = true;
                    }
                    mbar_wait(&a_full[j][aq.s], aq.ph, &s_ctl, b.err);
                    tc_fence_after();
                    if (2 * c.p + j < g.NB) {
                        const uint64_t d0 = desc_sw128(xbase + uint32_t(xq.s) * uint32_t(C::kX));
                        const uint32_t ta = tmem + C::kA + 64u * uint32_t(j * NA + aq.s);
#pragma unroll
                        for (int ks = 0; ks < 8; ++ks) {
                            // x box ks / 4 (k half), 16 k = 32 bytes per step inside the swizzle atom
                            const uint64_t dx = d0 + uint64_t(((ks >> 2) * MP * 128 + 32 * (ks & 3)) >> 4);
                            umma_ts(dt, ta + 8u * uint32_t(ks), dx, idesc, (fresh && ks == 0) ? 0u : 1u);
                        }
                        fresh = false;
                    }
                    umma_commit(&a_empty[j][aq.s]);  // frees the A buffer
                    aq.template next<NA>();
                    if (last) {
                        umma_commit(&acc_full[j]);
                        ++pieces;
                    }
                }
                umma_commit(&empty_x[xq.s]);  // this issuer is done with the slot
                xq.template next<SX>();
            }
            // every UMMA issued has completed before the memory is freed
            umma_commit(&fin);
            mbar_drain(&fin, 0u, s_ctl.limit_ns);
        } else if (lane == 0) {
            umma_commit(&fin);
            mbar_drain(&fin, 0u, s_ctl.limit_ns);
        }
        __syncwarp();
        if (warp == kMmaWarp) {
            // the decoders have read the accumulators back
            named_sync_id(kBarEnd, kDT + 32);
            tc_fence_after();
            asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(kTmemCols)
                         : "memory");
        }
        return;
    }

    // ---------------------------------------------------------------- decoders
    const int j = warp >> 3;               // tile of the pair = unit parity
    const int gtid = threadIdx.x - j * kGT;
    const int r = 32 * (warp & 3) + lane;  // tile row = tensor-memory lane
    const int h = (warp & 7) >> 2;         // k half of the group; token half of the epilogue
    const uint32_t lane_off = uint32_t(32 * (warp & 3)) << 16;
    // plane row r, logical 16-byte chunks 2h and 2h + 1 (the format stores
    // chunk q of row r at q ^ ((r >> 1) & 3): a warp's 32 rows read 8
    // different bank groups per quarter-warp)
    const uint32_t sw = uint32_t((r >> 1) & 3);
    const uint32_t p0 = uint32_t(r * 64) + ((uint32_t(2 * h) ^ sw) << 4);
    const uint32_t p1 = uint32_t(r * 64) + ((uint32_t(2 * h + 1) ^ sw) << 4);
    const uint32_t wst0 = wbase + uint32_t(j * SWG) * uint32_t(C::kW);
    const uint32_t a0col = tmem + lane_off + C::kA + 64u * uint32_t(j * NA) + 32u * uint32_t(h);
    const int M = b.M;
    Ring wq{0, 0u}, aq{0, 0u};
    int uses = 0, pieces = 0;
    int ua = -1;  // first unit of the current piece
    const int ufirst = (u0 & 1) == j ? u0 : u0 + 1;
    PCur c = p_at(b, ufirst < u1 ? ufirst : u0);
    for (int u = ufirst; u < u1; u += 2, p_next_step(b, c)) {
        const StreamOne &g = b.g[c.gi];
        const int nb = 2 * c.p + j;
        const bool real = nb < g.NB;
        if (c.kg == 0 || ua < 0) ua = u;
        mbar_wait(&full_w[j][wq.s], wq.ph, &s_ctl, b.err);
        uint32_t w[32];
        if (real) {
            const uint32_t st = wst0 + uint32_t(wq.s) * uint32_t(C::kW);
            const uint4 h0 = lds128(st + p0), h1 = lds128(st + p1);
            const uint4 l0 = lds128(st + kPlaneBlock + p0), l1 = lds128(st + kPlaneBlock + p1);
            const uint4 e0 = lds128(st + 2 * kPlaneBlock + p0), e1 = lds128(st + 2 * kPlaneBlock + p1);
            const uint2 mw = make_uint2(lds32(st + kMetaAt + 4u * uint32_t(r)),
                                        lds32(st + kMetaAt + 4u * uint32_t(r) + 4u));
            __syncwarp();
            if (lane == 0) mbar_arrive(&empty_w[j][wq.s]);  // planes and meta read
            uint32_t(&wlo)[16] = *reinterpret_cast<uint32_t(*)[16]>(&w[0]);
            uint32_t(&whi)[16] = *reinterpret_cast<uint32_t(*)[16]>(&w[16]);
            const uint32_t b4 = base4(mw.x);
            rebuild32(h0, l0, e0, b4, wlo);
            rebuild32(h1, l1, e1, b4, whi);
            if (nb * kTileN + r < g.N && (mw.x >> 8) != (mw.y >> 8)) {
                patch_escapes(wlo, mw.x, mw.y, uint32_t(64 * h), g.esc, g.n_esc, b.err);
                patch_escapes(whi, mw.x, mw.y, uint32_t(64 * h + 32), g.esc, g.n_esc, b.err);
            }
        } else {
            __syncwarp();
            if (lane == 0) mbar_arrive(&empty_w[j][wq.s]);
        }
        wq.template next<SWG>();
        // the UMMAs that read this A buffer last have completed
        if (uses >= NA) mbar_wait(&a_empty[j][aq.s], aq.ph ^ 1u, &s_ctl, b.err);
        tc_fence_after();
        if (real) tmem_st32(a0col + 64u * uint32_t(aq.s), w);
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&a_full[j][aq.s]);
        aq.template next<NA>();
        ++uses;

        if (!(c.kg == g.KG - 1 || u + 2 >= u1)) continue;

        // ---- epilogue of the piece: accumulator D_j, row r, tokens
        // [h MP / 2, (h + 1) MP / 2), read 8 at a time.  The decoders start
        // the next piece only after it, so the accumulator is released at
        // its end.
        mbar_wait(&acc_full[j], uint32_t(pieces) & 1u, &s_ctl, b.err);
        ++pieces;
        tc_fence_after();
        if (real) {
            constexpr int kHalf = MP / 2;
            const int pf = pair_first(b, c);
            const int cnt = (u - ua) / 2 + 1;
            const int n = nb * kTileN + r;
            const bool valid = n < g.N;
            const bool whole = cnt == g.KG;
            // the pair holds the CTA's first unit: slots 0 + j, else 2 + j
            const int slot = (pf <= u0 ? 0 : 2) + j;
            float *P = b.partial + (size_t(blockIdx.x) * 4 + slot) * size_t(M) * kTileN;
#pragma unroll 1
            for (int q = 0; q < kHalf / 8; ++q) {
                uint32_t t8[8];
                tmem_ld8(tmem + lane_off + uint32_t(j * MP + h * kHalf + 8 * q), t8);
                tmem_ld_wait();
                const int m0 = h * kHalf + 8 * q;
                if (m0 >= M) break;
#pragma unroll
                for (int e = 0; e < 8; ++e) {
                    const float v = __uint_as_float(t8[e]);
                    const int m = m0 + e;
                    if (!whole) {
                        if (m < M) P[m * kTileN + r] = v;
                        continue;
                    }
                    if (valid && m < M && (!FUSED || g.y)) store_out(g.y, b.y_dtype, g.N, m, n, v);
                    if (FUSED) {
                        // per token: the warp's 32 rows -> one key, then the CTA maximum
                        unsigned long long best = valid ? pack_key(v, uint32_t(n)) : 0ull;
#pragma unroll
                        for (int off = 16; off >= 1; off >>= 1) {
                            const unsigned long long o = __shfl_xor_sync(0xFFFFFFFFu, best, off);
                            best = o > best ? o : best;
                        }
                        if (lane == 0 && m < M && best != 0ull) atomicMax(&s_best[m], best);
                    }
                }
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&acc_empty[j]);
            if (!whole) tc_fixup<FUSED>(b, g, pf, nb, j, cnt, &s_last[j], gtid, s_best);
        } else {
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&acc_empty[j]);
        }
        ua = -1;
    }
    tc_fence_before();
    named_arrive_id(kBarEnd, kDT + 32);  // accumulators read: the owner may free the tensor memory

    if (FUSED) {
        // publish this CTA's per-token best; the last CTA to arrive folds
        // them and runs the acceptance rule
        const int tid = threadIdx.x;
        named_sync(kDT);
        for (int m = tid; m < M; m += kDT) b.row_best[size_t(blockIdx.x) * M + m] = s_best[m];
        __threadfence();
        named_sync(kDT);
        if (tid == 0) s_last[0] = (atomicAdd(b.done, 1u) == gridDim.x - 1);
        named_sync(kDT);
        if (s_last[0]) {
            __threadfence();
            verify_from_keys(b.row_best, int64_t(gridDim.x), M, b.vR, b.vT, b.draft, b.accept_len, b.next_tok,
                             b.gbuf, tid, kDT);
            if (tid == 0) *b.done = 0u;
        }
    }
}

template <int MP, bool FUSED = false>
int launch_tc_t(const StreamBatch &b, int grid, cudaStream_t s) {
    return launch_pdl(tc_kernel<MP, FUSED>, grid, kTT, TCfg<MP>::kDynSmem, s, b);
}

template <int MP, bool FUSED = false>
int occ_tc_t(int *blocks) {
    if (cudaFuncSetAttribute(tc_kernel<MP, FUSED>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             int(TCfg<MP>::kDynSmem)) != cudaSuccess)
        return W12_ERR_CUDA;
    return cudaOccupancyMaxActiveBlocksPerMultiprocessor(blocks, tc_kernel<MP, FUSED>, kTT, TCfg<MP>::kDynSmem) ==
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
