// device_common.cuh -- register-level W12 rebuild shared by the kernels.
//
// "Reconstructing bit by bit in GEMM registers" (SpecPilot summary,
// airadar.tv English edition, "Reasons" bullet 2): one 32-bit word from each
// of the H, L and E planes covers 8 consecutive k of one column; the nibble
// order inside each word (include/w12.h) is chosen so that the 8 bf16 values
// come out as 4 bf16x2 registers (k0,k0+1), (k0+2,k0+3), ... in 16 integer
// instructions (14 on the ALU pipe, 2 adds that can run as IMAD):
//   SMA = (H & 0xF0F0F0F0) | (L & 0x0F0F0F0F)   bytes SM'(k0..k0+3)
//   SMB = rotl((H & 0x0F0F0F0F) | (L & 0xF0F0F0F0), 4)      SM'(k0+4..k0+7)
//   XE  = (E & 0x0F0F0F0F) + b * 0x01010101      exponents of k0..k0+3
//   XO  = ((E >> 4) & 0x0F0F0F0F) + b * 0x01010101           k0+4..k0+7
//   P_i = rotr(prmt(SM, X, [SM'lo, e lo, SM'hi, e hi]), 1)
// where SM'(j) = m(j) << 1 | s(partner of j): after the byte gather a pair
// word reads [e_hi | m_hi | s_lo | e_lo | m_lo | s_hi] and one 32-bit rotate
// right moves every field of both halves into its bf16 place, the two signs
// crossing over.  The base is at most 240, so b + code (<= 255) never carries
// between bytes.  An escape (code 15) leaves a wrong exponent that
// patch_escapes() replaces (in the tcgen05 decoders: the column's first
// entry in tensor memory, esc_apply_rest() the others).
#pragma once

#include <cstdint>

#include "../../include/w12.h"

namespace w12 {

constexpr uint32_t kSignManMask = 0x807F807Fu;

// Record a device error in a workspace's error word: the first error of a
// call wins (a CTA that gave up on a bounded wait may read a stage that
// never filled and meet garbage escape indices afterwards; the timeout is
// what the caller must see).
__device__ __forceinline__ void record_error(int *err, int code) {
    if (err) atomicCAS(err, 0, code);
}

// Streaming 16-byte load: read once, keep out of L1, ask L2 for 256-byte lines.
__device__ __forceinline__ uint4 ldg_stream(const void *p) {
    uint4 r;
    asm("ld.global.nc.L1::no_allocate.L2::256B.v4.u32 {%0,%1,%2,%3}, [%4];"
        : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
        : "l"(p));
    return r;
}

__device__ __forceinline__ uint32_t ldg_u32(const uint32_t *p) {
    uint32_t r;
    asm("ld.global.nc.u32 %0, [%1];" : "=r"(r) : "l"(p));
    return r;
}

__device__ __forceinline__ uint4 ldg_v4(const void *p) {
    uint4 r;
    asm("ld.global.nc.v4.u32 {%0,%1,%2,%3}, [%4];"
        : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
        : "l"(p));
    return r;
}

// Byte gather from two registers: selector nibble i picks byte (0-3 of a,
// 4-7 of b) for result byte i.
__device__ __forceinline__ uint32_t prmt2(uint32_t a, uint32_t b, uint32_t sel) {
    uint32_t d;
    asm("prmt.b32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(sel));
    return d;
}

// Rebuild 8 weights (one word of each plane) into 4 bf16x2 registers.
// b4 = base * 0x01010101.
__device__ __forceinline__ void rebuild8(uint32_t h, uint32_t l, uint32_t e, uint32_t b4,
                                         uint32_t out[4]) {
    const uint32_t sma = (h & 0xF0F0F0F0u) | (l & 0x0F0F0F0Fu);
    const uint32_t xx = (h & 0x0F0F0F0Fu) | (l & 0xF0F0F0F0u);
    const uint32_t smb = __funnelshift_l(xx, xx, 4);
    const uint32_t xe = (e & 0x0F0F0F0Fu) + b4;
    const uint32_t xo = ((e >> 4) & 0x0F0F0F0Fu) + b4;
    const uint32_t p0 = prmt2(sma, xe, 0x5140u), p1 = prmt2(sma, xe, 0x7362u);
    const uint32_t p2 = prmt2(smb, xo, 0x5140u), p3 = prmt2(smb, xo, 0x7362u);
    out[0] = __funnelshift_r(p0, p0, 1);
    out[1] = __funnelshift_r(p1, p1, 1);
    out[2] = __funnelshift_r(p2, p2, 1);
    out[3] = __funnelshift_r(p3, p3, 1);
}

// Rebuild the 32 weights of one 16-byte vector of each plane.
__device__ __forceinline__ void rebuild32(const uint4 &h, const uint4 &l, const uint4 &e,
                                          uint32_t b4, uint32_t out[16]) {
    rebuild8(h.x, l.x, e.x, b4, out + 0);
    rebuild8(h.y, l.y, e.y, b4, out + 4);
    rebuild8(h.z, l.z, e.z, b4, out + 8);
    rebuild8(h.w, l.w, e.w, b4, out + 12);
}

__device__ __forceinline__ uint32_t base4(uint32_t meta_word) { return (meta_word & 0xFFu) * 0x01010101u; }

// acc_lo += w.lo * x.lo, acc_hi += w.hi * x.hi: bf16 operands, fp32
// accumulate, one rounding (the product of two bf16 values is exact in fp32).
__device__ __forceinline__ void fma_bf16x2(float &acc_lo, float &acc_hi, uint32_t w, uint32_t x) {
    asm("{\n .reg .b16 wl, wh, xl, xh;\n mov.b32 {wl, wh}, %2;\n mov.b32 {xl, xh}, %3;\n"
        " fma.rn.f32.bf16 %0, wl, xl, %0;\n fma.rn.f32.bf16 %1, wh, xh, %1;\n}\n"
        : "+f"(acc_lo), "+f"(acc_hi)
        : "r"(w), "r"(x));
}

// Replace the exponent of escaped weights among the 32 weights
// [pos0, pos0 + 32) of a group held in out[16] (pair r/2 of word r/8 ...).
// m0 = meta[g], m1 = meta[g+1].  Indices are bounds-checked; a corrupt entry
// range records W12_ERR_DEVICE and is skipped.
__device__ __forceinline__ void patch_escapes(uint32_t out[16], uint32_t m0, uint32_t m1,
                                                  uint32_t pos0, const uint16_t *esc,
                                                  uint64_t n_esc, int *err) {
    const uint32_t lo = m0 >> 8, hi = m1 >> 8;
    if (hi < lo || uint64_t(hi) > n_esc || hi - lo > 128u) {
        record_error(err, W12_ERR_DEVICE);
        return;
    }
    for (uint32_t i = lo; i < hi; ++i) {
        const uint32_t ent = esc[i];
        const uint32_t pos = ent & 0x7Fu;
        if ((pos & ~31u) != pos0) continue;
        const uint32_t j = pos & 31u;
        const uint32_t idx = (j >> 3) * 4 + ((j & 7u) >> 1);
        const uint32_t sh = (j & 1u) * 16u;
        const uint32_t mask = 0x7F80u << sh;
        const uint32_t val = (ent & 0x7F80u) << sh;
#pragma unroll
        for (int q = 0; q < 16; ++q)
            if (uint32_t(q) == idx) out[q] = (out[q] & ~mask) | val;
    }
}

// Escape patch-up split in two, so that the (rare) escape entries are read
// while the rebuild runs: esc_begin() is called as soon as a column's meta
// words m0 = meta[c], m1 = meta[c + 1] are in registers; it checks the
// column's entry range (a corrupt range records W12_ERR_DEVICE and is not
// followed) and starts the load of its first entry, which the caller
// patches once the rebuild is done; esc_apply_rest() patches every further
// entry (two or more escapes in one column of a group) whose pos falls in
// the 32 weights [pos0, pos0 + 32) held in out[16] (pair r/2 of word r/8
// ...), loading each.
struct EscPending {
    uint32_t lo, hi, e0;
};

__device__ __forceinline__ uint32_t ldg_u16(const uint16_t *p) {
    uint16_t r;
    asm("ld.global.nc.u16 %0, [%1];" : "=h"(r) : "l"(p));
    return r;
}

__device__ __forceinline__ EscPending esc_begin(bool col_valid, uint32_t m0, uint32_t m1, const uint16_t *esc,
                                                uint64_t n_esc, int *err) {
    EscPending e{m0 >> 8, m1 >> 8, 0u};
    if (!col_valid || e.lo == e.hi) {
        e.hi = e.lo;  // nothing to patch
        return e;
    }
    if (e.hi < e.lo || uint64_t(e.hi) > n_esc || e.hi - e.lo > 128u) {
        record_error(err, W12_ERR_DEVICE);
        e.hi = e.lo;
        return e;
    }
    e.e0 = ldg_u16(esc + e.lo);
    return e;
}

__device__ __forceinline__ void esc_patch_one(uint32_t out[16], uint32_t pos0, uint32_t ent) {
    const uint32_t pos = ent & 0x7Fu;
    if ((pos & ~31u) != pos0) return;
    const uint32_t j = pos & 31u;
    const uint32_t idx = (j >> 3) * 4 + ((j & 7u) >> 1);
    const uint32_t sh = (j & 1u) * 16u;
    const uint32_t mask = 0x7F80u << sh;
    const uint32_t val = (ent & 0x7F80u) << sh;
#pragma unroll
    for (int q = 0; q < 16; ++q)
        if (uint32_t(q) == idx) out[q] = (out[q] & ~mask) | val;
}

// Patch the 32 weights of out (positions [pos0, pos0 + 32)) from a pending
// escape range.
// The entries after a column's first one (the first is patched by the
// caller).
__device__ __forceinline__ void esc_apply_rest(const EscPending &e, uint32_t out[16], uint32_t pos0,
                                               const uint16_t *esc) {
    for (uint32_t i = e.lo + 1; i < e.hi; ++i) esc_patch_one(out, pos0, ldg_u16(esc + i));
}

// Float ordering key for the argmax: larger key = larger value; NaN above
// everything; -0 and +0 equal.  Packed with ~index so ties go to the lowest.
__device__ __forceinline__ uint32_t order_key(float f) {
    uint32_t u = __float_as_uint(f);
    if ((u & 0x7FFFFFFFu) > 0x7F800000u) return 0xFFFFFFFFu;  // NaN
    if ((u & 0x7FFFFFFFu) == 0u) u = 0u;                      // -0 -> +0
    return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

__device__ __forceinline__ unsigned long long pack_key(float f, uint32_t idx) {
    return (static_cast<unsigned long long>(order_key(f)) << 32) | (0xFFFFFFFFu - idx);
}

__device__ __forceinline__ uint32_t key_index(unsigned long long k) {
    return 0xFFFFFFFFu - static_cast<uint32_t>(k & 0xFFFFFFFFull);
}

__device__ __forceinline__ float bf16_bits_to_float(uint32_t b) { return __uint_as_float(b << 16); }

}  // namespace w12
