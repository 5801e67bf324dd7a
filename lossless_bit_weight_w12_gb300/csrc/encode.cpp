// encode.cpp -- host encoder and validator for the W12 v2 blob.
//
// W12 splits each bf16 weight into three 4-bit planes (SpecPilot summary,
// airadar.tv English edition, "Reasons" bullet 2): the high and low nibble of
// the byte (mantissa << 1 | sign of the pair partner), and a 4-bit exponent
// code relative to a per-group base with an escape list for exponents
// outside the group window.  The layout (plane-major units of 128 columns x
// one 128-k group, each one contiguous block with its meta words) is the one
// documented in include/w12.h.  Groups are independent: the scan runs
// OpenMP-parallel over groups, the packing over units.
#include <cstring>
#include <vector>

#include "w12_internal.h"

namespace w12 {

namespace {

// Nibble slot -> weight index inside an 8-weight word, per plane.
constexpr int kPermH[8] = {4, 0, 5, 1, 6, 2, 7, 3};
constexpr int kPermL[8] = {0, 5, 1, 6, 2, 7, 3, 4};
constexpr int kPermE[8] = {0, 4, 1, 5, 2, 6, 3, 7};

inline unsigned exp_of(uint16_t v) { return (v >> 7) & 0xFFu; }

// Base of a group: window [b, b+14] with the most exponents, largest b on ties.
unsigned group_base(const uint16_t *v) {
    int hist[256] = {0};
    for (int i = 0; i < kGroup; ++i) ++hist[exp_of(v[i])];
    int cover = 0;
    for (int e = 0; e < 15; ++e) cover += hist[e];
    int best = cover;
    unsigned best_b = 0;
    for (int b = 1; b <= kMaxBase; ++b) {
        cover += hist[b + 14] - hist[b - 1];
        if (cover >= best) {
            best = cover;
            best_b = unsigned(b);
        }
    }
    return best_b;
}

inline bool in_window(unsigned e, unsigned b) { return e >= b && e <= b + 14; }

// Copies group (n, kg) into out[128] for either input orientation.
inline void load_group(const uint16_t *w, int64_t K, int64_t N, int layout, int64_t n, int64_t kg,
                       uint16_t *out) {
    if (layout == W12_LAYOUT_NK) {
        std::memcpy(out, w + n * K + kg * kGroup, kGroup * sizeof(uint16_t));
    } else {
        const uint16_t *p = w + (kg * kGroup) * N + n;
        for (int i = 0; i < kGroup; ++i) out[i] = p[int64_t(i) * N];
    }
}

int check_shape(const uint16_t *w, int64_t K, int64_t N, int layout) {
    if (layout != W12_LAYOUT_KN && layout != W12_LAYOUT_NK) return W12_ERR_ARG;
    if (K < 0 || N < 0 || K % kGroup != 0) return W12_ERR_SHAPE;
    if (!w && K * N > 0) return W12_ERR_ARG;
    return W12_OK;
}

// Per-group base and escape count.  For the KN orientation groups are walked
// column-block by column-block so neighbouring columns share cache lines.
void scan_groups(const uint16_t *w, int64_t K, int64_t N, int layout, uint8_t *base,
                 uint32_t *count) {
    const int64_t KG = K / kGroup;
    const int64_t G = N * KG;
#pragma omp parallel for schedule(static)
    for (int64_t g = 0; g < G; ++g) {
        // KN: order the iteration so consecutive g share k (g = kg*N + n).
        int64_t n, kg;
        if (layout == W12_LAYOUT_KN) {
            kg = g / N;
            n = g % N;
        } else {
            n = g / KG;
            kg = g % KG;
        }
        uint16_t v[kGroup];
        load_group(w, K, N, layout, n, kg, v);
        unsigned b = group_base(v);
        uint32_t c = 0;
        for (int i = 0; i < kGroup; ++i) c += !in_window(exp_of(v[i]), b);
        const int64_t gid = n * KG + kg;
        base[gid] = uint8_t(b);
        count[gid] = c;
    }
}

inline void store_u32(uint8_t *p, uint32_t v) { std::memcpy(p, &v, 4); }
inline uint32_t load_u32(const uint8_t *p) {
    uint32_t v;
    std::memcpy(&v, p, 4);
    return v;
}
inline uint16_t load_u16(const uint8_t *p) {
    uint16_t v;
    std::memcpy(&v, p, 2);
    return v;
}

}  // namespace

void layout_v2(int64_t K, int64_t N, uint64_t n_esc, w12_desc *d) {
    d->version = W12_FORMAT_VERSION;
    d->reserved = 0;
    d->K = K;
    d->N = N;
    d->G = N * (K / kGroup);
    d->tiles = uint64_t((N + kTileCols - 1) / kTileCols);
    d->unit_bytes = kUnitBytes;
    d->n_units = d->tiles * uint64_t(K / kGroup);
    d->off_units = 0;
    d->off_esc = round256(d->n_units * kUnitBytes);
    d->n_esc = n_esc;
    d->total_bytes = round256(d->off_esc + 2u * n_esc);
}

}  // namespace w12

using namespace w12;

extern "C" int w12_encode_plan(const uint16_t *w, int64_t K, int64_t N, int layout,
                               w12_desc *d) {
    int st = check_shape(w, K, N, layout);
    if (st != W12_OK) return st;
    if (!d) return W12_ERR_ARG;
    const int64_t G = N * (K / kGroup);
    std::vector<uint8_t> base(size_t(G > 0 ? G : 1));
    std::vector<uint32_t> count(size_t(G > 0 ? G : 1));
    if (G > 0) scan_groups(w, K, N, layout, base.data(), count.data());
    uint64_t n_esc = 0;
    for (int64_t g = 0; g < G; ++g) n_esc += count[g];
    if (n_esc >= kMaxEscapes) return W12_ERR_TOO_MANY_ESCAPES;
    layout_v2(K, N, n_esc, d);
    return W12_OK;
}

namespace w12 {

namespace {

// Escape begin of every (unit, tile column): running count in unit, then
// column order (padding columns take no escapes).  begin has U * 129 + 1
// entries; entry u * 129 + 128 is where unit u + 1 starts.
uint64_t escape_begins(const uint32_t *count, int64_t K, int64_t N, uint64_t U, std::vector<uint64_t> &begin) {
    const int64_t KG = K / kGroup;
    begin.assign(size_t(U) * (kTileCols + 1) + 1, 0);
    uint64_t run = 0;
    for (uint64_t u = 0; u < U; ++u) {
        const int64_t t = int64_t(u) / KG, kg = int64_t(u) % KG;
        for (int c = 0; c < kTileCols; ++c) {
            begin[u * (kTileCols + 1) + c] = run;
            const int64_t n = t * kTileCols + c;
            if (n < N) run += count[n * KG + kg];
        }
        begin[u * (kTileCols + 1) + kTileCols] = run;
    }
    return run;
}

// Byte offset, inside its unit block, of word wi (0..15) of column c of a
// plane: 16-byte chunk wi / 4 stored at chunk position (wi / 4) ^ ((c >> 1) & 3).
inline uint32_t word_offset(int plane, int c, int wi) {
    const int j = (wi >> 2) ^ ((c >> 1) & 3);
    return uint32_t(plane * kPlaneBlock + c * 64 + j * 16 + (wi & 3) * 4);
}

}  // namespace

}  // namespace w12

extern "C" int w12_encode(const uint16_t *w, int64_t K, int64_t N, int layout, const w12_desc *d,
                          void *blob_host) {
    int st = check_shape(w, K, N, layout);
    if (st != W12_OK) return st;
    if (!d || !blob_host || d->K != K || d->N != N || d->version != W12_FORMAT_VERSION)
        return W12_ERR_ARG;
    const int64_t KG = K / kGroup, G = N * KG;
    std::vector<uint8_t> base(size_t(G > 0 ? G : 1));
    std::vector<uint32_t> count(size_t(G > 0 ? G : 1));
    if (G > 0) scan_groups(w, K, N, layout, base.data(), count.data());
    w12_desc want;
    layout_v2(K, N, 0, &want);
    const uint64_t U = want.n_units;
    std::vector<uint64_t> begin;
    const uint64_t run = escape_begins(count.data(), K, N, U, begin);
    if (run >= kMaxEscapes) return W12_ERR_TOO_MANY_ESCAPES;
    layout_v2(K, N, run, &want);
    if (std::memcmp(&want, d, sizeof want) != 0) return W12_ERR_ARG;

    uint8_t *blob = static_cast<uint8_t *>(blob_host);
    std::memset(blob, 0, d->total_bytes);
    uint8_t *esc = blob + d->off_esc;

#pragma omp parallel for schedule(dynamic, 16)
    for (int64_t u = 0; u < int64_t(U); ++u) {
        const int64_t t = u / KG, kg = u % KG;
        uint8_t *ub = blob + uint64_t(u) * kUnitBytes;
        const uint64_t *bg = &begin[uint64_t(u) * (kTileCols + 1)];
        for (int c = 0; c < kTileCols; ++c) {
            const int64_t n = t * kTileCols + c;
            if (n >= N) {
                store_u32(ub + kMetaAt + 4 * c, uint32_t(bg[c] << 8));  // padding: base 0
                continue;
            }
            const int64_t gid = n * KG + kg;
            uint16_t v[kGroup];
            load_group(w, K, N, layout, n, kg, v);
            const unsigned b = base[gid];
            store_u32(ub + kMetaAt + 4 * c, uint32_t(b) | uint32_t(bg[c] << 8));
            uint64_t at = bg[c];
            for (int p = 0; p < kGroup; ++p) {
                const unsigned e = exp_of(v[p]);
                if (!in_window(e, b)) {
                    const uint16_t ent = uint16_t(unsigned(p) | (e << 7));
                    std::memcpy(esc + 2 * at, &ent, 2);
                    ++at;
                }
            }
            for (int wi = 0; wi < kGroup / 8; ++wi) {
                const uint16_t *q = v + 8 * wi;
                uint32_t hw = 0, lw = 0, ew = 0;
                for (int s = 0; s < 8; ++s) {
                    // byte m << 1 | sign of the pair partner (weights 2i and 2i+1)
                    const int jh = kPermH[s], jl = kPermL[s];
                    const uint32_t smh = ((q[jh] & 0x7Fu) << 1) | (q[jh ^ 1] >> 15);
                    const uint32_t sml = ((q[jl] & 0x7Fu) << 1) | (q[jl ^ 1] >> 15);
                    const unsigned ee = exp_of(q[kPermE[s]]);
                    hw |= (smh >> 4) << (4 * s);
                    lw |= (sml & 0xFu) << (4 * s);
                    ew |= (in_window(ee, b) ? ee - b : 15u) << (4 * s);
                }
                store_u32(ub + word_offset(0, c, wi), hw);
                store_u32(ub + word_offset(1, c, wi), lw);
                store_u32(ub + word_offset(2, c, wi), ew);
            }
        }
        store_u32(ub + kMetaAt + 4 * kTileCols, uint32_t(bg[kTileCols] << 8));
    }
    return W12_OK;
}

extern "C" int w12_validate(const w12_desc *d, const void *blob_host) {
    if (!d || !blob_host) return W12_ERR_ARG;
    if (d->version != W12_FORMAT_VERSION || d->K < 0 || d->N < 0 || d->K % kGroup != 0)
        return W12_ERR_ARG;
    if (d->n_esc >= kMaxEscapes) return W12_ERR_BLOB;
    w12_desc want;
    layout_v2(d->K, d->N, d->n_esc, &want);
    if (std::memcmp(&want, d, sizeof want) != 0) return W12_ERR_BLOB;
    const uint8_t *blob = static_cast<const uint8_t *>(blob_host);
    const int64_t K = d->K, N = d->N, KG = K / kGroup;
    const int64_t U = int64_t(d->n_units);
    const uint8_t *esc = blob + d->off_esc;
    int bad = 0;
#pragma omp parallel for schedule(dynamic, 16) reduction(| : bad)
    for (int64_t u = 0; u < U; ++u) {
        const int64_t t = u / KG;
        const uint8_t *ub = blob + uint64_t(u) * kUnitBytes;
        // the unit's word 128 is the next unit's first begin (n_esc after the last)
        const uint32_t last = load_u32(ub + kMetaAt + 4 * kTileCols);
        const uint64_t next = (u + 1 < U) ? (load_u32(ub + kUnitBytes + kMetaAt) >> 8) : d->n_esc;
        if ((last & 0xFFu) != 0 || (last >> 8) != next) bad |= 1;
        for (int z = 0; z < kUnitBytes - kMetaAt - 4 * (kTileCols + 1); ++z)
            if (ub[kMetaAt + 4 * (kTileCols + 1) + z] != 0) bad |= 1;
        for (int c = 0; c < kTileCols && !bad; ++c) {
            const uint32_t m0 = load_u32(ub + kMetaAt + 4 * c), m1 = load_u32(ub + kMetaAt + 4 * (c + 1));
            const unsigned b = m0 & 0xFFu;
            const uint64_t lo = m0 >> 8, hi = m1 >> 8;
            if (b > unsigned(kMaxBase) || lo > hi || hi > d->n_esc) {
                bad |= 1;
                break;
            }
            if (t * kTileCols + c >= N) {
                // padding column: base 0, no escapes, zero planes
                if (b != 0 || lo != hi) bad |= 1;
                for (int plane = 0; plane < 3; ++plane)
                    for (int i = 0; i < 64; ++i)
                        if (ub[plane * kPlaneBlock + c * 64 + i] != 0) bad |= 1;
                continue;
            }
            // positions whose code is 15, in pos order
            int flagged[kGroup];
            int nf = 0;
            for (int wi = 0; wi < kGroup / 8; ++wi) {
                const uint32_t ew = load_u32(ub + word_offset(2, c, wi));
                for (int r = 0; r < 8; ++r) {
                    const int s = (r < 4) ? 2 * r : 2 * (r - 4) + 1;  // slot of weight r in E
                    if (((ew >> (4 * s)) & 0xFu) == 15u) flagged[nf++] = 8 * wi + r;
                }
            }
            if (uint64_t(nf) != hi - lo) {
                bad |= 1;
                break;
            }
            for (int i = 0; i < nf; ++i) {
                const uint16_t ent = load_u16(esc + 2 * (lo + i));
                const unsigned pos = ent & 0x7Fu, e = (ent >> 7) & 0xFFu;
                if ((ent >> 15) != 0 || int(pos) != flagged[i] || in_window(e, b)) bad |= 1;
            }
        }
    }
    if (U > 0 && (load_u32(blob + kMetaAt) >> 8) != 0) bad |= 1;  // escapes start at entry 0
    return bad ? W12_ERR_BLOB : W12_OK;
}
