// encode.cpp -- host encoder and validator for the W12 v1 blob.
//
// W12 splits each bf16 weight into three 4-bit planes (SpecPilot summary,
// airadar.tv English edition, "Reasons" bullet 2): the high and low nibble of
// the byte (mantissa << 1 | sign of the pair partner), and a 4-bit exponent
// code relative to a per-group base with an escape list for exponents
// outside the group window.  The layout is
// the one documented in include/w12.h.  Groups are independent, so both
// passes run OpenMP-parallel over groups.
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

void layout_v1(int64_t K, int64_t N, uint64_t n_esc, w12_desc *d) {
    const uint64_t plane = uint64_t(K) * uint64_t(N) / 2;
    d->version = W12_FORMAT_VERSION;
    d->reserved = 0;
    d->K = K;
    d->N = N;
    d->G = N * (K / kGroup);
    d->off_h = 0;
    d->off_l = round256(d->off_h + plane);
    d->off_e = round256(d->off_l + plane);
    d->off_meta = round256(d->off_e + plane);
    d->off_esc = round256(d->off_meta + 4u * uint64_t(d->G + 1));
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
    layout_v1(K, N, n_esc, d);
    return W12_OK;
}

extern "C" int w12_encode(const uint16_t *w, int64_t K, int64_t N, int layout, const w12_desc *d,
                          void *blob_host) {
    int st = check_shape(w, K, N, layout);
    if (st != W12_OK) return st;
    if (!d || !blob_host || d->K != K || d->N != N || d->version != W12_FORMAT_VERSION)
        return W12_ERR_ARG;
    const int64_t KG = K / kGroup, G = N * KG, KW = K / 8;
    std::vector<uint8_t> base(size_t(G > 0 ? G : 1));
    std::vector<uint32_t> count(size_t(G > 0 ? G : 1));
    if (G > 0) scan_groups(w, K, N, layout, base.data(), count.data());
    std::vector<uint64_t> begin(size_t(G + 1));
    uint64_t run = 0;
    for (int64_t g = 0; g < G; ++g) {
        begin[g] = run;
        run += count[g];
    }
    begin[G] = run;
    w12_desc want;
    if (run >= kMaxEscapes) return W12_ERR_TOO_MANY_ESCAPES;
    layout_v1(K, N, run, &want);
    if (std::memcmp(&want, d, sizeof want) != 0) return W12_ERR_ARG;

    uint8_t *blob = static_cast<uint8_t *>(blob_host);
    std::memset(blob, 0, d->total_bytes);
    uint8_t *H = blob + d->off_h, *L = blob + d->off_l, *E = blob + d->off_e;
    uint8_t *meta = blob + d->off_meta, *esc = blob + d->off_esc;

#pragma omp parallel for schedule(static)
    for (int64_t g = 0; g < G; ++g) {
        const int64_t n = g / KG, kg = g % KG;
        uint16_t v[kGroup];
        load_group(w, K, N, layout, n, kg, v);
        const unsigned b = base[g];
        store_u32(meta + 4 * g, uint32_t(b) | uint32_t(begin[g] << 8));
        uint64_t at = begin[g];
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
                const uint16_t ve = q[kPermE[s]];
                const uint32_t hn = smh >> 4;
                const uint32_t ln = sml & 0xFu;
                const unsigned ee = exp_of(ve);
                const uint32_t en = in_window(ee, b) ? ee - b : 15u;
                hw |= hn << (4 * s);
                lw |= ln << (4 * s);
                ew |= en << (4 * s);
            }
            const uint64_t word = uint64_t(n) * KW + uint64_t(kg) * 16 + wi;
            store_u32(H + 4 * word, hw);
            store_u32(L + 4 * word, lw);
            store_u32(E + 4 * word, ew);
        }
    }
    store_u32(meta + 4 * G, uint32_t(run << 8));
    return W12_OK;
}

extern "C" int w12_validate(const w12_desc *d, const void *blob_host) {
    if (!d || !blob_host) return W12_ERR_ARG;
    if (d->version != W12_FORMAT_VERSION || d->K < 0 || d->N < 0 || d->K % kGroup != 0)
        return W12_ERR_ARG;
    if (d->n_esc >= kMaxEscapes) return W12_ERR_BLOB;
    w12_desc want;
    layout_v1(d->K, d->N, d->n_esc, &want);
    if (std::memcmp(&want, d, sizeof want) != 0) return W12_ERR_BLOB;
    const uint8_t *blob = static_cast<const uint8_t *>(blob_host);
    const int64_t K = d->K, KG = K / kGroup, G = d->G, KW = K / 8;
    const uint8_t *E = blob + d->off_e, *meta = blob + d->off_meta, *esc = blob + d->off_esc;
    if ((load_u32(meta + 4 * G) & 0xFFu) != 0 || (load_u32(meta + 4 * G) >> 8) != d->n_esc)
        return W12_ERR_BLOB;
    int bad = 0;
#pragma omp parallel for schedule(static) reduction(| : bad)
    for (int64_t g = 0; g < G; ++g) {
        const uint32_t m0 = load_u32(meta + 4 * g), m1 = load_u32(meta + 4 * (g + 1));
        const unsigned b = m0 & 0xFFu;
        const uint64_t lo = m0 >> 8, hi = m1 >> 8;
        if (b > unsigned(kMaxBase) || lo > hi || hi > d->n_esc) {
            bad |= 1;
            continue;
        }
        const int64_t n = g / KG, kg = g % KG;
        // positions whose code is 15, in pos order
        int flagged[kGroup];
        int nf = 0;
        for (int wi = 0; wi < kGroup / 8; ++wi) {
            const uint32_t ew = load_u32(E + 4 * (uint64_t(n) * KW + uint64_t(kg) * 16 + wi));
            for (int r = 0; r < 8; ++r) {
                const int s = (r < 4) ? 2 * r : 2 * (r - 4) + 1;  // slot of weight r in E
                if (((ew >> (4 * s)) & 0xFu) == 15u) flagged[nf++] = 8 * wi + r;
            }
        }
        if (uint64_t(nf) != hi - lo) {
            bad |= 1;
            continue;
        }
        for (int i = 0; i < nf; ++i) {
            const uint16_t ent = load_u16(esc + 2 * (lo + i));
            const unsigned pos = ent & 0x7Fu, e = (ent >> 7) & 0xFFu;
            if ((ent >> 15) != 0 || int(pos) != flagged[i] || in_window(e, b)) bad |= 1;
        }
    }
    return bad ? W12_ERR_BLOB : W12_OK;
}
