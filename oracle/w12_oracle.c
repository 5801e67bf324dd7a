/*
 * w12_oracle.c -- plain, slow CPU oracle for the W12 hot path.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product library calls, links or
 * includes this file; only the test suite, the smoke check and the CPU-baseline
 * leg of the benchmark load it (through ctypes).  It shares no source with the
 * CUDA library: every constant, table and layout rule below is written out
 * here on its own.
 *
 * What it computes, and where each piece comes from:
 *
 *  - The W12 format: a BF16 weight is split into three 4-bit planes and
 *    rebuilt bit for bit ("SpecPilot" summary pages, p5 "Reasons", second
 *    bullet; p4 "项目介绍", second paragraph: decoded bit-exactly inside the
 *    GEMM).  The pages give no layout; the one coded here is the documented
 *    W12 v2 layout: planes H and L = the high and low nibble of the byte
 *    (mantissa << 1 | sign of the pair partner), plane E = the exponent as a
 *    4-bit offset from a base shared by a group of 128 consecutive k of one
 *    output column, with code 15 meaning "escape: the true exponent is in a
 *    side list"; the three planes and the group bases of 128 columns x one
 *    group are packed together as one block ("unit").
 *  - The GEMM: y[m,n] = sum_k x[m,k] * w[k,n], accumulated in fp64 in k order
 *    (products of two bf16 values are exact in fp64).
 *  - Greedy verification (p5 "Risks", third bullet: under greedy decoding
 *    every committed token is the target model's own choice; p4 "结果与验证":
 *    token-by-token check): per position the lowest index of the row maximum,
 *    then the longest prefix of draft tokens that agree, then the target's
 *    token at the first disagreement.
 *
 * Build: gcc -O2 -std=c11 -shared -fPIC (oracle/build.py).  Single thread.
 */
#include <stdint.h>
#include <stddef.h>
#include <string.h>
#include <stdlib.h>
#include <math.h>

/* Status codes.  The numbering is the one the W12 C interface documents, so a
 * test can compare the two sides' rejections of the same bad input. */
#define W12REF_OK 0
#define W12REF_ERR_ARG 1
#define W12REF_ERR_SHAPE 2
#define W12REF_ERR_BLOB 5
#define W12REF_ERR_TOO_MANY_ESCAPES 6

/* Input orientation of the weight matrix handed to the encoder. */
#define W12REF_LAYOUT_KN 0 /* w[k*N + n] : row-major [K][N]               */
#define W12REF_LAYOUT_NK 1 /* w[n*K + k] : row-major [N][K] (out x in)    */

#define W12REF_GROUP 128   /* weights per group, along k                  */
#define W12REF_WINDOW 15   /* exponent offsets 0..14 are coded directly   */
#define W12REF_ESC_CODE 15 /* code meaning "exponent is in the side list" */
#define W12REF_MAX_BASE 240 /* largest base: 240 + 15 = 255 fits a byte      */
#define W12REF_MAX_ESC (1u << 24)

typedef struct {
    uint32_t version;
    uint32_t reserved;
    int64_t K, N, G;
    uint64_t tiles, unit_bytes, n_units, off_units, off_esc;
    uint64_t n_esc;
    uint64_t total_bytes;
} w12ref_desc;

#define W12REF_VERSION 2
#define W12REF_TILE 128          /* columns per tile                         */
#define W12REF_PLANE_BYTES 8192  /* one plane of a unit: 128 columns x 64 B  */
#define W12REF_META_AT 24576     /* meta words of a unit: 3 plane blocks in  */
#define W12REF_UNIT_BYTES 25104  /* 3 planes + 129 meta words + 12 zero bytes */

/* ---------------------------------------------------------------------- */
/* BF16 fields                                                             */
/* ---------------------------------------------------------------------- */

static unsigned bf16_sign(uint16_t v) { return (v >> 15) & 1u; }
static unsigned bf16_exp(uint16_t v) { return (v >> 7) & 0xFFu; }
static unsigned bf16_man(uint16_t v) { return v & 0x7Fu; }

static double bf16_to_double(uint16_t v)
{
    uint32_t u = (uint32_t)v << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

static uint16_t weight_at(const uint16_t *w, int64_t K, int64_t N, int layout, int64_t k, int64_t n)
{
    return layout == W12REF_LAYOUT_KN ? w[k * N + n] : w[n * K + k];
}

/* ---------------------------------------------------------------------- */
/* Logical codec: base, codes, escapes                                      */
/* ---------------------------------------------------------------------- */

/* Base of one group of 128 exponents: the b in [0, 240] whose window
 * [b, b+14] holds the most exponents; among equally good b, the largest. */
int w12ref_group_base(const uint16_t *vals)
{
    int best_b = 0, best_cover = -1;
    for (int b = 0; b <= W12REF_MAX_BASE; ++b) {
        int cover = 0;
        for (int i = 0; i < W12REF_GROUP; ++i) {
            int e = (int)bf16_exp(vals[i]);
            if (e >= b && e <= b + W12REF_WINDOW - 1)
                ++cover;
        }
        if (cover >= best_cover) { /* ">=": a later (larger) b wins a tie */
            best_cover = cover;
            best_b = b;
        }
    }
    return best_b;
}

/* Code of one exponent under base b: the offset, or 15 for an escape. */
static unsigned exp_code(unsigned e, unsigned b)
{
    if (e >= b && e <= b + W12REF_WINDOW - 1)
        return e - b;
    return W12REF_ESC_CODE;
}

static void gather_group(const uint16_t *w, int64_t K, int64_t N, int layout, int64_t g,
                         uint16_t *out)
{
    int64_t kg_per_col = K / W12REF_GROUP;
    int64_t n = g / kg_per_col, kg = g % kg_per_col;
    for (int p = 0; p < W12REF_GROUP; ++p)
        out[p] = weight_at(w, K, N, layout, kg * W12REF_GROUP + p, n);
}

/* ---------------------------------------------------------------------- */
/* Physical layout v2                                                      */
/* ---------------------------------------------------------------------- */
/*
 * Columns are cut into tiles of 128 and k into groups of 128.  Unit
 * u = t * KG + kg (tile t, group kg) is one block of W12REF_UNIT_BYTES:
 * the H, L and E planes (8192 bytes each), then 129 meta words, then 12
 * zero bytes.  The blob is the U unit blocks followed (at the next 256-byte
 * boundary) by the escape list.
 *
 * In a plane block, column c of the tile owns 64 bytes at 64 c: four
 * 16-byte chunks, logical chunk j (pos 32 j .. 32 j + 31) stored at chunk
 * position j ^ ((c >> 1) & 3).  A chunk is four little-endian 32-bit words;
 * the word covering pos p0 .. p0 + 7 (p0 a multiple of 8) holds in nibble q
 * (bits 4q .. 4q+3) the nibble of pos p0 + PERM[q], one permutation per
 * plane.
 *
 * Weights pair up as (k0, k0+1), (k0+2, k0+3), ...  The two mantissa planes
 * together hold, for weight j, the byte SM'(j) = m(j) << 1 | s(j ^ 1): its
 * 7-bit mantissa shifted up one place and the SIGN OF ITS PAIR PARTNER in
 * bit 0.  H holds the high nibble of SM'(j), L the low nibble.  E holds the
 * exponent code.
 *
 * Meta word c (c < 128) of unit u = base | (index of column c's first
 * escape in unit u) << 8; word 128 = (index of the first escape of unit
 * u + 1) << 8, i.e. n_esc << 8 after the last unit.  Escapes are listed by
 * unit, then column, then pos.  Padding columns (past N) have base 0, no
 * escapes and zero plane bytes.
 */
static const int PERM_H[8] = {4, 0, 5, 1, 6, 2, 7, 3};
static const int PERM_L[8] = {0, 5, 1, 6, 2, 7, 3, 4};
static const int PERM_E[8] = {0, 4, 1, 5, 2, 6, 3, 7};

static int slot_of(const int *perm, int r)
{
    for (int q = 0; q < 8; ++q)
        if (perm[q] == r)
            return q;
    return -1; /* unreachable: each table is a permutation of 0..7 */
}

/* Byte (from the blob start) and nibble shift of weight (k, n) in plane
 * `plane` (0 = H, 1 = L, 2 = E). */
static uint64_t nibble_byte(int64_t K, int64_t k, int64_t n, int plane, const int *perm, int *shift)
{
    int64_t KG = K / W12REF_GROUP;
    int64_t t = n / W12REF_TILE, c = n % W12REF_TILE;
    int64_t kg = k / W12REF_GROUP, pos = k % W12REF_GROUP;
    int64_t u = t * KG + kg;
    int64_t j = pos / 32;                 /* logical chunk */
    int64_t word = (pos % 32) / 8;        /* word within the chunk */
    int q = slot_of(perm, (int)(pos % 8));
    int64_t chunk_at = j ^ ((c >> 1) & 3);
    *shift = (q % 2) * 4; /* even slots are the low nibble of their byte */
    return (uint64_t)u * W12REF_UNIT_BYTES + (uint64_t)plane * W12REF_PLANE_BYTES + (uint64_t)c * 64u +
           (uint64_t)chunk_at * 16u + (uint64_t)word * 4u + (uint64_t)(q / 2);
}

static void put_nibble(uint8_t *blob, int64_t K, int64_t k, int64_t n, int plane, const int *perm,
                       unsigned v)
{
    int sh;
    uint64_t at = nibble_byte(K, k, n, plane, perm, &sh);
    blob[at] = (uint8_t)((blob[at] & ~(0xFu << sh)) | ((v & 0xFu) << sh));
}

static unsigned get_nibble(const uint8_t *blob, int64_t K, int64_t k, int64_t n, int plane,
                           const int *perm)
{
    int sh;
    uint64_t at = nibble_byte(K, k, n, plane, perm, &sh);
    return (blob[at] >> sh) & 0xFu;
}

/* Meta word `word` (0..128) of unit u, little-endian. */
static uint64_t meta_byte(int64_t u, int word)
{
    return (uint64_t)u * W12REF_UNIT_BYTES + W12REF_META_AT + 4u * (uint64_t)word;
}

static void put_u32(uint8_t *p, uint32_t v)
{
    p[0] = (uint8_t)v;
    p[1] = (uint8_t)(v >> 8);
    p[2] = (uint8_t)(v >> 16);
    p[3] = (uint8_t)(v >> 24);
}

static uint32_t get_u32(const uint8_t *p)
{
    return (uint32_t)p[0] | (uint32_t)p[1] << 8 | (uint32_t)p[2] << 16 | (uint32_t)p[3] << 24;
}

static uint64_t round256(uint64_t x) { return (x + 255u) & ~(uint64_t)255u; }

static void fill_offsets(w12ref_desc *d, int64_t K, int64_t N, uint64_t n_esc)
{
    d->version = W12REF_VERSION;
    d->reserved = 0;
    d->K = K;
    d->N = N;
    d->G = N * (K / W12REF_GROUP);
    d->tiles = (uint64_t)((N + W12REF_TILE - 1) / W12REF_TILE);
    d->unit_bytes = W12REF_UNIT_BYTES;
    d->n_units = d->tiles * (uint64_t)(K / W12REF_GROUP);
    d->off_units = 0;
    d->off_esc = round256(d->n_units * W12REF_UNIT_BYTES);
    d->n_esc = n_esc;
    d->total_bytes = round256(d->off_esc + 2u * n_esc);
}

static int check_shape(int64_t K, int64_t N, int layout)
{
    if (layout != W12REF_LAYOUT_KN && layout != W12REF_LAYOUT_NK)
        return W12REF_ERR_ARG;
    if (K < 0 || N < 0 || K % W12REF_GROUP != 0)
        return W12REF_ERR_SHAPE;
    return W12REF_OK;
}

/* Size the blob: counts the escapes, fills every offset. */
int w12ref_plan(const uint16_t *w, int64_t K, int64_t N, int layout, w12ref_desc *d)
{
    int st = check_shape(K, N, layout);
    if (st != W12REF_OK)
        return st;
    if (!d || (!w && K * N > 0))
        return W12REF_ERR_ARG;
    int64_t G = N * (K / W12REF_GROUP);
    uint64_t n_esc = 0;
    uint16_t grp[W12REF_GROUP];
    for (int64_t g = 0; g < G; ++g) {
        gather_group(w, K, N, layout, g, grp);
        unsigned b = (unsigned)w12ref_group_base(grp);
        for (int p = 0; p < W12REF_GROUP; ++p)
            if (exp_code(bf16_exp(grp[p]), b) == W12REF_ESC_CODE)
                ++n_esc;
    }
    if (n_esc >= W12REF_MAX_ESC)
        return W12REF_ERR_TOO_MANY_ESCAPES;
    fill_offsets(d, K, N, n_esc);
    return W12REF_OK;
}

/* Encode into a host blob of d->total_bytes (every byte is written). */
int w12ref_encode(const uint16_t *w, int64_t K, int64_t N, int layout, const w12ref_desc *d,
                  uint8_t *blob)
{
    int st = check_shape(K, N, layout);
    if (st != W12REF_OK)
        return st;
    if (!d || !blob || d->K != K || d->N != N)
        return W12REF_ERR_ARG;
    memset(blob, 0, (size_t)d->total_bytes);
    uint8_t *esc = blob + d->off_esc;
    int64_t KG = K / W12REF_GROUP;
    uint64_t next = 0;
    uint16_t grp[W12REF_GROUP];
    /* units in order; in each unit the tile's 128 columns in order */
    for (int64_t u = 0; u < (int64_t)d->n_units; ++u) {
        int64_t t = u / KG, kg = u % KG;
        for (int c = 0; c < W12REF_TILE; ++c) {
            int64_t n = t * W12REF_TILE + c;
            if (n >= N) {
                put_u32(blob + meta_byte(u, c), (uint32_t)(next << 8)); /* padding: b = 0 */
                continue;
            }
            gather_group(w, K, N, layout, n * KG + kg, grp);
            unsigned b = (unsigned)w12ref_group_base(grp);
            put_u32(blob + meta_byte(u, c), (uint32_t)b | (uint32_t)(next << 8));
            for (int p = 0; p < W12REF_GROUP; ++p) {
                uint16_t v = grp[p];
                int64_t k = kg * W12REF_GROUP + p;
                unsigned e = bf16_exp(v), m = bf16_man(v);
                unsigned partner_sign = bf16_sign(grp[p ^ 1]); /* pairs never straddle a group */
                unsigned smp = (m << 1) | partner_sign;
                unsigned code = exp_code(e, b);
                put_nibble(blob, K, k, n, 0, PERM_H, smp >> 4);
                put_nibble(blob, K, k, n, 1, PERM_L, smp & 0xFu);
                put_nibble(blob, K, k, n, 2, PERM_E, code);
                if (code == W12REF_ESC_CODE) {
                    if (next >= d->n_esc)
                        return W12REF_ERR_ARG; /* desc does not belong to this w */
                    unsigned entry = (unsigned)p | (e << 7);
                    esc[2 * next] = (uint8_t)entry;
                    esc[2 * next + 1] = (uint8_t)(entry >> 8);
                    ++next;
                }
            }
        }
        /* word 128: where the next unit's escapes begin */
        put_u32(blob + meta_byte(u, W12REF_TILE), (uint32_t)(next << 8));
    }
    if (next != d->n_esc)
        return W12REF_ERR_ARG;
    return W12REF_OK;
}

/* One weight back from the blob: the logical decode rule, element by element. */
static int weight_from_blob(const w12ref_desc *d, const uint8_t *blob, int64_t k, int64_t n,
                            uint16_t *out)
{
    int64_t K = d->K, KG = K / W12REF_GROUP;
    int64_t u = (n / W12REF_TILE) * KG + k / W12REF_GROUP;
    int c = (int)(n % W12REF_TILE);
    unsigned pos = (unsigned)(k % W12REF_GROUP);
    const uint8_t *esc = blob + d->off_esc;
    unsigned h = get_nibble(blob, K, k, n, 0, PERM_H);
    unsigned l = get_nibble(blob, K, k, n, 1, PERM_L);
    /* the sign of weight k sits in bit 0 of its pair partner's L nibble */
    unsigned l_partner = get_nibble(blob, K, k ^ 1, n, 1, PERM_L);
    unsigned code = get_nibble(blob, K, k, n, 2, PERM_E);
    uint32_t m0 = get_u32(blob + meta_byte(u, c)), m1 = get_u32(blob + meta_byte(u, c + 1));
    unsigned b = m0 & 0xFFu;
    unsigned e;
    if (code != W12REF_ESC_CODE) {
        e = b + code;
    } else {
        uint64_t lo = m0 >> 8, hi = m1 >> 8;
        if (lo > hi || hi > d->n_esc)
            return W12REF_ERR_BLOB;
        int found = 0;
        e = 0;
        for (uint64_t i = lo; i < hi; ++i) {
            unsigned entry = (unsigned)esc[2 * i] | (unsigned)esc[2 * i + 1] << 8;
            if ((entry & 0x7Fu) == pos) {
                e = (entry >> 7) & 0xFFu;
                found = 1;
                break;
            }
        }
        if (!found)
            return W12REF_ERR_BLOB;
    }
    if (e > 255u)
        return W12REF_ERR_BLOB;
    unsigned smp = (h << 4) | l;          /* m << 1 | sign of the partner */
    unsigned m = smp >> 1, s = l_partner & 1u;
    *out = (uint16_t)((s << 15) | (e << 7) | m);
    return W12REF_OK;
}

static int check_desc(const w12ref_desc *d)
{
    if (!d || d->version != W12REF_VERSION || d->K < 0 || d->N < 0 || d->K % W12REF_GROUP != 0)
        return W12REF_ERR_ARG;
    w12ref_desc want;
    fill_offsets(&want, d->K, d->N, d->n_esc);
    if (d->G != want.G || d->tiles != want.tiles || d->unit_bytes != want.unit_bytes ||
        d->n_units != want.n_units || d->off_units != want.off_units || d->off_esc != want.off_esc ||
        d->total_bytes != want.total_bytes)
        return W12REF_ERR_BLOB;
    return W12REF_OK;
}

/* Decode the whole matrix into w (layout KN or NK). */
int w12ref_decode(const w12ref_desc *d, const uint8_t *blob, uint16_t *w, int layout)
{
    int st = check_desc(d);
    if (st != W12REF_OK)
        return st;
    if (layout != W12REF_LAYOUT_KN && layout != W12REF_LAYOUT_NK)
        return W12REF_ERR_ARG;
    for (int64_t n = 0; n < d->N; ++n)
        for (int64_t k = 0; k < d->K; ++k) {
            uint16_t v;
            st = weight_from_blob(d, blob, k, n, &v);
            if (st != W12REF_OK)
                return st;
            if (layout == W12REF_LAYOUT_KN)
                w[k * d->N + n] = v;
            else
                w[n * d->K + k] = v;
        }
    return W12REF_OK;
}

/* ---------------------------------------------------------------------- */
/* GEMM in fp64                                                            */
/* ---------------------------------------------------------------------- */

/* One output: y = sum_k x[m,k] * w[k,n] in k order, and s = sum_k |x w|. */
static int dot_one(const w12ref_desc *d, const uint8_t *blob, const uint16_t *x, int64_t m,
                   int64_t n, double *y, double *s)
{
    double acc = 0.0, mag = 0.0;
    for (int64_t k = 0; k < d->K; ++k) {
        uint16_t wv;
        int st = weight_from_blob(d, blob, k, n, &wv);
        if (st != W12REF_OK)
            return st;
        double p = bf16_to_double(x[m * d->K + k]) * bf16_to_double(wv);
        acc += p;
        mag += fabs(p);
    }
    *y = acc;
    *s = mag;
    return W12REF_OK;
}

/* Full product: x is [M][K] bf16, y and s are [M][N] fp64 (s may be NULL). */
int w12ref_gemm(const w12ref_desc *d, const uint8_t *blob, const uint16_t *x, int64_t M,
                double *y, double *s)
{
    int st = check_desc(d);
    if (st != W12REF_OK)
        return st;
    if (M < 0 || !y)
        return W12REF_ERR_ARG;
    for (int64_t m = 0; m < M; ++m)
        for (int64_t n = 0; n < d->N; ++n) {
            double yy, ss;
            st = dot_one(d, blob, x, m, n, &yy, &ss);
            if (st != W12REF_OK)
                return st;
            y[m * d->N + n] = yy;
            if (s)
                s[m * d->N + n] = ss;
        }
    return W12REF_OK;
}

/* Selected outputs (ms[i], ns[i]) only, for full-size shapes. */
int w12ref_gemm_at(const w12ref_desc *d, const uint8_t *blob, const uint16_t *x, int64_t M,
                   int64_t count, const int64_t *ms, const int64_t *ns, double *y, double *s)
{
    int st = check_desc(d);
    if (st != W12REF_OK)
        return st;
    for (int64_t i = 0; i < count; ++i) {
        if (ms[i] < 0 || ms[i] >= M || ns[i] < 0 || ns[i] >= d->N)
            return W12REF_ERR_ARG;
        double ss;
        st = dot_one(d, blob, x, ms[i], ns[i], &y[i], &ss);
        if (st != W12REF_OK)
            return st;
        if (s)
            s[i] = ss;
    }
    return W12REF_OK;
}

/* ---------------------------------------------------------------------- */
/* Greedy verification                                                     */
/* ---------------------------------------------------------------------- */

#define W12REF_F32 0
#define W12REF_BF16 1

static double logit_at(const void *logits, int dtype, int64_t i)
{
    if (dtype == W12REF_F32)
        return (double)((const float *)logits)[i];
    return bf16_to_double(((const uint16_t *)logits)[i]);
}

/* Lowest index of the maximum of one row.  NaN ranks above every number and
 * the first NaN wins; -0 and +0 are equal (an ordinary comparison says so). */
static int64_t row_argmax(const void *logits, int dtype, int64_t row, int64_t V)
{
    int64_t best = 0;
    double bv = logit_at(logits, dtype, row * V);
    if (isnan(bv))
        return 0;
    for (int64_t i = 1; i < V; ++i) {
        double v = logit_at(logits, dtype, row * V + i);
        if (isnan(v))
            return i;
        if (v > bv) {
            bv = v;
            best = i;
        }
    }
    return best;
}

int w12ref_argmax(const void *logits, int dtype, int64_t rows, int64_t V, int64_t *idx)
{
    if ((dtype != W12REF_F32 && dtype != W12REF_BF16) || rows < 0 || V < 1 || !idx)
        return W12REF_ERR_ARG;
    for (int64_t r = 0; r < rows; ++r)
        idx[r] = row_argmax(logits, dtype, r, V);
    return W12REF_OK;
}

/* logits: [R*T][V]; draft: [R][T-1]; row r*T+i is the target's prediction
 * after the block input [last committed token, d0 .. d(T-2)] position i,
 * so it is compared with draft token i.  accept_len = first i < T-1 where
 * they differ (T-1 if none); next = the target's token at that position. */
int w12ref_verify_greedy(const void *logits, int dtype, int64_t R, int64_t T, int64_t V,
                         const int32_t *draft, int32_t *accept_len, int32_t *next)
{
    if ((dtype != W12REF_F32 && dtype != W12REF_BF16) || R < 0 || T < 1 || V < 1)
        return W12REF_ERR_SHAPE;
    if (!accept_len || !next || (R > 0 && !logits) || (R > 0 && T > 1 && !draft))
        return W12REF_ERR_ARG;
    for (int64_t r = 0; r < R; ++r) {
        int64_t L = T - 1;
        for (int64_t i = 0; i < T - 1; ++i) {
            int64_t g = row_argmax(logits, dtype, r * T + i, V);
            if ((int64_t)draft[r * (T - 1) + i] != g) {
                L = i;
                break;
            }
        }
        accept_len[r] = (int32_t)L;
        next[r] = (int32_t)row_argmax(logits, dtype, r * T + L, V);
    }
    return W12REF_OK;
}
