// abi.cu -- the extern "C" entry points of libw12.so (declared in include/w12.h):
// argument checks, work planning and dispatch to the kernels.  Host code only.
#include <cuda_runtime.h>

#include <algorithm>
#include <cstring>
#include <map>
#include <mutex>
#include <utility>

#include "stream_common.h"
#include "w12_internal.h"

namespace w12 {

namespace {

bool aligned(const void *p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0; }

int64_t ceil_div(int64_t a, int64_t b) { return (a + b - 1) / b; }

// The descriptor must be exactly what the v1 layout gives for its K, N, n_esc.
int check_desc(const w12_desc *d) {
    if (!d) return W12_ERR_ARG;
    if (d->version != W12_FORMAT_VERSION || d->K < 0 || d->N < 0 || d->K % kGroup != 0)
        return W12_ERR_ARG;
    if (d->n_esc >= kMaxEscapes) return W12_ERR_BLOB;
    w12_desc want;
    layout_v2(d->K, d->N, d->n_esc, &want);
    if (std::memcmp(&want, d, sizeof want) != 0) return W12_ERR_BLOB;
    if (d->N >= (int64_t(1) << 31)) return W12_ERR_SHAPE;
    return W12_OK;
}

struct Device {
    int id = 0;
    int sms = 0;
};

// Per-device facts the planner needs on every call (SM count, occupancy of
// each kernel variant), queried once: the queries cost microseconds of host
// time, as much as a small GEMM takes on the device.
struct DeviceCache {
    int sms = 0;
    std::map<std::pair<int, size_t>, int> occ;  // (kernel key, smem) -> CTAs per SM
};
std::mutex g_cache_mu;
std::map<int, DeviceCache> g_cache;

int query_device(Device *dv) {
    if (cudaGetDevice(&dv->id) != cudaSuccess) return W12_ERR_CUDA;
    std::lock_guard<std::mutex> lock(g_cache_mu);
    DeviceCache &c = g_cache[dv->id];
    if (c.sms == 0 && device_sm_count(&c.sms) != W12_OK) return W12_ERR_CUDA;
    dv->sms = c.sms;
    return W12_OK;
}

// key: 32..47 tcgen05 variants with the fused lm_head verify, 48..63
// tcgen05 variants, 64..79 mma.sync stream variants, 80..95 the same with
// the fused lm_head verify, 96.. CUDA-core GEMV variants
int cached_occupancy(const Device &dv, int key, size_t smem, int *blocks) {
    {
        std::lock_guard<std::mutex> lock(g_cache_mu);
        auto &m = g_cache[dv.id].occ;
        auto it = m.find({key, smem});
        if (it != m.end()) {
            *blocks = it->second;
            return W12_OK;
        }
    }
    const int st = key < 48   ? tc_fused_occupancy(key - 32, blocks)
                   : key < 64 ? tc_occupancy(key - 48, blocks)
                   : key < 80 ? stream_occupancy(key - 64, blocks)
                   : key < 96 ? stream_fused_occupancy(key - 80, blocks)
                              : stream_gemv_occupancy(key - 96, blocks);
    if (st != W12_OK) return st;
    std::lock_guard<std::mutex> lock(g_cache_mu);
    g_cache[dv.id].occ[{key, smem}] = *blocks;
    return W12_OK;
}

// The batched kernels' index arithmetic is 32-bit.
bool gemv_fits_32bit(const w12_desc *d) {
    const int64_t lim = int64_t(1) << 31;
    return d->K < lim && d->N < lim && d->K / 8 * d->N < lim && d->G < lim;
}

// Workspace layout of a batch: header (error word), then per product its
// stream-K counters, then the partial sums (two slots per CTA).  Every path
// is the same weight stream (units of 128 columns x one 128-k group, one
// unit block of the blob each) with different consumers: CUDA-core GEMV
// (M <= 4), mma.sync, tcgen05.
struct BatchPlan {
    int path = W12_PATH_GEMV;
    int variant = 0, grid = 0;
    int64_t U = 0;
    size_t counters[kMaxBatch] = {}, partial[kMaxBatch] = {};
    int64_t steps[kMaxBatch] = {}, NB[kMaxBatch] = {}, ubase[kMaxBatch] = {};
    size_t stream_partial = 0;  // [grid][2][M][128] floats: a CTA's first and last tile pieces
    size_t total = 0;
};

// TMA-fed mma.sync kernel variant for M: NT = tokens padded to 8 .. 128 in
// powers of two; two CTAs per SM up to 32 tokens (measured faster on the
// 27B-class layer: 89 vs 104 us at M = 1, 97 vs 108 at 16, 110 vs 125 at
// 32), one CTA with the deepest ring beyond.
int stream_variant_for(int64_t M) {
    int l = 0;
    while ((8 << l) < M) ++l;
    return l <= 2 ? 2 * l + 1 : 2 * l;
}

int plan_batch(const w12_desc *d, int count, int64_t M, int path, BatchPlan *bp) {
    if (!d || count < 1 || count > kMaxBatch || M < 1 || M > W12_MAX_M) return W12_ERR_ARG;
    for (int i = 0; i < count; ++i) {
        const int st = check_desc(&d[i]);
        if (st != W12_OK) return st;
        if (!gemv_fits_32bit(&d[i])) return W12_ERR_SHAPE;
    }
    // Measured on the 27B-class layer (GB300, us per layer, GEMV / mma.sync
    // / tcgen05, early weight stream): M = 1: 78.9 / 79.0 / 77.7,
    // 4: 120.6 / 79.8 / 78.6, 8: - / 80.5 / 79.3, 16: - / 83.8 / 79.8,
    // 32: - / 95.6 / 81.2, 64: - / 151 / 86.0, 128: - / 231 / 100.0.  At
    // M = 1 the product is no dense contraction: the warp-shuffle GEMV
    // streams the weights on the CUDA cores (1.5 % behind tcgen05 on a
    // 16-token tile of which 15 rows would be padding); from 2 tokens on
    // tcgen05 is the fastest.
    if (path == W12_PATH_AUTO) path = M == 1 ? W12_PATH_GEMV : W12_PATH_TC;
    if (path == W12_PATH_GEMV && M > 4) return W12_ERR_SHAPE;
    if (path != W12_PATH_GEMV && path != W12_PATH_MMA && path != W12_PATH_TC) return W12_ERR_ARG;
    Device dv;
    if (query_device(&dv) != W12_OK) return W12_ERR_CUDA;
    bp->path = path;
    int64_t cpt, uk;
    int occ = 0;
    if (path == W12_PATH_TC) {
        int v = 0;
        while ((16 << v) < M) ++v;
        bp->variant = v;
        if (cached_occupancy(dv, 48 + v, 0, &occ) != W12_OK || occ < 1) return W12_ERR_CUDA;
        cpt = kMmaCols;
        uk = kGroup;
    } else if (path == W12_PATH_GEMV) {
        bp->variant = M <= 1 ? 0 : M <= 2 ? 1 : 2;
        if (cached_occupancy(dv, 96 + bp->variant, 0, &occ) != W12_OK || occ < 1) return W12_ERR_CUDA;
        cpt = kMmaCols;
        uk = kGroup;
    } else {
        bp->variant = stream_variant_for(M);
        if (cached_occupancy(dv, 64 + bp->variant, 0, &occ) != W12_OK || occ < 1) return W12_ERR_CUDA;
        cpt = kMmaCols;
        uk = kGroup;
    }
    size_t off = kWsHeader;
    for (int i = 0; i < count; ++i) {
        bp->steps[i] = ceil_div(d[i].K, uk);
        bp->NB[i] = ceil_div(d[i].N, cpt);
        bp->ubase[i] = bp->U;
        bp->U += bp->steps[i] * bp->NB[i];
        bp->counters[i] = off;
        off += round256(4u * uint64_t(std::max<int64_t>(bp->NB[i], 1)));
    }
    if (bp->U >= (int64_t(1) << 31)) return W12_ERR_SHAPE;
    bp->grid = int(std::min<int64_t>(int64_t(dv.sms) * occ, std::max<int64_t>(bp->U, 1)));
    bp->stream_partial = off;
    off += round256(uint64_t(bp->grid) * 2u * uint64_t(M) * uint64_t(cpt) * 4u);
    bp->total = off;
    return W12_OK;
}

// The TMA-fed mma.sync path: one tensor map per plane and one for x per product.
// Launch options of one call (defaults: weights read only after the
// previous kernel of the stream, no test hook, the default wait limit).
struct LaunchOpts {
    bool early_weights = false;
    int32_t withhold_unit = -1;
    uint64_t wait_ns = 0;
};

int fill_stream_batch(const w12_desc *d, const void *const *blobs, const uint16_t *const *xs, int64_t M,
                      void *const *ys, int y_dtype, int count, void *ws, const BatchPlan &bp,
                      const LaunchOpts &opt, StreamBatch *out) {
    uint8_t *w = static_cast<uint8_t *>(ws);
    StreamBatch &b = *out;
    b.early_weights = opt.early_weights ? 1 : 0;
    b.withhold_unit = opt.withhold_unit;
    b.wait_ns = opt.wait_ns;
    b.count = count;
    b.M = int(M);
    b.y_dtype = y_dtype;
    b.err = reinterpret_cast<int *>(w);
    b.U = int32_t(bp.U);
    b.partial = reinterpret_cast<float *>(w + bp.stream_partial);
    const bool tc = bp.path == W12_PATH_TC;
    const int MP = tc ? (16 << bp.variant) : bp.path == W12_PATH_GEMV ? 8 : (8 << (bp.variant / 2));
    for (int i = 0; i < count; ++i) {
        const uint8_t *bl = static_cast<const uint8_t *>(blobs[i]);
        StreamOne &g = b.g[i];
        const int st = stream_make_maps(g, d[i], xs[i], int(M), MP, tc);
        if (st != W12_OK) return st;
        g.units = bl + d[i].off_units;
        g.esc = reinterpret_cast<const uint16_t *>(bl + d[i].off_esc);
        g.y = ys[i];
        g.counters = reinterpret_cast<uint32_t *>(w + bp.counters[i]);
        g.n_esc = uint32_t(d[i].n_esc);
        g.K = int32_t(d[i].K);
        g.N = int32_t(d[i].N);
        g.KG = int32_t(d[i].K / kGroup);
        g.NB = int32_t(bp.NB[i]);
        g.ubase = int32_t(bp.ubase[i]);
    }
    return W12_OK;
}

int run_stream_batch(const w12_desc *d, const void *const *blobs, const uint16_t *const *xs, int64_t M,
                     void *const *ys, int y_dtype, int count, void *ws, const BatchPlan &bp,
                     const LaunchOpts &opt, void *stream) {
    StreamBatch b;
    std::memset(&b, 0, sizeof b);
    const int st = fill_stream_batch(d, blobs, xs, M, ys, y_dtype, count, ws, bp, opt, &b);
    if (st != W12_OK) return st;
    switch (bp.path) {
        case W12_PATH_TC: return launch_tc_batch(b, bp.variant, bp.grid, stream);
        case W12_PATH_GEMV: return launch_stream_gemv(b, bp.variant, bp.grid, stream);
    }
    return launch_stream_batch(b, bp.variant, bp.grid, stream);
}

// Launch a planned batch (all K_i, N_i > 0; pointers already checked).
int run_batch(const w12_desc *d, const void *const *blobs, const uint16_t *const *xs, int64_t M,
              void *const *ys, int y_dtype, int count, void *ws, const BatchPlan &bp, const LaunchOpts &opt,
              void *stream) {
    return run_stream_batch(d, blobs, xs, M, ys, y_dtype, count, ws, bp, opt, stream);
}

// Split the path argument of the _ex calls into the path and its options.
int split_path(int path_opts, int *path, LaunchOpts *opt) {
    if (path_opts & ~(W12_OPT_EARLY_WEIGHTS | 0xFF)) return W12_ERR_ARG;
    *path = path_opts & 0xFF;
    if (*path < W12_PATH_AUTO || *path > W12_PATH_TC) return W12_ERR_ARG;
    opt->early_weights = (path_opts & W12_OPT_EARLY_WEIGHTS) != 0;
    return W12_OK;
}

// Fused lm_head + verify: the stream-K plan of the one product, then the
// per-CTA argmax keys, the CTA arrival counter and the greedy tokens.
struct FusedPlan {
    BatchPlan bp;
    size_t off_best = 0, off_done = 0, off_gbuf = 0, total = 0;
};

int plan_fused(const w12_desc *d, int64_t M, FusedPlan *fp) {
    BatchPlan &bp = fp->bp;
    int st = plan_batch(d, 1, M, M == 1 ? W12_PATH_MMA : W12_PATH_TC, &bp);
    if (st != W12_OK) return st;
    Device dv;
    if (query_device(&dv) != W12_OK) return W12_ERR_CUDA;
    int occ = 0;
    const int key = bp.path == W12_PATH_TC ? 32 + bp.variant : 80 + bp.variant;
    if (cached_occupancy(dv, key, 0, &occ) != W12_OK || occ < 1) return W12_ERR_CUDA;
    bp.grid = int(std::min<int64_t>(int64_t(dv.sms) * occ, bp.U));
    size_t off = bp.stream_partial;
    off += round256(uint64_t(bp.grid) * 2u * uint64_t(M) * uint64_t(kMmaCols) * 4u);
    fp->off_best = off;
    off += round256(uint64_t(bp.grid) * uint64_t(M) * 8u);
    fp->off_done = off;
    off += 256;
    fp->off_gbuf = off;
    off += round256(uint64_t(M) * 4u);
    fp->total = off;
    return W12_OK;
}

}  // namespace

// Work split of the greedy verify kernel for `rows` rows of V logits: about
// four (row, slice) work items per SM, slices of `chunk` logits (a multiple
// of 8).  Shared by w12_verify_greedy and w12_verify_greedy_noalloc.
int verify_plan(int64_t rows, int64_t V, int *grid, int64_t *splits, int64_t *chunk) {
    Device dv;
    if (query_device(&dv) != W12_OK) return W12_ERR_CUDA;
    int64_t sp = std::max<int64_t>(1, ceil_div(4 * int64_t(dv.sms), rows));
    sp = std::min<int64_t>(sp, std::max<int64_t>(1, ceil_div(V, 1024)));
    int64_t ch = ceil_div(ceil_div(V, sp), 8) * 8;
    sp = ceil_div(V, ch);
    *splits = sp;
    *chunk = ch;
    *grid = int(std::min<int64_t>(rows * sp, int64_t(dv.sms) * 8));
    return W12_OK;
}

size_t verify_ws(int64_t rows, int64_t splits) {
    return kWsHeader + 256 + round256(uint64_t(rows * splits) * 8u) + round256(uint64_t(rows) * 4u);
}

void verify_layout(void *ws, int64_t rows, int64_t splits, VerifyArgs *a) {
    uint8_t *w = static_cast<uint8_t *>(ws);
    a->counter = reinterpret_cast<uint32_t *>(w + kWsHeader);
    a->partial = reinterpret_cast<unsigned long long *>(w + kWsHeader + 256);
    a->gbuf = reinterpret_cast<int32_t *>(w + kWsHeader + 256 + round256(uint64_t(rows * splits) * 8u));
}

}  // namespace w12

using namespace w12;

extern "C" const char *w12_status_string(int status) {
    switch (status) {
        case W12_OK: return "W12_OK";
        case W12_ERR_ARG: return "W12_ERR_ARG: bad argument";
        case W12_ERR_SHAPE: return "W12_ERR_SHAPE: unsupported shape";
        case W12_ERR_ALIGN: return "W12_ERR_ALIGN: pointer misaligned";
        case W12_ERR_WORKSPACE: return "W12_ERR_WORKSPACE: workspace missing or too small";
        case W12_ERR_BLOB: return "W12_ERR_BLOB: blob or descriptor inconsistent";
        case W12_ERR_TOO_MANY_ESCAPES: return "W12_ERR_TOO_MANY_ESCAPES: 2^24 or more escapes";
        case W12_ERR_CUDA: return "W12_ERR_CUDA: CUDA call failed";
        case W12_ERR_TIMEOUT: return "W12_ERR_TIMEOUT: bounded wait expired";
        case W12_ERR_DEVICE: return "W12_ERR_DEVICE: kernel detected a bad blob index";
    }
    return "unknown W12 status";
}

extern "C" int w12_version(void) { return W12_FORMAT_VERSION; }

extern "C" int w12_decode(const w12_desc *d, const void *blob, uint16_t *w, int layout, int *err,
                          void *stream) {
    int st = check_desc(d);
    if (st != W12_OK) return st;
    if (layout != W12_LAYOUT_KN && layout != W12_LAYOUT_NK) return W12_ERR_ARG;
    if (d->G == 0) return W12_OK;
    if (!blob || !w) return W12_ERR_ARG;
    if (!aligned(blob, 256) || !aligned(w, 16)) return W12_ERR_ALIGN;
    return launch_decode(d, blob, w, layout, err, stream);
}

extern "C" size_t w12_gemm_workspace_size(const w12_desc *d, int64_t M) {
    if (check_desc(d) != W12_OK || M < 1 || M > W12_MAX_M) return 0;
    // room for either path this M can take, so w12_gemm_ex can switch paths
    return w12_gemm_batched_workspace_size(d, 1, M);
}

extern "C" int w12_gemm_ex(const w12_desc *d, const void *blob, const uint16_t *x, int64_t M,
                           void *y, int y_dtype, void *ws, size_t ws_bytes, int path_opts,
                           void *stream) {
    int st = check_desc(d);
    if (st != W12_OK) return st;
    if (M < 1 || M > W12_MAX_M) return W12_ERR_SHAPE;
    if (y_dtype != W12_F32 && y_dtype != W12_BF16) return W12_ERR_ARG;
    int path;
    LaunchOpts opt;
    if (split_path(path_opts, &path, &opt) != W12_OK) return W12_ERR_ARG;
    if (d->N == 0) return W12_OK;
    if (!y) return W12_ERR_ARG;
    if (!aligned(y, y_dtype == W12_F32 ? 4 : 2)) return W12_ERR_ALIGN;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (d->K == 0) {
        const size_t bytes = size_t(M) * size_t(d->N) * (y_dtype == W12_F32 ? 4 : 2);
        return cudaMemsetAsync(y, 0, bytes, s) == cudaSuccess ? W12_OK : W12_ERR_CUDA;
    }
    if (!blob || !x) return W12_ERR_ARG;
    if (!aligned(blob, 256) || !aligned(x, 16)) return W12_ERR_ALIGN;
    BatchPlan bp;
    st = plan_batch(d, 1, M, path, &bp);
    if (st != W12_OK) return st;
    if (!ws || ws_bytes < bp.total) return W12_ERR_WORKSPACE;
    if (!aligned(ws, 256)) return W12_ERR_ALIGN;
    const void *blobs[1] = {blob};
    const uint16_t *xs[1] = {x};
    void *ys[1] = {y};
    return run_batch(d, blobs, xs, M, ys, y_dtype, 1, ws, bp, opt, stream);
}

extern "C" int w12_gemm(const w12_desc *d, const void *blob, const uint16_t *x, int64_t M, void *y,
                        int y_dtype, void *ws, size_t ws_bytes, void *stream) {
    return w12_gemm_ex(d, blob, x, M, y, y_dtype, ws, ws_bytes, W12_PATH_AUTO, stream);
}


extern "C" size_t w12_gemm_batched_workspace_size(const w12_desc *d, int count, int64_t M) {
    // room for every path this M can take, so the _ex call can switch paths
    size_t need = 0;
    for (int path = W12_PATH_GEMV; path <= W12_PATH_TC; ++path) {
        if (path == W12_PATH_GEMV && M > 4) continue;
        BatchPlan bp;
        if (plan_batch(d, count, M, path, &bp) == W12_OK) need = std::max(need, bp.total);
    }
    return need;
}

namespace {

int gemm_batched_opts(const w12_desc *d, const void *const *blobs, const uint16_t *const *xs, int64_t M,
                      void *const *ys, int y_dtype, int count, void *ws, size_t ws_bytes, int path,
                      const LaunchOpts &opt, void *stream) {
    if (!blobs || !xs || !ys) return W12_ERR_ARG;
    if (y_dtype != W12_F32 && y_dtype != W12_BF16) return W12_ERR_ARG;
    BatchPlan bp;
    int st = plan_batch(d, count, M, path, &bp);
    if (st != W12_OK) return st;
    for (int i = 0; i < count; ++i) {
        if (d[i].N == 0 || d[i].K == 0) return W12_ERR_SHAPE;  // empty products: use w12_gemm
        if (!blobs[i] || !xs[i] || !ys[i]) return W12_ERR_ARG;
        if (!aligned(blobs[i], 256) || !aligned(xs[i], 16) || !aligned(ys[i], y_dtype == W12_F32 ? 4 : 2))
            return W12_ERR_ALIGN;
    }
    if (!ws || ws_bytes < bp.total) return W12_ERR_WORKSPACE;
    if (!aligned(ws, 256)) return W12_ERR_ALIGN;
    if (opt.withhold_unit >= bp.U) return W12_ERR_ARG;
    return run_batch(d, blobs, xs, M, ys, y_dtype, count, ws, bp, opt, stream);
}

}  // namespace

extern "C" int w12_gemm_batched_ex(const w12_desc *d, const void *const *blobs, const uint16_t *const *xs,
                                   int64_t M, void *const *ys, int y_dtype, int count, void *ws,
                                   size_t ws_bytes, int path_opts, void *stream) {
    int path;
    LaunchOpts opt;
    if (split_path(path_opts, &path, &opt) != W12_OK) return W12_ERR_ARG;
    return gemm_batched_opts(d, blobs, xs, M, ys, y_dtype, count, ws, ws_bytes, path, opt, stream);
}

extern "C" int w12_gemm_batched_debug(const w12_desc *d, const void *const *blobs, const uint16_t *const *xs,
                                      int64_t M, void *const *ys, int y_dtype, int count, void *ws,
                                      size_t ws_bytes, int path_opts, const w12_debug_opts *dbg, void *stream) {
    int path;
    LaunchOpts opt;
    if (!dbg || split_path(path_opts, &path, &opt) != W12_OK) return W12_ERR_ARG;
    if (dbg->withhold_unit < -1 || dbg->wait_limit_us > 10000000u) return W12_ERR_ARG;
    opt.withhold_unit = dbg->withhold_unit;
    opt.wait_ns = uint64_t(dbg->wait_limit_us) * 1000u;
    return gemm_batched_opts(d, blobs, xs, M, ys, y_dtype, count, ws, ws_bytes, path, opt, stream);
}

extern "C" int w12_gemm_batched(const w12_desc *d, const void *const *blobs, const uint16_t *const *xs,
                                int64_t M, void *const *ys, int y_dtype, int count, void *ws,
                                size_t ws_bytes, void *stream) {
    return w12_gemm_batched_ex(d, blobs, xs, M, ys, y_dtype, count, ws, ws_bytes, W12_PATH_AUTO, stream);
}

extern "C" size_t w12_verify_workspace_size(int64_t R, int64_t T, int64_t V) {
    if (R < 1 || T < 1 || V < 1 || V >= (int64_t(1) << 31)) return 0;
    int grid;
    int64_t splits, chunk;
    if (verify_plan(R * T, V, &grid, &splits, &chunk) != W12_OK) return 0;
    return verify_ws(R * T, splits);
}

extern "C" int w12_verify_greedy(const void *logits, int dtype, int64_t R, int64_t T, int64_t V,
                                 const int32_t *draft, int32_t *accept_len, int32_t *next_tok,
                                 void *ws, size_t ws_bytes, void *stream) {
    if (dtype != W12_F32 && dtype != W12_BF16) return W12_ERR_ARG;
    if (R < 1 || T < 1 || V < 1 || V >= (int64_t(1) << 31)) return W12_ERR_SHAPE;
    if (!logits || !accept_len || !next_tok || (T > 1 && !draft)) return W12_ERR_ARG;
    if (!aligned(logits, dtype == W12_F32 ? 4 : 2) || !aligned(accept_len, 4) ||
        !aligned(next_tok, 4) || (draft && !aligned(draft, 4)))
        return W12_ERR_ALIGN;
    VerifyArgs a;
    int grid;
    a.rows = R * T;
    if (verify_plan(a.rows, V, &grid, &a.splits, &a.chunk) != W12_OK) return W12_ERR_CUDA;
    if (!ws || ws_bytes < verify_ws(a.rows, a.splits)) return W12_ERR_WORKSPACE;
    if (!aligned(ws, 256)) return W12_ERR_ALIGN;
    a.logits = logits;
    a.dtype = dtype;
    a.R = R;
    a.T = T;
    a.V = V;
    a.draft = draft;
    a.accept_len = accept_len;
    a.next_tok = next_tok;
    verify_layout(ws, a.rows, a.splits, &a);
    return launch_verify(a, grid, stream);
}

extern "C" size_t w12_verify_lmhead_workspace_size(const w12_desc *d, int64_t R, int64_t T) {
    if (check_desc(d) != W12_OK || R < 1 || T < 1 || R * T > W12_MAX_M || d->N < 1 || d->K < kGroup) return 0;
    FusedPlan fp;
    if (plan_fused(d, R * T, &fp) != W12_OK) return 0;
    return fp.total;
}

extern "C" int w12_verify_greedy_lmhead(const uint16_t *hidden, const w12_desc *d,
                                        const void *blob, int64_t R, int64_t T,
                                        const int32_t *draft, int32_t *accept_len,
                                        int32_t *next_tok, float *logits_out, void *ws,
                                        size_t ws_bytes, void *stream) {
    int st = check_desc(d);
    if (st != W12_OK) return st;
    if (R < 1 || T < 1 || R * T > W12_MAX_M || d->N < 1 || d->K < kGroup) return W12_ERR_SHAPE;
    if (!gemv_fits_32bit(d)) return W12_ERR_SHAPE;
    if (!hidden || !blob || !accept_len || !next_tok || (T > 1 && !draft)) return W12_ERR_ARG;
    if (!aligned(blob, 256) || !aligned(hidden, 16) || !aligned(accept_len, 4) ||
        !aligned(next_tok, 4) || (draft && !aligned(draft, 4)) ||
        (logits_out && !aligned(logits_out, 4)))
        return W12_ERR_ALIGN;
    const int64_t M = R * T;
    FusedPlan fp;
    st = plan_fused(d, M, &fp);
    if (st != W12_OK) return st;
    if (!ws || ws_bytes < fp.total) return W12_ERR_WORKSPACE;
    if (!aligned(ws, 256)) return W12_ERR_ALIGN;
    uint8_t *w = static_cast<uint8_t *>(ws);
    StreamBatch b;
    std::memset(&b, 0, sizeof b);
    const void *blobs[1] = {blob};
    const uint16_t *xs[1] = {hidden};
    void *ys[1] = {logits_out};
    st = fill_stream_batch(d, blobs, xs, M, ys, W12_F32, 1, ws, fp.bp, LaunchOpts{}, &b);
    if (st != W12_OK) return st;
    b.row_best = reinterpret_cast<unsigned long long *>(w + fp.off_best);
    b.done = reinterpret_cast<uint32_t *>(w + fp.off_done);
    b.gbuf = reinterpret_cast<int32_t *>(w + fp.off_gbuf);
    b.draft = draft;
    b.accept_len = accept_len;
    b.next_tok = next_tok;
    b.vR = int(R);
    b.vT = int(T);
    return fp.bp.path == W12_PATH_TC ? launch_tc_fused(b, fp.bp.variant, fp.bp.grid, stream)
                                     : launch_stream_fused(b, fp.bp.variant, fp.bp.grid, stream);
}

extern "C" size_t w12_encode_device_workspace_size(int64_t K, int64_t N) {
    if (K < 0 || N < 0) return 0;
    return std::max<size_t>(256, encode_device_ws(K, N));
}

extern "C" int w12_encode_plan_device(const uint16_t *w, int64_t K, int64_t N, int layout, w12_desc *d,
                                      void *ws, size_t ws_bytes, void *stream) {
    if (layout != W12_LAYOUT_KN && layout != W12_LAYOUT_NK) return W12_ERR_ARG;
    if (K < 0 || N < 0 || K % kGroup != 0) return W12_ERR_SHAPE;
    if (!d) return W12_ERR_ARG;
    if (K == 0 || N == 0) {
        layout_v2(K, N, 0, d);
        return W12_OK;
    }
    if (!w || !ws) return W12_ERR_ARG;
    if (!aligned(w, 16) || !aligned(ws, 256)) return W12_ERR_ALIGN;
    if (ws_bytes < encode_device_ws(K, N)) return W12_ERR_WORKSPACE;
    // the escape counts are scanned in 32 bits: at most 2^24 (unit, column)
    // slots of 128 weights (2^31 weights) per call
    if (N >= (int64_t(1) << 31) || (N + kTileCols - 1) / kTileCols * (K / kGroup) * kTileCols >= (int64_t(1) << 24))
        return W12_ERR_SHAPE;
    uint32_t *total = nullptr;
    int st = launch_encode_scan(w, K, N, layout, ws, stream, &total);
    if (st != W12_OK) return st;
    uint32_t n_esc = 0;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (cudaMemcpyAsync(&n_esc, total, sizeof n_esc, cudaMemcpyDeviceToHost, s) != cudaSuccess ||
        cudaStreamSynchronize(s) != cudaSuccess)
        return W12_ERR_CUDA;
    if (n_esc >= kMaxEscapes) return W12_ERR_TOO_MANY_ESCAPES;
    layout_v2(K, N, n_esc, d);
    return W12_OK;
}

extern "C" int w12_encode_device(const uint16_t *w, int64_t K, int64_t N, int layout, const w12_desc *d,
                                 void *blob, void *ws, size_t ws_bytes, void *stream) {
    if (layout != W12_LAYOUT_KN && layout != W12_LAYOUT_NK) return W12_ERR_ARG;
    const int st = check_desc(d);
    if (st != W12_OK) return st;
    if (d->K != K || d->N != N) return W12_ERR_ARG;
    if (d->total_bytes == 0) return W12_OK;
    if (!w || !blob || !ws) return W12_ERR_ARG;
    if (!aligned(w, 16) || !aligned(blob, 256) || !aligned(ws, 256)) return W12_ERR_ALIGN;
    if (ws_bytes < encode_device_ws(K, N)) return W12_ERR_WORKSPACE;
    return launch_encode_pack(w, d, layout, blob, ws, stream);
}

extern "C" int w12_get_device_error(void *ws, int *err_host, void *stream) {
    if (!ws || !err_host) return W12_ERR_ARG;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    int v = 0;
    if (cudaMemcpyAsync(&v, ws, sizeof v, cudaMemcpyDeviceToHost, s) != cudaSuccess) return W12_ERR_CUDA;
    if (cudaMemsetAsync(ws, 0, sizeof v, s) != cudaSuccess) return W12_ERR_CUDA;
    if (cudaStreamSynchronize(s) != cudaSuccess) return W12_ERR_CUDA;
    *err_host = v;
    return W12_OK;
}
