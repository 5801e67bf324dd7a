// w12_internal.h -- declarations shared by the library's own translation units.
// Not installed; the public interface is include/w12.h.
#pragma once

#include <cstddef>
#include <cstdint>

#include "../../include/w12.h"

namespace w12 {

constexpr int kGroup = 128;        // weights per group along k
constexpr int kMaxBase = 240;      // 240 + 15 = 255: b + code never leaves a byte
constexpr uint32_t kMaxEscapes = 1u << 24;

inline uint64_t round256(uint64_t x) { return (x + 255u) & ~uint64_t(255); }

// Offsets and sizes of format v1 for K x N with n_esc escapes.
void layout_v1(int64_t K, int64_t N, uint64_t n_esc, w12_desc *d);

// Workspace layout shared by the device calls: word 0 is the sticky error
// code, counters start at byte 256, the fp32 partials after them.
constexpr size_t kWsHeader = 256;

// Batched GEMV: up to kMaxBatch independent GEMMs with the same M in one
// launch; stream-K runs over the concatenation of their units.
constexpr int kMaxBatch = W12_MAX_BATCH;
struct GemvOne {
    const uint32_t *H, *L, *E, *meta;
    const uint16_t *esc;
    uint32_t n_esc;
    // 32-bit on purpose: the kernel's index arithmetic stays 32-bit (the
    // planner guarantees K*N/8, G and the unit counts stay below 2^31)
    int32_t K, N, KW, KG;
    int32_t steps, NB, ubase;  // units per column tile, column tiles, first unit of this GEMM
    const uint16_t *x;         // [M][K]
    void *y;                   // [M][N]
    float *partial;            // [NB * steps][M][cols] stream-K partial slots
    uint32_t *counters;        // [NB]
};
struct GemvBatch {
    GemvOne g[kMaxBatch];
    int count, M, y_dtype;
    int *err;
    int32_t U;       // total units
};
int launch_gemv_batch(const GemvBatch &b, int variant, int grid, void *stream);
constexpr int kMmaCols = 128;  // columns per tile of the tensor-core kernels

// Launchers (return W12_OK or W12_ERR_CUDA).
int launch_decode(const w12_desc *d, const void *blob, uint16_t *w, int layout, int *err,
                  void *stream);
int gemv_occupancy(int variant, int *blocks_per_sm);
int gemv_cols_per_tile();
int gemv_stage_k();
int device_sm_count(int *sms);

struct VerifyArgs {
    const void *logits;
    int dtype;
    int64_t R, T, V, rows;
    const int32_t *draft;
    int32_t *accept_len, *next_tok;
    unsigned long long *partial;  // [rows][splits] keys
    uint32_t *counter;
    int32_t *gbuf;                // [rows] greedy tokens (scratch)
    int64_t splits;
    int64_t chunk;                // columns per split
};
int launch_verify(const VerifyArgs &a, int grid, void *stream);

}  // namespace w12
