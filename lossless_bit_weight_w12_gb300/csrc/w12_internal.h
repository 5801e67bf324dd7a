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

// Format v2 geometry: tiles of 128 columns; a unit block holds the H, L, E
// planes of one 128-k group of a tile (8192 bytes each; column c's 64-byte
// row at 64 c, its 16-byte chunk j at chunk position j ^ ((c >> 1) & 3)),
// then 129 meta words at kMetaAt, then zero padding.
constexpr int kTileCols = 128;
constexpr int kPlaneBlock = 8192;
constexpr int kMetaAt = 3 * kPlaneBlock;
constexpr int kUnitBytes = W12_UNIT_BYTES;
static_assert(kUnitBytes == kMetaAt + 4 * (kTileCols + 1) + 12, "unit block layout");
static_assert(kUnitBytes % 16 == 0, "unit blocks must stay 16-byte aligned");

// Offsets and sizes of format v2 for K x N with n_esc escapes.
void layout_v2(int64_t K, int64_t N, uint64_t n_esc, w12_desc *d);

// Workspace layout shared by the device calls: word 0 is the sticky error
// code, counters start at byte 256, the fp32 partials after them.
constexpr size_t kWsHeader = 256;

constexpr int kMaxBatch = W12_MAX_BATCH;
constexpr int kMmaCols = 128;  // columns per tile of the tensor-core kernels

// Launchers (return W12_OK or W12_ERR_CUDA).
int launch_decode(const w12_desc *d, const void *blob, uint16_t *w, int layout, int *err,
                  void *stream);
int device_sm_count(int *sms);

// Device encoder (kernels_encode.cu): workspace bytes; steps 1-2 (bases,
// escape counts and their exclusive scan; *total_dev = escape count);
// step 3 (pack into a blob of d's layout).
size_t encode_device_ws(int64_t K, int64_t N);
int launch_encode_scan(const uint16_t *w, int64_t K, int64_t N, int layout, void *ws, void *stream,
                       uint32_t **total_dev);
int launch_encode_pack(const uint16_t *w, const w12_desc *d, int layout, void *blob, void *ws, void *stream);

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

// The greedy verify kernel's work split for `rows` rows of V logits (grid,
// slices per row, logits per slice; W12_ERR_CUDA if the device query
// fails), the scratch bytes it needs, and the scratch layout (counter,
// per-slice keys, per-row tokens) inside a buffer of that size.  Shared by
// w12_verify_greedy and w12_verify_greedy_noalloc.
int verify_plan(int64_t rows, int64_t V, int *grid, int64_t *splits, int64_t *chunk);
size_t verify_ws(int64_t rows, int64_t splits);
void verify_layout(void *ws, int64_t rows, int64_t splits, VerifyArgs *a);

}  // namespace w12
