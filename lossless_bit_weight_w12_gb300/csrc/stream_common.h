// stream_common.h -- argument block of the TMA-fed stream-K decode-GEMM
// (kernels_stream.cu).  Included by CUDA translation units only (it needs
// cuda.h for CUtensorMap).
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>

#include <cstddef>
#include <cstdint>

#include "w12_internal.h"

namespace w12 {

// One product y = x . W of a batch.  The weights are the blob's unit blocks
// (format v2: unit nb * KG + kg holds group kg of the 128 columns of tile
// nb, kUnitBytes each, streamed with one bulk copy).  The tensor map
// describes x for the Tensor Memory Accelerator: for the mma.sync kernel a
// 3-D array [M tokens][K/64][64] bf16 (box 64 x 2 x MP: one group for every
// token), for the tcgen05 kernel a 2-D array [M][K] (box 64 k x MP); rows
// past M read as zeros, 128-byte swizzle.
struct StreamOne {
    CUtensorMap tx;
    const uint8_t *units;  // unit blocks
    const uint16_t *esc;   // n_esc entries
    void *y;               // [M][N]
    uint32_t *counters;    // [NB] stream-K arrival counters (zero between calls)
    uint32_t n_esc;
    int32_t K, N, KG, NB;  // KG = K / 128 groups per column, NB = column tiles
    int32_t ubase;         // first unit of this product
};

// A batch: units are (product, 128-column tile, 128-k group), concatenated
// in that order; CTA c takes a balanced contiguous range of them.
struct StreamBatch {
    StreamOne g[kMaxBatch];
    float *partial;  // [grid][2][M][128] partial sums of split tiles
    int *err;        // workspace word 0
    int count, M, y_dtype;
    int32_t U;       // total units
    // Fused greedy verify (lm_head; count == 1, y = the optional fp32
    // logits copy or NULL): per-CTA best (value, index) keys of each row, a
    // CTA arrival counter, and the acceptance rule's inputs and outputs.
    unsigned long long *row_best;  // [grid][M]
    uint32_t *done;                // zero between calls
    const int32_t *draft;          // [vR][vT - 1]
    int32_t *accept_len, *next_tok, *gbuf;
    int vR, vT;
    // Launch options.  early_weights: the producers request the first ring's
    // worth of weight unit blocks before griddepcontrol.wait (the blob must
    // not be written by the kernel launched just before; W12_OPT_EARLY_WEIGHTS).
    // wait_ns: the limit of one bounded wait (0: kWaitLimitNs).  withhold_unit:
    // a test hook (w12_gemm_batched_debug), -1 normally; the unit whose weight
    // copy the producer never issues, so that a wait on it runs out.
    int early_weights;
    int32_t withhold_unit;
    uint64_t wait_ns;
};

// Kernel variants: v = 2 * log2(NT) + (ctas_per_sm - 1), NT = ceil(M / 8)
// rounded up to a power of two (1..16); two CTAs per SM for NT <= 4.
int stream_occupancy(int v, int *blocks_per_sm);
// Fills the tensor map of x in g, for the mma.sync kernel (tc = false: one
// 3-D box per group) or the tcgen05 kernel (tc = true: 2-D boxes of 64 k x
// MP tokens).  Returns W12_ERR_CUDA if the driver's tensor-map encoder is
// unavailable or rejects the map.
int stream_make_maps(StreamOne &g, const w12_desc &d, const uint16_t *x, int M, int MP, bool tc);
int launch_stream_batch(const StreamBatch &b, int variant, int grid, void *stream);
// The CUDA-core GEMV consumers on the same stream (variant v = log2(MT),
// M <= MT = 1, 2, 4).
int stream_gemv_occupancy(int v, int *blocks_per_sm);
int launch_stream_gemv(const StreamBatch &b, int variant, int grid, void *stream);
// The fused lm_head + greedy verify variants (same v).
int stream_fused_occupancy(int v, int *blocks_per_sm);
int launch_stream_fused(const StreamBatch &b, int variant, int grid, void *stream);
// The tcgen05 kernel (kernels_tc.cu) over the same batch and units; variant
// v: MP = 16 << v tokens.
int launch_tc_batch(const StreamBatch &b, int variant, int grid, void *stream);
int tc_occupancy(int variant, int *blocks_per_sm);
int launch_tc_fused(const StreamBatch &b, int variant, int grid, void *stream);
int tc_fused_occupancy(int variant, int *blocks_per_sm);

#ifdef __CUDACC__
// Launch a stream kernel with programmatic stream serialization: it may
// begin (and stream its first weights) while the previous kernel of the
// stream finishes; the kernel itself waits for that kernel (griddepcontrol)
// before it reads x or writes outputs.
template <class Kernel>
int launch_pdl(Kernel kernel, int grid, int threads, size_t smem, cudaStream_t s, const StreamBatch &b) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(unsigned(grid));
    cfg.blockDim = dim3(unsigned(threads));
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kernel, b) == cudaSuccess ? W12_OK : W12_ERR_CUDA;
}
#endif

}  // namespace w12
