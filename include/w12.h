/*
 * w12.h -- C interface of libw12.so: the W12 lossless 12-bit BF16 weight
 * format, the fused W12 decode-GEMM for skinny M, and greedy draft-block
 * verification, for NVIDIA GB300 (sm_103a).
 *
 * Sources.  The SpecPilot summary pages (airadar.tv, English edition,
 * "Reasons" bullet 2, and its French, Japanese and Korean editions) describe
 * W12 as BF16 split into three 4-bit planes and rebuilt bit for bit inside the
 * GEMM's registers; the hotrepo.ai page on StargazerX0/SpecPilot ("项目介绍",
 * paragraph 2) adds that the decode is bit-exact and serves batch 1-32.  The
 * same English page ("Risks", bullet 3) defines the greedy acceptance rule:
 * every committed token is the target model's own greedy choice.  No layout,
 * interface or kernel is printed there; the layout and calls below are this
 * library's own.
 *
 * Conventions for every call:
 *  - Status: every function returns an int status (W12_OK = 0 or a W12_ERR_*
 *    code); w12_status_string() names it.  A non-zero status means nothing
 *    was launched or written.
 *  - Memory: the caller owns every buffer.  The library allocates no device
 *    memory and no host memory beyond stack and OpenMP temporaries.
 *  - Streams: `stream` is a cudaStream_t passed as void* (NULL = the legacy
 *    default stream).  Device calls are asynchronous on that stream and never
 *    synchronise, except w12_get_device_error().
 *  - The GEMM and fused-verify kernels use programmatic dependent launch:
 *    they may start while the kernel launched just before them on the same
 *    stream is finishing, but by default they read nothing in global memory
 *    (blob, x, hidden, draft, workspace) before that kernel has completed,
 *    so any producer of their inputs is safe.  The GEMM calls take one
 *    option, W12_OPT_EARLY_WEIGHTS (OR-ed into the path argument of the
 *    _ex calls): the first weight copies then start before the wait, under
 *    the previous kernel's tail; the caller promises that the blob was not
 *    written by the kernel launched just before the call on the same stream
 *    (another launch, an event or a synchronisation in between suffices;
 *    w12_encode_device ends with such a launch; copies and memsets are not
 *    kernels and need nothing).
 *  - Pointers named *_dev are device pointers, *_host host pointers.
 *  - Workspaces: a workspace of the size the matching *_workspace_size()
 *    call returns, 256-byte aligned, zero-filled by the caller before its
 *    first use.  Every kernel leaves its workspace counters at zero again, so
 *    a workspace is reused without clearing.  Word 0 of a workspace is a
 *    sticky device error code (see w12_get_device_error).  Calls that share
 *    one workspace must be ordered (same stream, or events).
 */
#ifndef W12_H
#define W12_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define W12_FORMAT_VERSION 2

/* Status codes. */
#define W12_OK 0
#define W12_ERR_ARG 1               /* NULL pointer, bad enum, inconsistent desc   */
#define W12_ERR_SHAPE 2             /* K % 128 != 0, negative sizes, M or T range  */
#define W12_ERR_ALIGN 3             /* a pointer misses its required alignment     */
#define W12_ERR_WORKSPACE 4         /* workspace NULL or smaller than required     */
#define W12_ERR_BLOB 5              /* blob contents inconsistent with the desc    */
#define W12_ERR_TOO_MANY_ESCAPES 6  /* 2^24 or more escapes in one matrix          */
#define W12_ERR_CUDA 7              /* a CUDA runtime call or launch failed        */
#define W12_ERR_TIMEOUT 8           /* a bounded device wait gave up               */
#define W12_ERR_DEVICE 9            /* a kernel recorded an error (bad blob index) */

/* Orientation of a dense weight matrix in memory. */
#define W12_LAYOUT_KN 0 /* w[k*N + n]: row-major [K][N]                         */
#define W12_LAYOUT_NK 1 /* w[n*K + k]: row-major [N][K] (a linear layer's weight) */

/* Element types of y and of logits. */
#define W12_F32 0
#define W12_BF16 1

/* GEMM paths (w12_gemm_ex, w12_gemm_batched_ex).  All three stream the
 * weights' unit blocks with bulk copies (TMA) through a shared-memory ring,
 * stream-K over the whole GPU; they differ in the contraction.
 * W12_PATH_AUTO takes the GEMV at M = 1 and tcgen05 above (the fastest on
 * GB300 from 2 tokens on). */
#define W12_PATH_AUTO 0
#define W12_PATH_GEMV 1 /* CUDA-core bf16 FMA GEMV with warp-shuffle reduction, M <= 4   */
#define W12_PATH_MMA 2  /* mma.sync tiles, M <= 128                                     */
#define W12_PATH_TC 3   /* tcgen05: weights rebuilt into tensor memory, fp32 accumulator
                           in tensor memory, M <= 128                                    */

#define W12_MAX_M 128

/* Option bit of the path argument of w12_gemm_ex / w12_gemm_batched_ex:
 * start streaming the weights before the previous kernel of the stream has
 * completed (see the conventions above).  Default off. */
#define W12_OPT_EARLY_WEIGHTS 0x100

/*
 * Descriptor of one encoded K x N matrix (format v2).
 *
 * Logical format.  A group is 128 consecutive k of one output column n
 * (pos = k % 128).  A bf16 weight has sign s (bit 15), exponent e (bits
 * 14..7) and mantissa m (bits 6..0).  Each group has a base b in [0, 240]:
 * the b whose window [b, b+14] holds the most of the group's exponents, the
 * largest such b on a tie.  A weight's exponent code is c = e - b inside the
 * window and 15 ("escape") outside it; an escaped weight gets a 16-bit entry
 * pos | e << 7 in the escape list.  Weights k and k^1 (an even k and the
 * next) form a pair; each stores its pair partner's sign.
 *
 * Physical format: plane-major, 16-byte-aligned tiles.
 *  - Columns are cut into tiles of 128 (T = ceil(N / 128) tiles; columns
 *    past N are padding) and k into groups (KG = K / 128).  Unit
 *    u = t * KG + kg holds group kg of the 128 columns of tile t; the blob
 *    starts with the U = T * KG unit blocks, each W12_UNIT_BYTES long:
 *      [0, 8192)      H plane: nibble = SM'(k) >> 4
 *      [8192, 16384)  L plane: nibble = SM'(k) & 15
 *      [16384, 24576) E plane: nibble = c(k)
 *      [24576, 25092) meta: 129 little-endian uint32
 *      [25092, 25104) zero
 *    with SM'(k) = m(k) << 1 | s(k ^ 1).
 *  - In a plane block, column c of the tile owns the 64-byte row
 *    [64 c, 64 c + 64): four 16-byte chunks, chunk j holding pos
 *    32 j .. 32 j + 31 as four little-endian 32-bit words (word q: pos
 *    32 j + 8 q + 0..7).  Logical chunk j is stored at chunk position
 *    j ^ ((c >> 1) & 3).  Nibble p (bits 4p..4p+3) of a word covering pos
 *    p0..p0+7 holds the weight p0 + P[p]:
 *      H: P = {4,0,5,1,6,2,7,3}   L: P = {0,5,1,6,2,7,3,4}   E: P = {0,4,1,5,2,6,3,7}
 *  - Meta word c < 128 = b | first_escape_index(u, c) << 8; word 128 =
 *    first_escape_index(u + 1, 0) << 8 (n_esc << 8 for the last unit), so
 *    column c's escapes in unit u are entries [word c >> 8, word c+1 >> 8).
 *    Padding columns have b = 0 and no escapes; their plane bytes are 0.
 *  - The escape list (n_esc uint16 entries, ordered by unit, then column,
 *    then pos) starts at off_esc, the first 256-byte boundary after the
 *    units.  total_bytes = off_esc + 2 n_esc rounded up to 256.
 * Every unit is one contiguous, 16-byte-aligned block (the blob itself must
 * be 256-byte aligned on the device), so a kernel streams a unit with one
 * bulk copy.
 */
#define W12_UNIT_BYTES 25104
typedef struct w12_desc {
    uint32_t version;    /* W12_FORMAT_VERSION */
    uint32_t reserved;   /* 0 */
    int64_t K, N, G;     /* G = N * K / 128 groups of real columns */
    uint64_t tiles;      /* T = ceil(N / 128) */
    uint64_t unit_bytes; /* W12_UNIT_BYTES */
    uint64_t n_units;    /* U = T * K / 128 */
    uint64_t off_units;  /* 0 */
    uint64_t off_esc;
    uint64_t n_esc;
    uint64_t total_bytes;
} w12_desc;

/* Name of a status code (static string, never NULL). */
const char *w12_status_string(int status);

/* Library format version (W12_FORMAT_VERSION). */
int w12_version(void);

/* --------------------------------------------------------------------- */
/* Host encoder                                                          */
/* --------------------------------------------------------------------- */

/*
 * Defined by: the W12 format (SpecPilot summary, airadar.tv English edition,
 * "Reasons" bullet 2: BF16 split into three 4-bit planes; hotrepo.ai
 * StargazerX0/SpecPilot page, "项目介绍" paragraph 2: lossless, decoded
 * bit-exactly).  The group size, base rule, escape list and packing are this
 * library's reading (the format description above).
 *
 * Size the blob for a bf16 matrix w (host, layout W12_LAYOUT_KN or _NK,
 * K % 128 == 0; K or N may be 0).  Fills every field of *d, counting the
 * escapes.  Errors: W12_ERR_ARG, W12_ERR_SHAPE, W12_ERR_TOO_MANY_ESCAPES.
 * Multithreaded (OpenMP) over groups.
 */
int w12_encode_plan(const uint16_t *w_host, int64_t K, int64_t N, int layout, w12_desc *d);

/*
 * Defined by: as w12_encode_plan ("Reasons" bullet 2; "项目介绍" paragraph 2).
 *
 * Encode w into blob_host (d->total_bytes bytes, any alignment; padding is
 * written as zeros).  *d must come from w12_encode_plan on the same w.
 * Errors: W12_ERR_ARG (d does not match w), W12_ERR_SHAPE.
 */
int w12_encode(const uint16_t *w_host, int64_t K, int64_t N, int layout, const w12_desc *d,
               void *blob_host);

/*
 * Defined by: the format description above (this library's reading of
 * "Reasons" bullet 2).
 *
 * Check a host blob against its descriptor: the offsets and sizes, base
 * range, meta monotonicity and sentinel, escape positions and order, that
 * every code-15 nibble has exactly one escape entry and that every escape is
 * canonical (its exponent lies outside the group window).  Returns W12_OK,
 * W12_ERR_ARG or W12_ERR_BLOB.  The device calls do not run this check:
 * they only bound every index they read, recording W12_ERR_DEVICE.
 */
int w12_validate(const w12_desc *d, const void *blob_host);

/* --------------------------------------------------------------------- */
/* Device encoder (the same bytes as the host encoder)                  */
/* --------------------------------------------------------------------- */

/* Bytes of workspace w12_encode_plan_device / w12_encode_device need for a
 * K x N matrix (>= 256; 0 for a negative size). */
size_t w12_encode_device_workspace_size(int64_t K, int64_t N);

/*
 * Defined by: as w12_encode_plan ("Reasons" bullet 2; "项目介绍" paragraph 2).
 *
 * w12_encode_plan on the GPU, for weights already in device memory (a model
 * loaded straight to HBM: no pass over the weights on the host).  w_dev: the
 * bf16 matrix in layout W12_LAYOUT_KN or _NK, 16-byte aligned.  Computes
 * every group's base and escape count into the workspace, fills *d (the
 * descriptor w12_encode_plan gives for the same matrix) and waits for
 * `stream` (the escape count is read back to size the blob).  Keep the
 * workspace for w12_encode_device.  Up to 2^24 unit columns (ceil(N/128) *
 * K/128 * 128 <= 2^24, about 2^31 weights) per matrix.
 * Errors: W12_ERR_ARG, W12_ERR_SHAPE, W12_ERR_ALIGN, W12_ERR_WORKSPACE,
 * W12_ERR_TOO_MANY_ESCAPES, W12_ERR_CUDA.
 */
int w12_encode_plan_device(const uint16_t *w_dev, int64_t K, int64_t N, int layout, w12_desc *d,
                           void *ws_dev, size_t ws_bytes, void *stream);

/*
 * Defined by: as w12_encode ("Reasons" bullet 2; "项目介绍" paragraph 2).
 *
 * w12_encode on the GPU: writes the blob of *d (from w12_encode_plan_device
 * on the same w_dev, layout and workspace) into blob_dev (d->total_bytes,
 * 256-byte aligned), byte for byte what w12_encode writes.  Asynchronous on
 * `stream`.  Errors: W12_ERR_ARG (d does not match K, N), W12_ERR_ALIGN,
 * W12_ERR_WORKSPACE, W12_ERR_CUDA.
 */
int w12_encode_device(const uint16_t *w_dev, int64_t K, int64_t N, int layout, const w12_desc *d,
                      void *blob_dev, void *ws_dev, size_t ws_bytes, void *stream);

/* --------------------------------------------------------------------- */
/* Device calls                                                          */
/* --------------------------------------------------------------------- */

/*
 * Defined by: "项目介绍" paragraph 2 (W12 is decoded bit-exactly) and
 * "Reasons" bullet 2 (the three planes are rebuilt bit by bit).
 *
 * Decode a device blob (256-byte aligned) back to bf16 bit patterns in w_dev
 * (K*N uint16, 16-byte aligned) in the given layout.  Bit-exact inverse of
 * w12_encode.  Errors: W12_ERR_ARG, W12_ERR_ALIGN, W12_ERR_CUDA.  Escape
 * indices are bounds-checked; a bad one is not followed (the weight keeps
 * the garbage exponent) and W12_ERR_DEVICE goes to *err_dev if err_dev is
 * not NULL.
 */
int w12_decode(const w12_desc *d, const void *blob_dev, uint16_t *w_dev, int layout,
               int *err_dev, void *stream);

/* Bytes of workspace w12_gemm needs for this matrix and M (>= 256). */
size_t w12_gemm_workspace_size(const w12_desc *d, int64_t M);

/*
 * Defined by: "Reasons" bullet 2 (the planes are rebuilt bit by bit inside the
 * GEMM's registers) and "项目介绍" paragraph 2 (a bit-exact decode inside the
 * GEMM, batch 1-32); the first paragraph of the summary (a decode step reads
 * every weight) makes it a weight stream.
 *
 * y[m, n] = sum_k x[m, k] * W[k, n] for m < M, n < N.
 *   x_dev: [M][K] row-major bf16, 16-byte aligned.
 *   y_dev: [M][N] row-major, y_dtype W12_F32 (4-byte aligned) or W12_BF16
 *          (2-byte aligned; rounded to nearest even from the fp32 sum).
 *   1 <= M <= W12_MAX_M.  Accumulation is fp32; the summation order is fixed
 *   for a given (desc, M) so repeated calls give identical bits.
 * Errors: W12_ERR_ARG, W12_ERR_SHAPE, W12_ERR_ALIGN, W12_ERR_WORKSPACE,
 * W12_ERR_CUDA.  Device-detected blob errors: W12_ERR_DEVICE in word 0 of ws.
 */
int w12_gemm(const w12_desc *d, const void *blob_dev, const uint16_t *x_dev, int64_t M,
             void *y_dev, int y_dtype, void *ws_dev, size_t ws_bytes, void *stream);

/* w12_gemm with an explicit path (W12_PATH_*, optionally OR-ed with
 * W12_OPT_EARLY_WEIGHTS); W12_ERR_SHAPE if the path does not serve this M,
 * W12_ERR_ARG for an unknown path or option bit. */
int w12_gemm_ex(const w12_desc *d, const void *blob_dev, const uint16_t *x_dev, int64_t M,
                void *y_dev, int y_dtype, void *ws_dev, size_t ws_bytes, int path,
                void *stream);

#define W12_MAX_BATCH 8

/* Bytes of workspace w12_gemm_batched (and w12_gemm_batched_ex, on any path
 * that serves this M) needs for these matrices and M (0 on invalid
 * arguments). */
size_t w12_gemm_batched_workspace_size(const w12_desc *descs, int count, int64_t M);

/*
 * Defined by: as w12_gemm ("Reasons" bullet 2; "项目介绍" paragraph 2).
 *
 * count independent products y_i = x_i . W_i (1 <= count <= W12_MAX_BATCH,
 * every K_i, N_i > 0) with one M, e.g. the linears of a decoder layer, in ONE
 * kernel launch: the work units of all products (stream-K units of columns x
 * 1024 k) are split evenly over the GPU, so small products (a layer's k and
 * v) neither run alone on a part of the SMs nor pay their own launch and
 * tail.  descs, blobs_dev, x_dev, y_dev are host arrays of count entries
 * (device pointers in the last three), with the layouts and alignments of
 * w12_gemm.  The bits of the results depend only on the descriptors, M, the
 * path and the GPU's SM count (the units' split over the CTAs fixes where
 * fp32 partial sums are cut), so repeated calls give identical results.
 * Errors: as w12_gemm; W12_ERR_SHAPE for an empty product.
 */
int w12_gemm_batched(const w12_desc *descs, const void *const *blobs_dev,
                     const uint16_t *const *x_dev, int64_t M, void *const *y_dev, int y_dtype,
                     int count, void *ws_dev, size_t ws_bytes, void *stream);

/* w12_gemm_batched with an explicit path (W12_PATH_*, optionally OR-ed with
 * W12_OPT_EARLY_WEIGHTS); W12_ERR_SHAPE if the path does not serve this M,
 * W12_ERR_ARG for an unknown path or option bit. */
int w12_gemm_batched_ex(const w12_desc *descs, const void *const *blobs_dev,
                        const uint16_t *const *x_dev, int64_t M, void *const *y_dev, int y_dtype,
                        int count, void *ws_dev, size_t ws_bytes, int path, void *stream);

/*
 * Test hooks of w12_gemm_batched_debug (no counterpart on the pages: they
 * exist to exercise the kernels' bounded waits on a GPU).
 *   withhold_unit: -1, or a work unit (0 <= unit < the batch's unit count)
 *     whose weight copy the producer never issues, so that the consumers'
 *     wait on it runs out and the call records W12_ERR_TIMEOUT.
 *   wait_limit_us: the limit of one bounded wait in microseconds (0: the
 *     default of 2 s; at most 10 s).
 */
typedef struct w12_debug_opts {
    int32_t withhold_unit;
    uint32_t wait_limit_us;
} w12_debug_opts;

/*
 * w12_gemm_batched_ex with test hooks.  With withhold_unit = -1 and
 * wait_limit_us = 0 it is w12_gemm_batched_ex.  After a withheld unit the
 * outputs are undefined and word 0 of the workspace reads W12_ERR_TIMEOUT;
 * every kernel still runs to its end (no wait is unbounded), the
 * workspace's counters are left at zero, and the next call on the same
 * workspace is correct.  Errors: as w12_gemm_batched_ex; W12_ERR_ARG for a
 * NULL dbg or a hook out of range.
 */
int w12_gemm_batched_debug(const w12_desc *descs, const void *const *blobs_dev,
                           const uint16_t *const *x_dev, int64_t M, void *const *y_dev, int y_dtype,
                           int count, void *ws_dev, size_t ws_bytes, int path,
                           const w12_debug_opts *dbg, void *stream);

/* Bytes of workspace w12_verify_greedy needs (>= 256). */
size_t w12_verify_workspace_size(int64_t R, int64_t T, int64_t V);

/*
 * Defined by: "Risks" bullet 3 of the SpecPilot summary (lossless means every
 * committed token is the target model's own greedy choice) and the
 * hotrepo.ai page's "结果与验证" (each committed token is checked against the
 * target's choice at its position).  Tie, NaN and -0 handling and the draft
 * alignment are this library's reading (the pages are silent on them).
 *
 * Greedy verification of R draft blocks of T positions on logits.
 *   logits_dev: [R*T][V] row-major, dtype W12_F32 or W12_BF16, 16-byte aligned.
 *   draft_dev:  [R][T-1] int32 (may be NULL when T == 1).
 *   For each row i of block r, g[r,i] is the lowest index of the row maximum
 *   (NaN above every number, the first NaN wins, -0 == +0).  Row i is the
 *   target's prediction after block input [last token, d0 .. d(i-1)], so it
 *   is compared with draft token i:
 *     accept_len_dev[r] = first i < T-1 with draft[r,i] != g[r,i], else T-1;
 *     next_tok_dev[r]   = g[r, accept_len[r]].
 *   R >= 1, T >= 1, 1 <= V < 2^31.
 * Errors: W12_ERR_ARG, W12_ERR_SHAPE, W12_ERR_ALIGN, W12_ERR_WORKSPACE,
 * W12_ERR_CUDA.
 */
int w12_verify_greedy(const void *logits_dev, int dtype, int64_t R, int64_t T, int64_t V,
                      const int32_t *draft_dev, int32_t *accept_len_dev, int32_t *next_tok_dev,
                      void *ws_dev, size_t ws_bytes, void *stream);

/* Bytes of workspace w12_verify_greedy_lmhead needs (>= 256). */
size_t w12_verify_lmhead_workspace_size(const w12_desc *d_lm, int64_t R, int64_t T);

/*
 * Defined by: as w12_gemm (the lm_head product) and w12_verify_greedy (the
 * acceptance rule): "Reasons" bullet 2, "Risks" bullet 3, "结果与验证".
 *
 * Fused lm_head + greedy verification: logits = hidden @ W_lm (the W12
 * decode-GEMM, fp32 accumulation), then the rule of w12_verify_greedy on
 * those fp32 logits, without writing them unless logits_out_dev is given.
 *   hidden_dev: [R*T][K] bf16, 16-byte aligned; R*T <= W12_MAX_M.
 *   logits_out_dev: NULL, or [R*T][N] fp32 receiving the exact logits the
 *   argmax was taken on.
 * Errors: as w12_gemm and w12_verify_greedy.
 */
int w12_verify_greedy_lmhead(const uint16_t *hidden_dev, const w12_desc *d_lm,
                             const void *blob_lm_dev, int64_t R, int64_t T,
                             const int32_t *draft_dev, int32_t *accept_len_dev,
                             int32_t *next_tok_dev, float *logits_out_dev, void *ws_dev,
                             size_t ws_bytes, void *stream);

/*
 * Scratch memory that w12_verify_greedy_noalloc() keeps, once, on every GPU
 * that loads this library (held until the process exits).
 */
#define W12_NOALLOC_SCRATCH_BYTES (256u * 1024u)

/*
 * w12_verify_greedy() for callers that cannot allocate device memory: a
 * serving loop whose device memory is planned once and may not grow, a host
 * framework that owns every device allocation and passes only inputs and
 * outputs, or a latency-critical path that cannot afford cudaMalloc's
 * implicit device synchronisation.  The paper has no counterpart: this entry
 * point exists only for such callers.
 *
 * Same arguments and results as w12_verify_greedy() without the workspace:
 * the scratch (an arrival counter, the per-slice argmax keys and the
 * per-row tokens) is a fixed W12_NOALLOC_SCRATCH_BYTES array inside the
 * library.  The call allocates nothing, host or device.
 *  - Size limit: a call needs 512 + 8 * R*T * splits + 4 * R*T bytes (each
 *    term rounded up to 256), with splits = max(1, ceil(4 * SMs / (R*T)))
 *    capped at ceil(V / 1024); beyond W12_NOALLOC_SCRATCH_BYTES (about 20000
 *    rows of R*T) it returns W12_ERR_WORKSPACE and launches nothing.
 *  - The first call on each device looks up the array's device address
 *    (cudaGetSymbolAddress, with that device current) and caches it; make
 *    that first call before any stream capture begins.
 *  - Every call on a device shares the one array, which keeps the previous
 *    call's contents; each call clears what has to start at zero.  Calls
 *    that may overlap on the GPU (different streams without ordering, or
 *    several host threads) race on the array and give wrong results:
 *    order them.
 * Errors: as w12_verify_greedy, plus W12_ERR_WORKSPACE for the size limit.
 */
int w12_verify_greedy_noalloc(const void *logits_dev, int dtype, int64_t R, int64_t T, int64_t V,
                              const int32_t *draft_dev, int32_t *accept_len_dev,
                              int32_t *next_tok_dev, void *stream);

/*
 * Read (and clear) the sticky device error word of a workspace: waits for
 * `stream`, copies word 0 to *err_host, then zeroes it.  Returns W12_OK or
 * W12_ERR_CUDA.  *err_host is W12_OK or the first error recorded since the
 * word was last cleared: W12_ERR_DEVICE (a kernel met an escape index
 * outside the escape list) or W12_ERR_TIMEOUT (a bounded wait ran out; the
 * call's outputs are undefined).
 */
int w12_get_device_error(void *ws_dev, int *err_host, void *stream);

#ifdef __cplusplus
}
#endif

#endif /* W12_H */
