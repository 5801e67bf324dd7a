// kernels_decode.cu -- W12 blob -> bf16 matrix, bit-exact (the codec check).
//
// Each thread takes one 16-byte chunk of each plane of a unit block: 32
// consecutive k of one column (a quarter group), rebuilds them with
// rebuild32() and patches escapes.  For [N][K] output consecutive threads
// read consecutive chunks of a unit block (coalesced reads) and write 64
// contiguous bytes each; [K][N] output goes through a shared-memory
// transpose of a 64-column x 128-k tile so stores stay coalesced.
// HBM-bound: 1.5 B read + 2 B written per weight.
#include <cuda_runtime.h>

#include "device_common.cuh"
#include "w12_internal.h"

namespace w12 {

namespace {

struct DecodeArgs {
    const uint8_t *units;
    const uint16_t *esc;
    uint64_t n_esc;
    int64_t K, N, KG, U;  // KG = K/128 groups per column, U unit blocks
    uint16_t *w;
    int *err;
};

// Rebuild quarter j (k = 128 kg + 32 j .. + 31) of column n into out[16].
__device__ __forceinline__ void decode_vector(const DecodeArgs &a, int64_t n, int64_t kg, int j, uint32_t out[16]) {
    const int64_t u = (n / kTileCols) * a.KG + kg;
    const int c = int(n % kTileCols);
    const uint8_t *ub = a.units + u * kUnitBytes;
    const uint32_t off = uint32_t(c * 64 + ((j ^ ((c >> 1) & 3)) << 4));
    const uint4 h = ldg_stream(ub + off);
    const uint4 l = ldg_stream(ub + kPlaneBlock + off);
    const uint4 e = ldg_stream(ub + 2 * kPlaneBlock + off);
    const uint32_t *meta = reinterpret_cast<const uint32_t *>(ub + kMetaAt);
    const uint32_t m0 = ldg_u32(meta + c), m1 = ldg_u32(meta + c + 1);
    rebuild32(h, l, e, base4(m0), out);
    if (m0 >> 8 != m1 >> 8) patch_escapes(out, m0, m1, uint32_t(j) * 32u, a.esc, a.n_esc, a.err);
}

__global__ void __launch_bounds__(256) decode_nk_kernel(const DecodeArgs a) {
    // v = (unit, column, quarter): consecutive threads read consecutive chunks
    const int64_t total = a.U * kTileCols * 4;
    for (int64_t v = int64_t(blockIdx.x) * blockDim.x + threadIdx.x; v < total;
         v += int64_t(gridDim.x) * blockDim.x) {
        const int64_t u = v / (kTileCols * 4);
        const int c = int((v / 4) % kTileCols), j = int(v % 4);
        const int64_t n = (u / a.KG) * kTileCols + c, kg = u % a.KG;
        if (n >= a.N) continue;
        uint32_t out[16];
        decode_vector(a, n, kg, j, out);
        uint4 *dst = reinterpret_cast<uint4 *>(a.w + n * a.K + kg * 128 + 32 * j);
        dst[0] = make_uint4(out[0], out[1], out[2], out[3]);
        dst[1] = make_uint4(out[4], out[5], out[6], out[7]);
        dst[2] = make_uint4(out[8], out[9], out[10], out[11]);
        dst[3] = make_uint4(out[12], out[13], out[14], out[15]);
    }
}

constexpr int kTCols = 64;
constexpr int kTilePad = 66;  // uint16 row pitch of the transpose tile (breaks bank aliasing)

__global__ void __launch_bounds__(256) decode_kn_kernel(const DecodeArgs a) {
    __shared__ uint16_t tile[128 * kTilePad];
    const int64_t KG = a.K / 128;
    const int64_t ncb = (a.N + kTCols - 1) / kTCols;
    const int64_t tiles = ncb * KG;
    const int col = threadIdx.x >> 2, quarter = threadIdx.x & 3;
    for (int64_t t = blockIdx.x; t < tiles; t += gridDim.x) {
        const int64_t kg = t / ncb, cb = t % ncb;
        const int64_t n = cb * kTCols + col;
        if (n < a.N) {
            uint32_t out[16];
            decode_vector(a, n, kg, quarter, out);
#pragma unroll
            for (int i = 0; i < 16; ++i) {
                const int k = quarter * 32 + 2 * i;
                tile[k * kTilePad + col] = uint16_t(out[i] & 0xFFFFu);
                tile[(k + 1) * kTilePad + col] = uint16_t(out[i] >> 16);
            }
        }
        __syncthreads();
        // 128 rows x 64 columns: each thread writes 32 consecutive uint16 pairs
        for (int idx = threadIdx.x; idx < 128 * (kTCols / 2); idx += blockDim.x) {
            const int r = idx / (kTCols / 2), c2 = (idx % (kTCols / 2)) * 2;
            const int64_t n0 = cb * kTCols + c2;
            uint16_t *dst = a.w + (kg * 128 + r) * a.N + n0;
            if (n0 + 1 < a.N && ((reinterpret_cast<uintptr_t>(dst) & 3u) == 0)) {
                const uint32_t pair = uint32_t(tile[r * kTilePad + c2]) |
                                      (uint32_t(tile[r * kTilePad + c2 + 1]) << 16);
                *reinterpret_cast<uint32_t *>(dst) = pair;
            } else {
                if (n0 < a.N) dst[0] = tile[r * kTilePad + c2];
                if (n0 + 1 < a.N) dst[1] = tile[r * kTilePad + c2 + 1];
            }
        }
        __syncthreads();
    }
}

}  // namespace

int device_sm_count(int *sms) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return W12_ERR_CUDA;
    if (cudaDeviceGetAttribute(sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
        return W12_ERR_CUDA;
    return W12_OK;
}

int launch_decode(const w12_desc *d, const void *blob, uint16_t *w, int layout, int *err,
                  void *stream) {
    if (d->G == 0) return W12_OK;
    const uint8_t *b = static_cast<const uint8_t *>(blob);
    DecodeArgs a;
    a.units = b + d->off_units;
    a.esc = reinterpret_cast<const uint16_t *>(b + d->off_esc);
    a.n_esc = d->n_esc;
    a.K = d->K;
    a.N = d->N;
    a.KG = d->K / kGroup;
    a.U = int64_t(d->n_units);
    a.w = w;
    a.err = err;
    int sms = 0;
    if (device_sm_count(&sms) != W12_OK) return W12_ERR_CUDA;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (layout == W12_LAYOUT_NK) {
        const int64_t total = a.U * kTileCols * 4;
        int64_t grid = (total + 255) / 256;
        if (grid > int64_t(sms) * 8) grid = int64_t(sms) * 8;
        decode_nk_kernel<<<unsigned(grid), 256, 0, s>>>(a);
    } else {
        const int64_t tiles = ((a.N + kTCols - 1) / kTCols) * (a.K / 128);
        int64_t grid = tiles < int64_t(sms) * 8 ? tiles : int64_t(sms) * 8;
        decode_kn_kernel<<<unsigned(grid), 256, 0, s>>>(a);
    }
    return cudaGetLastError() == cudaSuccess ? W12_OK : W12_ERR_CUDA;
}

}  // namespace w12
