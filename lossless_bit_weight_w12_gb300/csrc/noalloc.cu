// noalloc.cu -- greedy verification that needs no caller-provided workspace.
//
// w12_verify_greedy() takes its scratch memory (an arrival counter, one
// partial argmax key per row and logits slice, one token per row) from a
// workspace the caller allocates.  Some callers cannot allocate device memory
// at all: a serving loop whose device memory is planned once at start-up and
// may not grow, a host framework that owns every device allocation and hands
// the library only its inputs and outputs, or a latency-critical path where
// the implicit device synchronisation of cudaMalloc is not acceptable.  For
// them, w12_verify_greedy_noalloc() runs the same kernel on a scratch array
// that lives in this library's own device memory: the array below, reserved
// on every GPU that loads the library until the process exits.
#include <cuda_runtime.h>

#include <mutex>

#include "w12_internal.h"

namespace w12 {

namespace {

// The one scratch array (W12_NOALLOC_SCRATCH_BYTES per device, 256-byte
// aligned).  Host code must not use its name as a pointer: on the host it is
// only a stand-in for the symbol; the device address comes from
// cudaGetSymbolAddress() below.
static __device__ __align__(256) unsigned char g_verify_scratch[W12_NOALLOC_SCRATCH_BYTES];

constexpr int kMaxDevices = 256;
std::mutex g_mu;
void *g_scratch_addr[kMaxDevices] = {};

// Device address of the scratch array on the current device, looked up once
// per device (with that device current) and cached.
int scratch_address(void **out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return W12_ERR_CUDA;
    std::lock_guard<std::mutex> lock(g_mu);
    if (!g_scratch_addr[dev]) {
        void *p = nullptr;
        if (cudaGetSymbolAddress(&p, g_verify_scratch) != cudaSuccess || !p) return W12_ERR_CUDA;
        g_scratch_addr[dev] = p;
    }
    *out = g_scratch_addr[dev];
    return W12_OK;
}

bool aligned(const void *p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0; }

}  // namespace

}  // namespace w12

using namespace w12;

extern "C" int w12_verify_greedy_noalloc(const void *logits, int dtype, int64_t R, int64_t T,
                                         int64_t V, const int32_t *draft, int32_t *accept_len,
                                         int32_t *next_tok, void *stream) {
    if (dtype != W12_F32 && dtype != W12_BF16) return W12_ERR_ARG;
    if (R < 1 || T < 1 || V < 1 || V >= (int64_t(1) << 31)) return W12_ERR_SHAPE;
    if (!logits || !accept_len || !next_tok || (T > 1 && !draft)) return W12_ERR_ARG;
    if (!aligned(logits, dtype == W12_F32 ? 4 : 2) || !aligned(accept_len, 4) ||
        !aligned(next_tok, 4) || (draft && !aligned(draft, 4)))
        return W12_ERR_ALIGN;

    // The same work split and scratch layout as w12_verify_greedy.
    VerifyArgs a;
    int grid;
    const int64_t rows = R * T;
    if (verify_plan(rows, V, &grid, &a.splits, &a.chunk) != W12_OK) return W12_ERR_CUDA;
    if (verify_ws(rows, a.splits) > W12_NOALLOC_SCRATCH_BYTES) return W12_ERR_WORKSPACE;

    void *scratch = nullptr;
    int st = scratch_address(&scratch);
    if (st != W12_OK) return st;
    uint8_t *ws = static_cast<uint8_t *>(scratch);
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    // The array keeps whatever the previous call left; the error word and the
    // arrival counter must start at zero.
    if (cudaMemsetAsync(ws, 0, kWsHeader + 256, s) != cudaSuccess) return W12_ERR_CUDA;

    a.logits = logits;
    a.dtype = dtype;
    a.R = R;
    a.T = T;
    a.V = V;
    a.rows = rows;
    a.draft = draft;
    a.accept_len = accept_len;
    a.next_tok = next_tok;
    verify_layout(ws, rows, a.splits, &a);
    return launch_verify(a, grid, stream);
}
