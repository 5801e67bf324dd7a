// verify_common.cuh -- the greedy acceptance step, run by the last CTA.
//
// "Lossless" greedy speculative decoding: every committed token is the
// target model's own greedy choice (SpecPilot summary, airadar.tv English
// edition, "Risks" bullet 3; repository page "结果与验证": each committed
// token is checked against the target's choice at that position).  Per
// position the target token is the lowest index of the row maximum; the
// accepted prefix is the longest run of draft tokens equal to the target's,
// and the next token is the target's token at the first mismatch (or at the
// last position when all drafts agree).
#pragma once

#include "device_common.cuh"

namespace w12 {

// keys[c * rows + row] for c < ncol hold partial (value, ~index) maxima of
// each row.  Called by threads tid = 0 .. nthreads - 1 of one CTA: the
// whole CTA (nthreads == blockDim.x) or its first nthreads threads, which
// then synchronise on named barrier 1.  gbuf: rows int32 scratch.
__device__ __forceinline__ void verify_from_keys(const unsigned long long *keys, int64_t ncol,
                                                 int64_t rows, int64_t R, int64_t T,
                                                 const int32_t *draft, int32_t *accept_len,
                                                 int32_t *next_tok, int32_t *gbuf,
                                                 int tid = -1, int nthreads = -1) {
    if (tid < 0) {
        tid = int(threadIdx.x);
        nthreads = int(blockDim.x);
    }
    for (int64_t row = tid; row < rows; row += nthreads) {
        unsigned long long best = 0ull;
        for (int64_t c = 0; c < ncol; ++c) {
            const unsigned long long k = __ldcg(&keys[c * rows + row]);
            best = k > best ? k : best;
        }
        gbuf[row] = int32_t(key_index(best));
    }
    if (nthreads == int(blockDim.x))
        __syncthreads();
    else
        asm volatile("bar.sync 1, %0;" ::"r"(nthreads) : "memory");
    for (int64_t r = tid; r < R; r += nthreads) {
        int64_t L = T - 1;
        for (int64_t i = 0; i < T - 1; ++i) {
            if (__ldcg(&draft[r * (T - 1) + i]) != __ldcg(&gbuf[r * T + i])) {
                L = i;
                break;
            }
        }
        accept_len[r] = int32_t(L);
        next_tok[r] = __ldcg(&gbuf[r * T + L]);
    }
}

}  // namespace w12
