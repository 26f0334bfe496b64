/*
 * tg_reduce.h -- the pages' block-reduction study as a measured GB300
 * workload: result = x[0] + x[1] + ... + x[n-1] in fp32.
 *
 * "03 CUDA Shared Memory: Tiling, Bank Conflicts, and Reduction", section
 * "Reduction" (and the reduction cards of "PMPP 단권화"): every block folds
 * its values in shared memory; the partial sums are folded again by the same
 * kernel until one value remains (2^24 inputs with 256-thread blocks:
 * 65,536 -> 256 -> 1).  Variants:
 *  - TG_REDUCE_INTERLEAVED: version 0, `if (tid % (2*s) == 0)` with s
 *    doubling: scattered active lanes and an integer remainder per step.
 *  - TG_REDUCE_SEQUENTIAL: version 1, `if (tid < s)` with s halving: active
 *    lanes packed at the front (47 -> 12 busy warps over a 256-value block).
 *  - TG_REDUCE_SHUFFLE: version 2, as 1 down to 64 values, then the first
 *    warp finishes with __shfl_down_sync (no barriers for the last 6 steps).
 *  - TG_REDUCE_ATOMIC: version 3, one pass; each block adds its partial to
 *    the result with atomicAdd (the result's bits depend on the order the
 *    blocks finish).
 *  - TG_REDUCE_FAST: the GB300 form: float4 loads in a grid-stride loop over
 *    one wave of resident blocks with four independent accumulators, warp
 *    shuffles, then one block folds the per-block partials in fixed order.
 * Every variant but TG_REDUCE_ATOMIC gives the same bits on every run.
 *
 * x and result are device pointers of the current device (compute capability
 * 10.3); result points to one float, which the call overwrites.  n >= 0
 * (n == 0 gives +0.0).  The partial sums live in workspace taken
 * stream-ordered from the library's per-device pool.  Returns TG_OK,
 * TG_ERR_INVALID_VALUE, TG_ERR_UNSUPPORTED_DEVICE, TG_ERR_OUT_OF_MEMORY or
 * TG_ERR_CUDA; the call only enqueues work on `stream`.
 */
#ifndef TG_REDUCE_H
#define TG_REDUCE_H

#include "tg_sgemm.h"

#ifdef __cplusplus
extern "C" {
#endif

typedef enum tg_reduce_variant {
    TG_REDUCE_INTERLEAVED = 0,
    TG_REDUCE_SEQUENTIAL = 1,
    TG_REDUCE_SHUFFLE = 2,
    TG_REDUCE_ATOMIC = 3,
    TG_REDUCE_FAST = 4
} tg_reduce_variant;

tg_status tg_reduce_sum(int variant, long long n, const float* x, float* result, cudaStream_t stream);

/* The launches one call makes (host arithmetic only): *passes kernels
 * (at most 8 listed), counts[p] = values left after launch p (the last is 1),
 * *workspace_bytes for the partial sums.  num_sms = SMs planned for (used by
 * TG_REDUCE_FAST; 0 = query the current device). */
tg_status tg_reduce_plan(int variant, long long n, int num_sms, int* passes, long long* counts,
                         size_t* workspace_bytes);

#ifdef __cplusplus
}
#endif

#endif /* TG_REDUCE_H */
