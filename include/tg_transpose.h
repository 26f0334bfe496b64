/*
 * tg_transpose.h -- the tiled matrix transpose of the pages' bank-conflict
 * study, as a measured GB300 workload.
 *
 * out[c][r] = in[r][c] for 0 <= r < rows, 0 <= c < cols, row-major:
 * in[r*ld_in + c] (ld_in >= max(1,cols)), out[c*ld_out + r]
 * (ld_out >= max(1,rows)).  Pointers are device pointers of the current
 * device (compute capability 10.3); in and out must not overlap.  The call
 * enqueues one kernel on `stream` and returns TG_OK, TG_ERR_INVALID_VALUE
 * (bad variant, size, stride, null or overlapping pointer),
 * TG_ERR_UNSUPPORTED_DEVICE or TG_ERR_CUDA.
 *
 * Variants ("03 CUDA Shared Memory: Tiling, Bank Conflicts, and Reduction",
 * sections "Global Memory와 Coalescing" and "Bank Conflict"); every tiled
 * variant reads a 32 x 32 tile along rows (coalesced) into shared memory and
 * writes it out along rows of the output (coalesced), reading the tile down
 * its columns:
 *  - TG_TRANSPOSE_DIRECT: no shared memory; coalesced reads, writes strided
 *    by ld_out (one 32-byte sector per element).
 *  - TG_TRANSPOSE_TILE32: __shared__ float tile[32][32]; the column read puts
 *    all 32 lanes on one bank (32-way conflict).
 *  - TG_TRANSPOSE_PADDED: tile[32][33]; conflict degree gcd(33, 32) = 1.
 *  - TG_TRANSPOSE_SWIZZLED: tile[32][32] with column c of row r stored at
 *    c ^ r; rows and columns both touch every bank once.
 * All variants give the same result bit for bit.
 */
#ifndef TG_TRANSPOSE_H
#define TG_TRANSPOSE_H

#include "tg_sgemm.h"

#ifdef __cplusplus
extern "C" {
#endif

typedef enum tg_transpose_variant {
    TG_TRANSPOSE_DIRECT = 0,
    TG_TRANSPOSE_TILE32 = 1,
    TG_TRANSPOSE_PADDED = 2,
    TG_TRANSPOSE_SWIZZLED = 3
} tg_transpose_variant;

tg_status tg_transpose(int variant, int rows, int cols, const float* in, int ld_in, float* out,
                       int ld_out, cudaStream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* TG_TRANSPOSE_H */
