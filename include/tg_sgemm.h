/*
 * tg_sgemm.h -- C ABI of the GB300 (sm_103a) row-major FP32 matrix product.
 *
 * The operation is C = A x B:
 *
 *     C[i][j] = sum_{k=0}^{K-1} A[i][k] * B[k][j],   0 <= i < M, 0 <= j < N
 *
 * as defined in "03 CUDA Shared Memory: Tiling, Bank Conflicts, and
 * Reduction" (section "Shared Memory와 Tiling": one row of A times one column
 * of B, two FLOP per k) and in the PMPP ch. 5 notes ("메모리 계층과 데이터
 * 지역성", §5.4 tiled kernel, §5.5 ghost elements: out-of-range tile entries
 * are zeros, only the final store is range-checked).  The pages show square
 * matrices; this library takes any M, N, K >= 0 with row strides.
 *
 * Layout: every matrix is row-major with a leading dimension (row stride, in
 * elements): A[i*lda + k], B[k*ldb + j], C[i*ldc + j] (row-major linear index
 * r*W + c, "PMPP 단권화" ch. 3).  Requirements: lda >= max(1,K),
 * ldb >= max(1,N), ldc >= max(1,N).  No alignment is required of the
 * pointers or strides.  C is overwritten (there is no alpha/beta); columns
 * j >= N of a padded C row are never written.  K == 0 writes +0.0 to the
 * whole M x N block of C.  C must not overlap A or B.
 *
 * Pointers are device pointers of the current CUDA device (except for
 * tg_sgemm_host).  The caller owns A, B, C and any workspace; the library
 * never frees or keeps them.
 *
 * Execution follows the CUDA host-program pattern of "PMPP 단권화" ch. 2
 * (caller-owned buffers, cudaError_t-style return codes, streams): calls only
 * enqueue work on `stream` and return without synchronising the host.  Errors
 * found before launch (bad arguments, unsupported device, launch failure) are
 * returned at once.  A kernel that gives up a bounded wait records a timeout
 * in a per-device error word instead of trapping; tg_sgemm_sync_status
 * reports it.
 *
 * Only GB300-class devices (compute capability 10.3) are supported; there is
 * no CPU fallback and no other backend.
 */
#ifndef TG_SGEMM_H
#define TG_SGEMM_H

#include <stddef.h>
#include <cuda_runtime_api.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Return codes. */
typedef enum tg_status {
    TG_OK = 0,
    TG_ERR_INVALID_VALUE = 1,      /* bad size, stride, null or overlapping pointer, bad option */
    TG_ERR_UNSUPPORTED_DEVICE = 2, /* current device is not compute capability 10.3 */
    TG_ERR_OUT_OF_MEMORY = 3,      /* workspace allocation failed */
    TG_ERR_CUDA = 4,               /* a CUDA runtime call or launch failed (sticky errors stay set) */
    TG_ERR_TIMEOUT = 5,            /* a kernel gave up a bounded wait (reported by tg_sgemm_sync_status) */
    TG_ERR_WORKSPACE_TOO_SMALL = 6 /* caller workspace smaller than tg_sgemm_plan's workspace_bytes */
} tg_status;

/* Operand form for tg_sgemm_general: TG_OP_N = as stored, TG_OP_T =
 * transposed (the stored matrix is op(X)^T). */
typedef enum tg_op { TG_OP_N = 0, TG_OP_T = 1 } tg_op;

/* Math paths, all hand-written sm_103a kernels.
 *  - TG_PATH_TF32X3: tensor cores (tcgen05.mma kind::tf32, accumulator in
 *    tensor memory), fed through an mbarrier pipeline by a producer warp.
 *    Each float is split into hi = tf32(x) and lo = tf32(x - hi); the product
 *    is lo*hi + hi*lo + hi*hi.  A pre-pass writes hi/lo tiles of B
 *    transposed; A stored untransposed with a 16-byte-aligned base and row
 *    pitch is read in place and split inside the GEMM kernel (hi = x
 *    truncated to tf32, as the tensor core reads it), else the pre-pass
 *    writes A's tiles too (tg_plan_info.fused_split).
 *  - TG_PATH_FFMA: register-blocked fused multiply-add on the CUDA cores, fp32
 *    throughout, TMA-fed through the same kind of pipeline.
 *  - TG_PATH_TILED: the shared-memory tiled kernel for small products: one
 *    launch, no pre-pass and no workspace, 64 x 64 tiles, fp32 fused
 *    multiply-adds; operands read in place with any alignment.  A block of
 *    256 threads handles one tile (with few tiles, a cluster of up to 8
 *    blocks handles one tile over slices of K and adds the slices in shared
 *    memory, in a fixed order), so large products run it far below the other
 *    paths.
 *  - TG_PATH_TF32_BF16: the TG_PATH_TF32X3 kernels and split (hi = tf32(x),
 *    lo = x - hi), with the two cross products taken in bf16: the product is
 *    hi*hi (kind::tf32) + bf16(hi)*bf16(lo) + bf16(lo)*bf16(hi) (kind::f16,
 *    bf16 operands, fp32 accumulator).  A cross product is at most 2^-11 of
 *    the main one, so rounding its operands to bf16's 8 significant bits adds
 *    at most about 2^-18 of |a*b| each, about 2^-17 per product with the
 *    dropped lo*lo (3xTF32: about 2^-21); bf16 has fp32's exponent range, so
 *    no operand scaling is needed.  Two of the three products run at bf16
 *    rate: four tensor instructions per 16-wide K block instead of six.
 *    Integers with |x| <= 2^11 (and partial sums below 2^24) stay exact: lo
 *    is zero, so the cross products vanish.  Only on request; TG_PATH_AUTO
 *    never picks it.
 *  - TG_PATH_AUTO: TG_PATH_TILED for small products (where one launch beats
 *    the three of the 3xTF32 path; see tg_sgemm_plan), else TG_PATH_TF32X3. */
typedef enum tg_path {
    TG_PATH_AUTO = 0,
    TG_PATH_FFMA = 1,
    TG_PATH_TF32X3 = 2,
    TG_PATH_TILED = 3,
    TG_PATH_TF32_BF16 = 4
} tg_path;

/* Options for tg_sgemm_ex.  Zero-initialise and set what you need.
 *  path            tg_path value.
 *  split_k         0 = automatic; S >= 1 = split K into S slices whose fp32
 *                  partial products are summed in fixed slice order by a
 *                  reduce kernel (deterministic: no float atomics).  S is
 *                  capped at the number of K blocks.
 *  workspace       optional device buffer of at least workspace_bytes (as
 *                  reported by tg_sgemm_plan), 256-byte aligned.  NULL = the
 *                  library allocates it stream-ordered on `stream` from its
 *                  own per-device memory pool and frees it stream-ordered.
 *  main_begin/end  optional events, recorded on `stream` immediately before
 *                  and after the main GEMM kernel (for timing it alone). */
typedef struct tg_sgemm_opts {
    int path;
    int split_k;
    void* workspace;
    size_t workspace_bytes;
    cudaEvent_t main_begin;
    cudaEvent_t main_end;
} tg_sgemm_opts;

/* What one call would launch (filled by tg_sgemm_plan). */
typedef struct tg_plan_info {
    int path;          /* TG_PATH_FFMA, TG_PATH_TF32X3, TG_PATH_TILED or TG_PATH_TF32_BF16 */
    int split_k;       /* K slices */
    int block_m, block_n, block_k, stages; /* CTA tile and pipeline depth */
    int tiles_m, tiles_n;
    long long units;   /* tiles x split_k work units */
    int grid;          /* persistent CTAs launched (<= SM count) */
    int prepass;       /* 1 = an operand re-layout kernel runs first */
    int launches;      /* kernels one call launches */
    size_t workspace_bytes;
    int pair;          /* 3xTF32: CTAs per cluster sharing one B tile through a pair MMA (1 or 2);
                          a unit is then `pair` vertically adjacent tiles */
    long long tail_units; /* units after the last whole round of lanes, balanced (0 = none) */
    int tail_lanes;       /* lanes (CTAs, or CTA pairs) sharing those units' K blocks equally */
    int tail_kx;          /* 0: the lanes run the units' K blocks laid end to end (stream-K) or
                             equal K slices; > 0: unit q's first tail_kx K blocks run on lane q,
                             all in step, the rest of every unit over the other lanes */
    int fused_split;      /* tensor paths: 1 = A is staged raw from the caller's buffer and split
                             inside the GEMM kernel (no pre-pass copy of A; B always takes the
                             pre-pass); 0 = both operands are split by the pre-pass */
} tg_plan_info;

/* C = A x B with automatic path and split choice (see the file comment for
 * layout, ownership and errors).  Returns TG_OK, TG_ERR_INVALID_VALUE,
 * TG_ERR_UNSUPPORTED_DEVICE, TG_ERR_OUT_OF_MEMORY or TG_ERR_CUDA. */
tg_status tg_sgemm(int M, int N, int K, const float* A, int lda, const float* B, int ldb,
                   float* C, int ldc, cudaStream_t stream);

/* tg_sgemm with options (opts may be NULL = defaults).  Additionally returns
 * TG_ERR_WORKSPACE_TOO_SMALL. */
tg_status tg_sgemm_ex(int M, int N, int K, const float* A, int lda, const float* B, int ldb,
                      float* C, int ldc, cudaStream_t stream, const tg_sgemm_opts* opts);

/* General form: C = alpha * op(A) * op(B) + beta * C, with op(A) M x K and
 * op(B) K x N.  A is stored M x K (lda >= max(1,K)) for TG_OP_N and K x M
 * (lda >= max(1,M)) for TG_OP_T; B is stored K x N (ldb >= max(1,N)) for
 * TG_OP_N and N x K (ldb >= max(1,K)) for TG_OP_T; all row-major.  These are
 * the products of a fully connected layer's forward and backward passes
 * ("PMPP 단권화", deep-learning chapter: FC layer = GEMM, dW = X^T dY,
 * dX = dY W^T).  When beta == 0, C is not read (it may hold NaN); K == 0 gives
 * C = beta * C.  alpha and beta are applied in fp32 where C is written
 * (alpha * sum + beta * C with one fused multiply-add).  tg_sgemm_ex is this
 * call with TG_OP_N, TG_OP_N, alpha = 1, beta = 0.  Other semantics and
 * return codes as tg_sgemm_ex, plus TG_ERR_INVALID_VALUE for an op other than
 * TG_OP_N / TG_OP_T. */
tg_status tg_sgemm_general(int op_a, int op_b, int M, int N, int K, float alpha, const float* A,
                           int lda, const float* B, int ldb, float beta, float* C, int ldc,
                           cudaStream_t stream, const tg_sgemm_opts* opts);

/* Plan a call without launching anything: host arithmetic only.  Pointers
 * may be NULL (then the most conservative alignment is assumed).  num_sms is
 * the SM count to plan for; 0 = query the current device.  path/split_k as in
 * tg_sgemm_opts.  Returns TG_OK or TG_ERR_INVALID_VALUE (bad sizes, strides,
 * path, split_k < 0, out == NULL). */
tg_status tg_sgemm_plan(int M, int N, int K, const void* A, int lda, const void* B, int ldb,
                        const void* C, int ldc, int path, int split_k, int num_sms,
                        tg_plan_info* out);

/* tg_sgemm_plan for tg_sgemm_general's operand forms (op_a, op_b as there;
 * the leading dimensions refer to the stored matrices). */
tg_status tg_sgemm_plan_general(int op_a, int op_b, int M, int N, int K, const void* A, int lda,
                                const void* B, int ldb, const void* C, int ldc, int path,
                                int split_k, int num_sms, tg_plan_info* out);

/* Workspace bytes tg_sgemm_ex needs for these arguments on the current
 * device (0 on invalid arguments).  Same as tg_sgemm_plan(...).workspace_bytes. */
size_t tg_sgemm_workspace_bytes(int M, int N, int K, const void* A, int lda, const void* B,
                                int ldb, const void* C, int ldc, int path, int split_k);

/* Host-buffer convenience call: A, B and C are HOST pointers (pinned memory
 * gives asynchronous copies).  Copies A and B to device memory allocated
 * stream-ordered on `stream`, computes C = A x B there, copies C back and
 * synchronises `stream` before returning, so C is ready on return.  Also
 * returns TG_ERR_TIMEOUT if a kernel of this call gave up a wait.
 * Large products are pipelined: C is cut into row blocks, the first of them
 * also into column blocks (see tg_sgemm_host_blocks); the first product
 * starts once its A row block and B column block are on the device, later
 * row blocks are computed full width once all of B is in, and the copies of
 * the other blocks (in on one copy stream, C out on another) overlap the
 * products.  TG_HOST_TRACE=1 in the environment prints the call's timeline
 * (copies, products) to stderr.  opts->split_k
 * and path apply to every block's product; workspace, main_begin and main_end
 * are ignored.  Below 2^33 multiply-adds (M*N*K) there is one block and C is
 * bit-identical to tg_sgemm's; above, each block's product is planned on its
 * own, so the K split and the order of the partial sums (the low bits) may
 * differ, within the same error bounds. */
tg_status tg_sgemm_host(int M, int N, int K, const float* A, int lda, const float* B, int ldb,
                        float* C, int ldc, cudaStream_t stream, const tg_sgemm_opts* opts);

/* The output blocks tg_sgemm_host uses for a shape (host arithmetic only).
 * C is cut into row_blocks row blocks: row block 0 has first_block_rows rows
 * (a short first block lets the first product start sooner), the next ones
 * block_rows, the last one the remaining rows (possibly fewer).  Row blocks
 * 0 .. split_row_blocks - 1 are cut into col_blocks column blocks of
 * block_cols columns (the last ragged); the later row blocks are one
 * full-width product each.  With defer_copies_out != 0 the copies of C out
 * wait until every copy in is done (the host link then carries one direction
 * at a time).  model_ms is the modelled time of the call (copy rates measured
 * on GB300). */
typedef struct {
    int row_blocks;
    int col_blocks;
    int first_block_rows;
    int block_rows;
    int block_cols;
    int split_row_blocks;
    int defer_copies_out;
    double model_ms;
} tg_host_blocks_info;

/* Fill *out with the blocks tg_sgemm_host would use, chosen to minimise the
 * modelled time.  path as in tg_sgemm_opts; num_sms = SMs planned for (0 =
 * the current device).  TG_ERR_INVALID_VALUE on negative sizes, an unknown
 * path or out == NULL. */
tg_status tg_sgemm_host_blocks(int M, int N, int K, int path, int num_sms, tg_host_blocks_info* out);

/* Device memory tg_sgemm_host allocates (stream-ordered, from the device's
 * memory pool) for these sizes, with the blocks tg_sgemm_host_blocks reports:
 * *total = the copies of A, B and C (16-byte row pitches), the split tiles
 * and the largest workspace any one product needs (also in
 * *product_workspace, which may be NULL).  Host arithmetic only; path and
 * split_k as in tg_sgemm_opts, num_sms as in tg_sgemm_host_blocks.
 * TG_ERR_INVALID_VALUE on negative sizes, an unknown path or total == NULL. */
tg_status tg_sgemm_host_device_bytes(int M, int N, int K, int path, int split_k, int num_sms, size_t* total,
                                     size_t* product_workspace);

/* Synchronise `stream`, then read and clear the current device's error word.
 * Returns TG_ERR_TIMEOUT if any kernel of this library on this device gave up
 * a bounded wait since the last check (the word is shared by all streams),
 * TG_ERR_CUDA if the synchronisation failed, else TG_OK. */
tg_status tg_sgemm_sync_status(cudaStream_t stream);

/* Raw value of the current device's error word (0 = none; otherwise a site
 * code of the wait that gave up) without clearing it.  Synchronises `stream`. */
unsigned int tg_sgemm_error_site(cudaStream_t stream);

/* Self-test of the bounded wait: launches one tiny kernel that waits on an
 * mbarrier nothing will ever arrive on, with a limit of timeout_us
 * microseconds (1..10,000,000).  The kernel records a timeout in the error
 * word and returns; the context stays usable.  Returns the launch status;
 * the caller then expects tg_sgemm_sync_status == TG_ERR_TIMEOUT. */
tg_status tg_selftest_wait_timeout(unsigned int timeout_us, cudaStream_t stream);

/* Bytes of the fixed device scratch array behind tg_sgemm_noalloc (64 MiB). */
#define TG_SGEMM_NOALLOC_SCRATCH_BYTES ((size_t)64 << 20)

/* C = A x B on the 3xTF32 path without allocating any memory.  The source
 * pages have no counterpart of this entry point; it exists for callers that
 * cannot allocate device memory at call time -- for example a host
 * application that owns the whole device-memory budget through its own
 * allocator and does not let libraries allocate, a latency-critical loop that
 * must never enter the CUDA allocator, or code that must not be able to fail
 * with out-of-memory once it runs.  tg_sgemm needs scratch memory (the hi/lo
 * copies of B, and of A unless the GEMM kernel splits A itself, and K-slice
 * partials); here that scratch is a fixed
 * array of TG_SGEMM_NOALLOC_SCRATCH_BYTES in device memory that CUDA reserves
 * when it loads this library's device code on a GPU (with CUDA's default lazy
 * loading: at the first tg_sgemm_noalloc call there) and that every such GPU
 * holds until the process exits.  This call makes no cudaMalloc, cudaFree or
 * other allocating call.
 *
 * Arguments, layout, ownership and results are those of tg_sgemm.  Limit: the
 * hi/lo copies need 8*(M'+N')*K' bytes, with M' = M rounded up to a multiple
 * of 256 (128 when M <= 128), N' = N rounded up to a multiple of 256 and K' =
 * K rounded up to a multiple of 16 (the split tiles are whole 128-row tiles,
 * paired along M); M' is 0 when the GEMM kernel splits A itself (M > 128, A's
 * base and lda*4 multiples of 16 bytes; see tg_plan_info.fused_split).
 * Split-K and balanced-tail partials come on top and are dropped when they
 * would not fit.  A product whose split tiles exceed
 * TG_SGEMM_NOALLOC_SCRATCH_BYTES returns TG_ERR_WORKSPACE_TOO_SMALL and
 * launches nothing (M = 2048, N = 4096, K = 2048 with A split in the kernel
 * fits exactly; N = 4097 does not).
 *
 * The first call on each device does a one-time set-up there (capability
 * check, kernel attributes, and the scratch's device address via
 * cudaGetSymbolAddress); make that first call before any stream capture.
 * Every call on a device shares the one scratch array, which keeps the last
 * call's contents (nothing in it needs to start at zero): calls whose work
 * overlaps on the GPU -- on different streams, or from host threads that do
 * not order them -- race on it and give wrong results.  Order such calls, for
 * example by issuing them on one stream. */
tg_status tg_sgemm_noalloc(int M, int N, int K, const float* A, int lda, const float* B, int ldb,
                           float* C, int ldc, cudaStream_t stream);

/* Static description of a status code (never NULL). */
const char* tg_status_string(tg_status status);

/* Library ABI version (major*100 + minor). */
int tg_sgemm_version(void);

#ifdef __cplusplus
}
#endif

#endif /* TG_SGEMM_H */
