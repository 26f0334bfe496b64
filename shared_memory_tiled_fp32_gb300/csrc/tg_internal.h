// Internal declarations shared by the host planner, the C-ABI entry points
// and the kernel launchers.  Not part of the public interface.
#pragma once

#include <cstddef>
#include <cstdint>

#include "../../include/tg_sgemm.h"

namespace tg {

// The tensor-core paths (3xTF32 and its bf16-cross-product variant) share
// the plan, the pre-pass tiles and the GEMM kernel.
inline bool tensor_path(int path) { return path == TG_PATH_TF32X3 || path == TG_PATH_TF32_BF16; }

// CTA tile shapes of the two math paths.
//
// TF32x3: a 128 x 256 output tile per CTA (a 256 x 256 tile per CTA pair;
// N=256 accumulator rows of 256 of the 512 tensor-memory columns, so two
// chunks are in flight), K staged 16 values at a time (hi and lo: one
// 128-byte swizzle row per tile row); kTf32Stages stages of 48 KiB in the
// per-CTA form (the pair-MMA form holds 6 of 32 KiB, see tg_kernels.cu).
constexpr int kTf32BM = 128, kTf32BN = 256, kTf32BK = 16, kTf32Stages = 4;
// FFMA: a 128 x 256 output tile, 256 math threads each holding an 8 x 16
// register block, K staged 32 floats at a time, 4 stages of 48 KiB.
constexpr int kFfmaBM = 128, kFfmaBN = 256, kFfmaBK = 32, kFfmaStages = 4;

// Tiled path (small products): 64 x 64 tiles, K staged 16 at a time; K
// split over at most 8 blocks per tile (one cluster, the portable size).
constexpr int kTiledBM = 64, kTiledBN = 64, kTiledBK = 16, kTiledMaxSplit = 8;
// The automatic path takes the tiled kernel up to 2^26 multiply-adds with K
// at most 512 (one block per tile: its time grows with K, and past that size
// the 3xTF32 path's three launches cost less than the tiled path's math;
// measured on GB300: 256^3 15.9 vs 21.2 us, 384^3 21.0 vs 23.6, 512^3 27.9
// vs 22.2, 128 x 128 x 8192 416 vs 35).
constexpr double kTiledMaxMacs = 67108864.0;  // 2^26
constexpr int kTiledMaxK = 512;

constexpr size_t kWsAlign = 256;

#ifdef __CUDACC__
#define TG_HOST_DEVICE __host__ __device__
#else
#define TG_HOST_DEVICE
#endif

// Tile-unit index t (K slices aside) -> (tile-unit row, tile column).  Tiles
// are visited in groups of kGroupM tile-unit rows, column by column inside a
// group, so CTAs running at the same time share A rows and B columns in L2.
// With 76 CTA pairs a round of pair units is then a block of 19 pair rows x
// 4 columns, and the next round (the next 4 columns) keeps the same A rows;
// the 3xTF32 kernel walks K backwards on every second work item, so a round
// starts on the K range of A the previous one ended with, still in L2.
// Measured on GB300, 8192^3 DRAM read per launch (same kernel time within
// 1 %): groups of 8 pair rows 3.30 GB, 12 2.96, 16 2.96, 19 2.80, 24 3.27,
// 32 4.00; before K was walked backwards, 8 rows 3.41 and 12 rows 3.14;
// grouping by columns instead (8 tile columns, rows inside) read 3.41 GB.
constexpr int kGroupM = 19;

TG_HOST_DEVICE inline void unit_tile(int tiles_m, int tiles_n, long long t, int* tm, int* tn) {
    const long long per_group = (long long)kGroupM * tiles_n;
    const int g = (int)(t / per_group);
    const int first_m = g * kGroupM;
    const int gm = tiles_m - first_m < kGroupM ? tiles_m - first_m : kGroupM;
    const int r = (int)(t - g * per_group);
    *tm = first_m + r % gm;
    *tn = r / gm;
}

// Stream-K tail: every lane's share of the tail is at least this much of K
// (so a partial store is amortised over at least two 256-wide chunks).
constexpr int kTailMinK = 512;
// The 3xTF32 kernel needs most of its operand tiles from L2 (each byte read
// by several CTAs at about the same K): a stream-K tail, whose lanes run at
// different K, keeps that only while the tail's A and B rows fit in L2, so
// larger tails are cut into equal K slices instead (measured on GB300: a
// 96 MiB tail ran as fast stream-K as sliced, a 208 MiB one 3 % slower
// overall and a 512 MiB one 10 %).
constexpr long long kTailL2Bytes = 112ll << 20;

// Whether the 3xTF32 kernel splits raw K-major operands itself (TMA copies of
// the caller's fp32 tile; the raw value is the tensor core's hi operand, since
// kind::tf32 reads only the top 19 bits, and lo is written beside it in shared
// memory).  TG_FUSED_SPLIT=0 keeps the pre-pass for every operand.
bool fused_split_enabled();

struct Plan {
    int M = 0, N = 0, K = 0;
    long long lda = 0, ldb = 0, ldc = 0;
    int op_a = TG_OP_N, op_b = TG_OP_N;  // stored A / B transposed (TG_OP_T)
    float alpha = 1.0f, beta = 0.0f;      // C = alpha * op(A) op(B) + beta * C
    int path = TG_PATH_TF32X3;
    int split = 1;
    int bm = 0, bn = 0, bk = 0, stages = 0;
    int tiles_m = 0, tiles_n = 0;
    int pair = 1;        // 3xTF32: CTAs per cluster on vertically adjacent tiles
    bool pair_mma = false;  // 3xTF32 pairs: one M = 256 product over both CTAs (cta_group::2)
    // tensor paths with the pair MMA: A stored M x K with a 16-byte-aligned
    // base and pitch is staged raw by TMA and split inside the GEMM kernel
    // (no pre-pass copy of it)
    bool raw_a = false;
    long long units = 0; // work units (a unit is `pair` vertically adjacent tiles x one K slice)
    // stream-K tail: the tile units past full_units (tail_units of them) are
    // shared out over tail_lanes lanes, each running an equal share of their
    // K blocks; pieces of a unit go to partial slots, then a tail reduce
    long long full_units = 0;
    long long tail_units = 0;
    int tail_lanes = 0;
    // split point (3xTF32, tails larger than L2 with more than half the lanes
    // busy): the first tail_kx K blocks of tail unit q run on lane q, all
    // units in step; the remaining K blocks of every unit are shared out over
    // the other lanes; tail_slots partial slots per unit (0: runs as above)
    int tail_kx = 0;
    int tail_slots = 0;
    int grid = 0;
    int num_sms = 0;     // SMs planned for
    int nkb = 0;         // K blocks of bk
    int k4 = 0, n4 = 0;  // K and N rounded up to a multiple of 4 (16-byte rows)
    int k16 = 0;         // K rounded up to a multiple of 16 (3xTF32 split rows)
    int a_rows = 0, b_rows = 0;  // 3xTF32: rows of the split tiles (M, N padded to whole tiles)
    bool zero_fill = false;  // K == 0: C = beta * C, nothing else runs
    bool pack_a = false, pack_b = false;  // FFMA: copy an operand to a 16-byte-pitched buffer
    bool vec_c = false;  // C rows start on 16-byte boundaries
    // workspace layout (byte offsets; a region absent from the plan has size 0)
    size_t off_a0 = 0, off_b0 = 0, off_part = 0, off_tail = 0;
    long long ldp = 0;           // partial-product row stride (elements)
    long long part_stride = 0;   // elements between two K-slice partials
    size_t ws_bytes = 0;
    int launches = 0;
    // 3xTF32 only: A's split tiles (a_rows x 2*k16 floats; B^T's, b_rows x
    // 2*k16) live outside the workspace at ext_a (ext_b), planned with external_a
    // (external_b); a_ready (b_ready) = it already holds that operand's split,
    // so the pre-pass skips it (and is not launched if both are).  An operand
    // the kernel splits itself (raw_a) has no split tiles.
    float* ext_a = nullptr;
    float* ext_b = nullptr;
    bool a_ready = false;
    bool b_ready = false;
};

// Argument checks of the C ABI (pure host arithmetic).  With need_pointers
// false (planning only) NULL pointers are accepted and skip the overlap check.
tg_status validate(int op_a, int op_b, int M, int N, int K, const void* A, int lda, const void* B,
                   int ldb, const void* C, int ldc, int path, int split_k, bool need_pointers = true);

// Output blocks of the host-buffer pipeline: pm row blocks (the first of
// `first` rows, the others of `mb`, the last one the remainder); row blocks
// [0, split) are cut into pn column blocks of nb columns (the last ragged),
// the later ones are computed full width (all of B is on the device by then).
// With defer_out the copies of C out wait until every copy in is done (the
// two directions then do not share the host link).
struct HostBlocks {
    int pm = 1, pn = 1, first = 0, mb = 0, nb = 0, split = 1;
    bool defer_out = false;
    double model_ms = 0.0;
    int row0(int i) const { return i == 0 ? 0 : first + (i - 1) * mb; }
    int rows(int i, int M) const {
        const int r = M - row0(i), cap = i == 0 ? first : mb;
        return r < cap ? r : cap;
    }
    int col_blocks(int i) const { return i < split ? pn : 1; }
};
HostBlocks choose_host_blocks(int M, int N, int K, int path, int num_sms);

// Fill `p` for the given call; num_sms > 0.  Assumes validate() passed.
// allow_fuse = false keeps every operand on the pre-pass (raw_a = false), for
// callers that share split tiles between products.
void make_plan(int op_a, int op_b, int M, int N, int K, float alpha, const void* A, int lda,
               const void* B, int ldb, float beta, const void* C, int ldc, int path, int split_k,
               int num_sms, Plan* p, bool external_b = false, bool external_a = false, bool allow_fuse = true);

// Enqueue every kernel of plan `p` on `stream` (defined in tg_kernels.cu).
tg_status launch_plan(const Plan& p, const float* A, const float* B, float* C, void* ws,
                      cudaStream_t stream, cudaEvent_t ev_begin, cudaEvent_t ev_end);

// Device-side error word (defined in tg_kernels.cu).
tg_status read_error_word(cudaStream_t stream, bool clear, unsigned int* value);
tg_status launch_wait_selftest(unsigned int timeout_us, cudaStream_t stream);

// One-time per-device set-up of kernel attributes (tg_kernels.cu).
tg_status prepare_device_kernels();

// Stream-ordered scratch from the library's per-device memory pool
// (tg_api.cpp); for the auxiliary workloads.
tg_status workspace_alloc(size_t bytes, cudaStream_t stream, void** out);
void workspace_free(void* p, cudaStream_t stream);

}  // namespace tg
