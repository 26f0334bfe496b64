// Host planner of the FP32 GEMM: argument checks, path and tile choice,
// split-K choice and workspace layout.  Pure host arithmetic; no CUDA calls.
//
// The tile decomposition follows the pages' tiling scheme ("03 CUDA Shared
// Memory: Tiling, Bank Conflicts, and Reduction", section "Shared Memory와
// Tiling"; PMPP ch. 5 notes §5.3-§5.4): every CTA owns one BM x BN block of C
// and walks K in phases of BK, with ceil(K/BK) phases and zero-filled ghost
// elements past the edges (§5.5).  What differs from the pages is the
// scheduling: CTAs are persistent (one per SM, looping over tiles), because a
// GB300 SM holds one such CTA at a time (the occupancy trade-off of "Occupancy와
// Block 크기", taken at its extreme: few warps, each with much work).
#include <algorithm>
#include <cstdint>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <map>
#include <mutex>
#include <tuple>
#include <vector>

#include "tg_internal.h"

namespace tg {

namespace {

inline long long cdiv(long long a, long long b) { return (a + b - 1) / b; }
inline size_t round_up(size_t a, size_t b) { return (a + b - 1) / b * b; }

bool ranges_overlap(uintptr_t a0, uintptr_t a1, uintptr_t b0, uintptr_t b1) {
    return a0 < b1 && b0 < a1;
}

// Bytes of the 3xTF32 operands (hi/lo copies: 8 bytes per element; raw
// operands split in the kernel: 4) that the last `rem` tile units of the
// raster read.
long long tail_operand_bytes(const Plan& p, long long rem) {
    const int prow = (int)cdiv(p.tiles_m, p.pair);
    const long long units = (long long)prow * p.tiles_n;
    std::vector<int> rows_seen, cols_seen;
    for (long long t = units - rem; t < units; ++t) {
        int tm = 0, tn = 0;
        unit_tile(prow, p.tiles_n, t, &tm, &tn);
        rows_seen.push_back(tm);
        cols_seen.push_back(tn);
    }
    std::sort(rows_seen.begin(), rows_seen.end());
    std::sort(cols_seen.begin(), cols_seen.end());
    rows_seen.erase(std::unique(rows_seen.begin(), rows_seen.end()), rows_seen.end());
    cols_seen.erase(std::unique(cols_seen.begin(), cols_seen.end()), cols_seen.end());
    long long rows = 0, cols = 0;
    for (int i : rows_seen) rows += std::min<long long>((long long)p.pair * p.bm, p.M - (long long)i * p.pair * p.bm);
    for (int j : cols_seen) cols += std::min<long long>(p.bn, p.N - (long long)j * p.bn);
    return (rows * (p.raw_a ? 4 : 8) + cols * 8) * p.k16;
}

// Whether the one-launch tiled path beats the 3xTF32 path's pre-pass, GEMM
// and reduce for this product (see its definition for the measured basis).
bool tiled_is_faster(int M, int N, int K, int num_sms) {
    (void)num_sms;
    return (double)M * N * K <= kTiledMaxMacs && K <= kTiledMaxK;
}

}  // namespace

bool fused_split_enabled() {
    const char* e = std::getenv("TG_FUSED_SPLIT");
    return !(e != nullptr && e[0] == '0');
}

tg_status validate(int op_a, int op_b, int M, int N, int K, const void* A, int lda, const void* B,
                   int ldb, const void* C, int ldc, int path, int split_k, bool need_pointers) {
    if (op_a != TG_OP_N && op_a != TG_OP_T) return TG_ERR_INVALID_VALUE;
    if (op_b != TG_OP_N && op_b != TG_OP_T) return TG_ERR_INVALID_VALUE;
    if (M < 0 || N < 0 || K < 0) return TG_ERR_INVALID_VALUE;
    // stored shapes: A is M x K (op N) or K x M (op T); B is K x N or N x K
    const int a_rows = op_a == TG_OP_N ? M : K, a_cols = op_a == TG_OP_N ? K : M;
    const int b_rows = op_b == TG_OP_N ? K : N, b_cols = op_b == TG_OP_N ? N : K;
    if (lda < std::max(1, a_cols) || ldb < std::max(1, b_cols) || ldc < std::max(1, N))
        return TG_ERR_INVALID_VALUE;
    if (path != TG_PATH_AUTO && path != TG_PATH_FFMA && path != TG_PATH_TF32X3 && path != TG_PATH_TILED &&
        path != TG_PATH_TF32_BF16)
        return TG_ERR_INVALID_VALUE;
    if (split_k < 0) return TG_ERR_INVALID_VALUE;
    if (M == 0 || N == 0) return TG_OK;  // nothing is read or written
    if (!need_pointers && (A == nullptr || B == nullptr || C == nullptr)) return TG_OK;
    if (C == nullptr) return TG_ERR_INVALID_VALUE;
    if (K > 0 && (A == nullptr || B == nullptr)) return TG_ERR_INVALID_VALUE;
    // C must not overlap the operands (checked on the address ranges spanned)
    const uintptr_t c0 = reinterpret_cast<uintptr_t>(C);
    const uintptr_t c1 = c0 + 4ull * ((unsigned long long)(M - 1) * ldc + N);
    if (K > 0) {
        const uintptr_t a0 = reinterpret_cast<uintptr_t>(A);
        const uintptr_t a1 = a0 + 4ull * ((unsigned long long)(a_rows - 1) * lda + a_cols);
        const uintptr_t b0 = reinterpret_cast<uintptr_t>(B);
        const uintptr_t b1 = b0 + 4ull * ((unsigned long long)(b_rows - 1) * ldb + b_cols);
        if (ranges_overlap(c0, c1, a0, a1) || ranges_overlap(c0, c1, b0, b1))
            return TG_ERR_INVALID_VALUE;
    }
    return TG_OK;
}

void make_plan(int op_a, int op_b, int M, int N, int K, float alpha, const void* A, int lda,
               const void* B, int ldb, float beta, const void* C, int ldc, int path, int split_k,
               int num_sms, Plan* p, bool external_b, bool external_a, bool allow_fuse) {
    *p = Plan{};
    p->M = M;
    p->N = N;
    p->K = K;
    p->lda = lda;
    p->ldb = ldb;
    p->ldc = ldc;
    p->op_a = op_a;
    p->op_b = op_b;
    p->alpha = alpha;
    p->beta = beta;
    p->num_sms = num_sms;
    if (path == TG_PATH_FFMA || path == TG_PATH_TILED || path == TG_PATH_TF32_BF16)
        p->path = path;
    else if (path == TG_PATH_AUTO && split_k <= 1 && tiled_is_faster(M, N, K, num_sms))
        p->path = TG_PATH_TILED;
    else
        p->path = TG_PATH_TF32X3;
    p->vec_c = C != nullptr && (reinterpret_cast<uintptr_t>(C) % 16 == 0) && (ldc % 4 == 0);
    if (tensor_path(p->path)) {
        p->bm = kTf32BM; p->bn = kTf32BN; p->bk = kTf32BK; p->stages = kTf32Stages;
    } else if (p->path == TG_PATH_FFMA) {
        p->bm = kFfmaBM; p->bn = kFfmaBN; p->bk = kFfmaBK; p->stages = kFfmaStages;
    } else {
        p->bm = kTiledBM; p->bn = kTiledBN; p->bk = kTiledBK; p->stages = 2;
    }
    p->k4 = (int)round_up((size_t)K, 4);
    p->k16 = (int)round_up((size_t)K, 16);
    p->n4 = (int)round_up((size_t)N, 4);
    if (M == 0 || N == 0) {
        p->launches = 0;
        return;
    }
    if (K == 0) {  // the empty sum: C = beta * C, one kernel
        p->zero_fill = true;
        p->split = 1;
        p->launches = 1;
        return;
    }
    p->tiles_m = (int)cdiv(M, p->bm);
    p->tiles_n = (int)cdiv(N, p->bn);
    p->nkb = (int)cdiv(K, p->bk);
    const long long tiles = (long long)p->tiles_m * p->tiles_n;
    if (p->path == TG_PATH_TILED) {
        // one block per tile and K slice.  K is split when the tiles would
        // leave more than half the SMs idle and K has at least 8 blocks of 16,
        // into as many slices as keep one block per SM, each at least two
        // 16-wide stages, at most 8 (256^3: 16 tiles x 8 slices).  The
        // slices of a tile run as one cluster and add their partials in
        // shared memory: still one launch, no workspace
        int S = 1;
        if (split_k > 0)
            S = std::min(split_k, p->nkb);
        else if (tiles < num_sms / 2 && p->nkb >= 8)
            S = (int)std::max<long long>(1, std::min<long long>({(long long)num_sms / tiles, (long long)p->nkb / 2,
                                                                 (long long)kTiledMaxSplit}));
        S = std::min(S, kTiledMaxSplit);
        p->split = S;
        p->units = tiles * S;
        p->full_units = p->units;
        p->grid = (int)std::min<long long>(p->units, 0x7fffffffLL);
        p->launches = 1;
        return;
    }

    // 3xTF32: two CTAs of a cluster take vertically adjacent tiles; the
    // pair's first CTA issues one M = 256 product over both (cta_group::2),
    // each CTA holding its A tile and half of the shared B tile, which halves
    // the B traffic from L2.  TG_TF32X3_PAIR=0 turns this off.
    const char* pair_env = std::getenv("TG_TF32X3_PAIR");
    const bool pair_off = pair_env != nullptr && std::strcmp(pair_env, "0") == 0;
    p->pair = (tensor_path(p->path) && p->tiles_m >= 2 && num_sms >= 2 && !pair_off) ? 2 : 1;
    if (tensor_path(p->path)) {
        // split tiles of 128 rows x (16 hi + 16 lo): A's rows padded to whole
        // units (pair x 128), B^T's to whole 256-row B tiles
        p->a_rows = (int)round_up((size_t)M, 128 * (size_t)p->pair);
        p->b_rows = (int)round_up((size_t)N, 256);
        // CTA pairs issue one M = 256 product over both CTAs unless
        // TG_TF32X3_PAIRMMA=0, or the tile arrays' row coordinates (32-bit in
        // the tensor maps) would overflow
        const char* pm_env = std::getenv("TG_TF32X3_PAIRMMA");
        const long long kbs = p->k16 / 16;
        p->pair_mma = p->pair == 2 && !(pm_env != nullptr && pm_env[0] == '0') &&
                      (long long)p->a_rows * kbs < (1ll << 31) && (long long)p->b_rows * kbs < (1ll << 31);
        // raw A: stored M x K (K-major), base and row pitch on 16-byte
        // boundaries (TMA), pair-MMA tensor kernel (3xTF32 or the tf32 +
        // bf16 variant).  B always takes the pre-pass (see tg_kernels.cu:
        // two operands split in the kernel measured slower than the
        // pre-pass of one)
        const bool fuse = allow_fuse && p->pair_mma && fused_split_enabled();
        p->raw_a = fuse && op_a == TG_OP_N && A != nullptr && reinterpret_cast<uintptr_t>(A) % 16 == 0 &&
                   lda % 4 == 0;
    }
    // Split K when the tile units alone would leave most lanes (CTAs, or CTA
    // pairs) idle, into as many slices as keep every unit in one round of
    // the lanes: each slice keeps at least 4 K blocks, at most 16 slices.
    // (Counting 128 x 256 tiles against all SMs instead planned 777 x 1029 x
    // 513 as 20 pair units x 4 slices = 80 units on 76 pairs: a second round
    // for 4 units.)
    const long long tile_units = cdiv(p->tiles_m, p->pair) * (long long)p->tiles_n;
    const long long lanes = num_sms / p->pair;
    int S = 1;
    if (split_k > 0) {
        S = std::min(split_k, p->nkb);
    } else if (tile_units < lanes / 2 && p->nkb >= 8) {
        long long s = std::min<long long>({lanes / tile_units, (long long)p->nkb / 4, 16});
        S = (int)std::max<long long>(1, s);
    }
    p->split = S;
    p->units = tile_units * S;
    const long long cap = num_sms / p->pair;  // units in flight at once (lanes)
    p->grid = p->pair * (int)std::min<long long>(p->units, cap);
    p->full_units = p->units;

    // Balancing the last round.  When the units do not divide into whole
    // rounds of the lanes (or there are fewer units than lanes), the last
    // round would leave lanes idle.  Instead its rem units (the tail) are
    // shared out over L lanes: lane v runs K blocks [v*T/L, (v+1)*T/L) of the
    // tail's T = rem * nkb K blocks laid end to end.  A run that holds a whole
    // unit stores it to C; a part of a unit goes to a partial slot that the
    // tail reduce adds up in lane order.
    //  * stream-K (FFMA, and 3xTF32 while the tail's A and B rows fit in L2):
    //    L = every lane, each share at least kTailMinK of K;
    //  * equal K slices (3xTF32, larger tails): L = rem * ts, so each run is
    //    one of ts equal K slices of one unit and the runs of a slice stay
    //    at the same K across units (ts <= 4, each slice >= 8 K blocks, only
    //    when that at least halves the last round);
    //  * split point (3xTF32, larger tails filling more than half the lanes):
    //    lane q < rem runs the first kx = rem * nkb / L K blocks of unit q,
    //    all in step, and the other E = L - rem lanes share the remaining
    //    nkb - kx blocks of every unit as runs laid end to end (each share at
    //    least kTailMinK of K), so every lane gets about kx blocks.  The
    //    reduce adds each unit's first part and its remainder's pieces.
    // Taken when it shortens the last round by at least 10 %; only with the
    // automatic split and no K split.
    if (split_k == 0 && S == 1) {
        const long long rem = p->units % cap;
        const long long min_share = std::max<long long>(1, kTailMinK / p->bk);
        if (rem > 0) {
            long long L = 0, kx = 0, slots = 0;
            if (p->path == TG_PATH_FFMA || tail_operand_bytes(*p, rem) <= kTailL2Bytes) {
                L = std::min<long long>(cap, rem * p->nkb / min_share);
            } else if (2 * rem <= cap) {
                long long ts = std::min<long long>(cap / rem, 4);
                while (ts > 1 && p->nkb < 8 * ts) --ts;
                L = rem * ts;
            } else {
                for (long long E = cap - rem; E > 0; --E) {
                    const long long l = rem + E, x = rem * p->nkb / l;
                    const long long share = rem * (p->nkb - x) / E;
                    if (x > 0 && x < p->nkb && share >= min_share) {
                        L = l;
                        kx = x;
                        // lanes meeting one unit's remainder: at most ceil(rl / share) + 1
                        slots = 1 + (p->nkb - x + share - 1) / share + 1;
                        break;
                    }
                }
            }
            const bool better = kx > 0 ? 10 * kx <= 9 * p->nkb : (L > rem && 10 * rem <= 9 * L);
            if (L > 0 && better) {
                p->full_units = p->units - rem;
                p->tail_units = rem;
                p->tail_lanes = (int)L;
                p->tail_kx = (int)kx;
                p->tail_slots = (int)slots;
                p->grid = p->pair * (int)std::max<long long>(std::min<long long>(p->units, cap), L);
            }
        }
    }

    size_t off = 0;
    auto take = [&](size_t bytes) {
        size_t at = off;
        off = round_up(off + bytes, kWsAlign);
        return at;
    };
    if (tensor_path(p->path)) {
        // the split tiles of each operand not split in the kernel, unless the
        // caller provides them
        if (!external_a && !p->raw_a) p->off_a0 = take(8ull * p->a_rows * p->k16);
        if (!external_b) p->off_b0 = take(8ull * p->b_rows * p->k16);
    } else {
        // TMA reads the operands in place when they are stored untransposed,
        // their base is 16-byte aligned and their row pitch a multiple of 16
        // bytes; otherwise a pre-pass copies them (transposing a transposed
        // one) to a padded buffer (A: [M][k4], B: [K][n4]).
        p->pack_a = op_a == TG_OP_T || A == nullptr || (reinterpret_cast<uintptr_t>(A) % 16 != 0) ||
                    (lda % 4 != 0);
        p->pack_b = op_b == TG_OP_T || B == nullptr || (reinterpret_cast<uintptr_t>(B) % 16 != 0) ||
                    (ldb % 4 != 0);
        if (p->pack_a) p->off_a0 = take(4ull * M * p->k4);
        if (p->pack_b) p->off_b0 = take(4ull * K * p->n4);
    }
    if (S > 1) {
        p->ldp = p->n4;
        p->part_stride = (long long)M * p->n4;
        p->off_part = take(4ull * S * M * p->n4);
    }
    if (p->tail_lanes > 0) {  // stream-K: two slots per lane (its first and last piece)
        const size_t slots = p->tail_kx > 0 ? (size_t)p->tail_units * p->tail_slots : 2ull * p->tail_lanes;
        p->off_tail = take(4ull * slots * p->pair * p->bm * p->bn);
    }
    p->ws_bytes = off;
    const bool prepass = tensor_path(p->path) || p->pack_a || p->pack_b;
    p->launches = (prepass ? 1 : 0) + 1 + (S > 1 ? 1 : 0) + (p->tail_lanes > 0 ? 1 : 0);
}

// Modelled duration (seconds) of one planned product: its rounds of work
// units over the lanes (whole rounds, plus the tail's share of a unit per
// lane), each unit taking its tile's flops at the path's per-lane rate, plus
// a fixed 35 us per product (pipeline fill and drain, reduce, launch gaps
// and the host's own issue of the product's copies and launches; fitted on
// GB300 to 80 measured 8192^3 host-buffer layouts, RMS error 0.04 ms).
double product_seconds(const Plan& p, double rate) {
    if (p.M == 0 || p.N == 0 || p.K == 0) return 5e-6;
    const long long lanes = std::max(1, p.grid / p.pair);
    double rounds;
    if (p.tail_lanes > 0)
        rounds = (double)(p.full_units / lanes) + (double)p.tail_units / p.tail_lanes;
    else
        rounds = (double)cdiv(p.units, lanes);
    const double unit_flops = 2.0 * p.pair * p.bm * p.bn * ((double)p.K / p.split);
    return rounds * unit_flops / (rate / std::max(1, p.num_sms / p.pair)) + 35e-6;
}

// Host-buffer pipeline model: a small event simulation of one call.  Copies
// in run on one copy stream in the order the products first need them (A_0,
// B_0, B_1, ..., A_1, ...); the products run in row-block-major order on the
// compute stream, each once its A row block and B column block (all of B for
// a full-width one) are in; each C block is copied out on a second copy
// stream once its product is done (with defer_out, not before the last copy
// in).  Rates measured on GB300 over NVLink-C2C with pinned host memory:
// 205 GB/s in alone, 190 GB/s out alone, about 150 GB/s each way while both
// directions are busy, plus ~40 us per copy out that does not start right
// behind another (a queued copy out follows the previous one without it:
// with this term the model ranks the layouts whose copies out wait for the
// last copy in correctly; without it, it put them up to 0.33 ms too slow);
// the split pre-pass about 5.7 TB/s; a full round of work units 375 (3xTF32,
// A split in the kernel; products inside the pipeline are smaller than a
// whole call) or 62 (FFMA) useful TFLOP/s.  Fitted to 80 measured 8192^3
// layouts, RMS error 0.04 ms; its choice was the measured best within
// 0.1 %.
namespace {

struct HostCopy {
    double bytes;
    int a_block, b_block;  // which block it brings in (-1: none)
};
struct HostProduct {
    int a_block, b_block;  // inputs it waits for
    double seconds, out_bytes;
};

double simulate_host_pipeline(const std::vector<HostCopy>& ins, const std::vector<HostProduct>& prods, int pm,
                              int pn, bool defer_out) {
    const double r_in = 205e9, r_out = 190e9, r_both = 150e9, out_fixed_bytes = 40e-6 * 190e9;
    std::vector<char> a_in(pm, 0), b_in(pn, 0);
    size_t ik = 0, pk = 0, oh = 0;
    double t = 0.0, in_rem = ins.empty() ? 0.0 : ins[0].bytes, gpu_end = -1.0, out_rem = -1.0;
    std::vector<double> outq;
    double out_done = -1.0;  // when the last copy out ended
    for (int iter = 0; iter < 100000; ++iter) {
        if (gpu_end < 0.0 && pk < prods.size() && a_in[prods[pk].a_block] && b_in[prods[pk].b_block])
            gpu_end = t + prods[pk].seconds;
        if (out_rem < 0.0 && oh < outq.size() && (!defer_out || ik >= ins.size()))
            out_rem = outq[oh++] + (out_done == t ? 0.0 : out_fixed_bytes);
        const bool in_busy = ik < ins.size(), out_busy = out_rem >= 0.0;
        if (!in_busy && !out_busy && gpu_end < 0.0) return pk == prods.size() ? t : 1e30;
        const double ri = in_busy ? (out_busy ? r_both : r_in) : 0.0;
        const double ro = out_busy ? (in_busy ? r_both : r_out) : 0.0;
        double dt = 1e30;
        if (in_busy) dt = std::min(dt, in_rem / ri);
        if (out_busy) dt = std::min(dt, out_rem / ro);
        if (gpu_end >= 0.0) dt = std::min(dt, gpu_end - t);
        dt = std::max(dt, 0.0);
        t += dt;
        if (in_busy) {
            in_rem -= ri * dt;
            if (in_rem <= 1.0) {
                if (ins[ik].a_block >= 0) a_in[ins[ik].a_block] = 1;
                if (ins[ik].b_block >= 0) b_in[ins[ik].b_block] = 1;
                if (++ik < ins.size()) in_rem = ins[ik].bytes;
            }
        }
        if (out_busy) {
            out_rem -= ro * dt;
            if (out_rem <= 1.0) {
                out_rem = -1.0;
                out_done = t;
            }
        }
        if (gpu_end >= 0.0 && gpu_end <= t + 1e-12) {
            outq.push_back(prods[pk++].out_bytes);
            gpu_end = -1.0;
        }
    }
    return 1e30;
}

}  // namespace

// Modelled time of host calls of one shape, for any blocks.
class HostModel {
  public:
    HostModel(int M, int N, int K, int path, int num_sms)
        : M_(M), N_(N), K_(K), path_(path), sms_(num_sms), tf32_(path != TG_PATH_FFMA) {}

    double ms(const HostBlocks& hb) {
        const double bw_split = 5.7e12;
        ins_.clear();
        prods_.clear();
        ins_.push_back({4.0 * hb.rows(0, M_) * K_, 0, -1});
        for (int j = 0; j < hb.pn; ++j) ins_.push_back({4.0 * std::min(hb.nb, N_ - j * hb.nb) * K_, -1, j});
        for (int i = 1; i < hb.pm; ++i) ins_.push_back({4.0 * hb.rows(i, M_) * K_, i, -1});
        for (int i = 0; i < hb.pm; ++i) {
            const int rows = hb.rows(i, M_), nc = hb.col_blocks(i);
            for (int j = 0; j < nc; ++j) {
                const int cols = nc == 1 ? N_ : std::min(hb.nb, N_ - j * hb.nb);
                double sec = product(rows, cols);
                if (tf32_) {  // the split passes: A_i's only when the kernel does not split it
                    if (j == 0 && !raw_a(rows, cols)) sec += 12.0 * rows * K_ / bw_split;
                    if (i == 0) sec += 12.0 * cols * K_ / bw_split;
                }
                prods_.push_back({i, nc == 1 ? hb.pn - 1 : j, sec, 4.0 * rows * cols});
            }
        }
        return simulate_host_pipeline(ins_, prods_, hb.pm, hb.pn, hb.defer_out) * 1e3;
    }

  private:
    Plan plan(int rows, int cols) const {
        const void* al = reinterpret_cast<const void*>(static_cast<uintptr_t>(1) << 20);
        const int k4 = (int)round_up((size_t)std::max(K_, 1), 4), n4 = (int)round_up((size_t)std::max(N_, 1), 4);
        Plan pl;
        make_plan(TG_OP_N, TG_OP_N, rows, cols, K_, 1.0f, al, k4, al, n4, 0.0f, al, n4, path_, 0, sms_, &pl,
                  tf32_, tf32_);
        return pl;
    }
    // (modelled seconds, whether the kernel splits A itself) of one product
    const std::pair<double, bool>& product_info(int rows, int cols) {
        auto it = product_s_.find({rows, cols});
        if (it != product_s_.end()) return it->second;
        const Plan pl = plan(rows, cols);
        const double t = product_seconds(pl, path_ == TG_PATH_TF32_BF16 ? 525e12 : (tf32_ ? 375e12 : 62e12));
        return product_s_[{rows, cols}] = {t, pl.raw_a};
    }
    double product(int rows, int cols) { return product_info(rows, cols).first; }
    bool raw_a(int rows, int cols) { return product_info(rows, cols).second; }
    int M_, N_, K_, path_, sms_;
    bool tf32_;
    std::map<std::pair<int, int>, std::pair<double, bool>> product_s_;  // by (rows, columns)
    std::vector<HostCopy> ins_;
    std::vector<HostProduct> prods_;
};

HostBlocks model_host_blocks(int M, int N, int K, int path, int num_sms) {
    HostBlocks best;
    best.mb = best.first = (int)round_up((size_t)std::max(M, 1), 128);
    best.nb = (int)round_up((size_t)std::max(N, 1), 256);
    best.model_ms = -1.0;
    if (M == 0 || N == 0) return best;
    // below 2^33 multiply-adds one block: the launches would cost more than
    // the copies they hide, and the result is then bit-identical to tg_sgemm's
    const int max_blocks = (double)M * N * K >= 8589934592.0 ? 8 : 1;
    HostModel model(M, N, K, path, num_sms);
    auto evaluate = [&](int pm, int first, int mb, int pn, int nb, int split) {
        HostBlocks hb;
        hb.pm = pm;
        hb.pn = pn;
        hb.first = first;
        hb.mb = mb;
        hb.nb = nb;
        hb.split = split;
        for (int defer = 0; defer < 2; ++defer) {
            hb.defer_out = defer != 0;
            hb.model_ms = model.ms(hb);
            // candidates come simplest first; a later one must win by 0.5 %
            if (best.model_ms < 0.0 || hb.model_ms < best.model_ms * 0.995) best = hb;
        }
    };
    // B column blocks are strided copies; on GB300 rows of a multiple of 4 KiB
    // copied at the full rate (8 KiB: 185-208 GB/s) while 6 KiB rows ran at
    // 140-200 and 2 KiB rows at 117, so wide B keeps to 1024-column blocks
    const int nb_align = N >= 4096 ? 1024 : 256;
    for (int pn = 1; pn <= max_blocks; ++pn) {
        const int nb = (int)round_up((size_t)cdiv(N, pn), nb_align);
        if (cdiv(N, nb) != pn || (pn > 1 && nb < 512)) continue;
        // equal row blocks, every row block cut into the column blocks
        for (int pm = 1; pm <= max_blocks; ++pm) {
            const int mb = (int)round_up((size_t)cdiv(M, pm), 128);
            if (cdiv(M, mb) == pm && (pm == 1 || mb >= 512)) evaluate(pm, mb, mb, pn, nb, pm);
        }
        if (max_blocks == 1) continue;
        // a first row block of `first` rows (the first product starts once it
        // and B_0 are in), then blocks of mb rows and a shorter remainder;
        // only the first row block cut into column blocks, or all of them
        for (int first = 256; first < M && first <= 4096; first += 256) {
            const int lo = std::max(512, (int)round_up((size_t)cdiv(M - first, max_blocks - 1), 256));
            for (int mb = lo; mb <= lo + 4096 && mb < M; mb += 256) {
                const int pm = 1 + cdiv(M - first, mb);
                if (pm > max_blocks) continue;
                evaluate(pm, first, mb, pn, nb, 1);
                if (pn > 1) evaluate(pm, first, mb, pn, nb, pm);
            }
        }
    }
    return best;
}

// TG_HOST_BLOCKS="first,mb,nb,split[,defer_out]" fixes the blocks (for tests
// of each layout); ignored unless it describes at most 8 x 8 valid blocks of C.
bool host_blocks_override(int M, int N, HostBlocks* hb) {
    const char* e = std::getenv("TG_HOST_BLOCKS");
    int first = 0, mb = 0, nb = 0, split = 0, defer = 0;
    if (e == nullptr || std::sscanf(e, "%d,%d,%d,%d,%d", &first, &mb, &nb, &split, &defer) < 4) return false;
    if (M <= 0 || N <= 0 || first <= 0 || mb <= 0 || nb <= 0 || first % 128 || mb % 128 || nb % 256) return false;
    const int pm = first >= M ? 1 : 1 + cdiv(M - first, mb), pn = cdiv(N, nb);
    if (pm > 8 || pn > 8 || split < 1 || split > pm) return false;
    hb->pm = pm;
    hb->pn = pn;
    hb->first = first;
    hb->mb = mb;
    hb->nb = nb;
    hb->split = split;
    hb->defer_out = defer != 0;
    return true;
}

// The model's answer is remembered per shape (a few thousand layouts are
// evaluated on first use; later calls with the same shape only look it up).
HostBlocks choose_host_blocks(int M, int N, int K, int path, int num_sms) {
    HostBlocks fixed;
    if (host_blocks_override(M, N, &fixed)) {
        fixed.model_ms = HostModel(M, N, K, path, num_sms).ms(fixed);
        return fixed;
    }
    static std::mutex mu;
    static std::map<std::tuple<int, int, int, int, int>, HostBlocks> memo;
    const auto key = std::make_tuple(M, N, K, path, num_sms);
    {
        std::lock_guard<std::mutex> lock(mu);
        auto it = memo.find(key);
        if (it != memo.end()) return it->second;
    }
    const HostBlocks hb = model_host_blocks(M, N, K, path, num_sms);
    std::lock_guard<std::mutex> lock(mu);
    if (memo.size() > 4096) memo.clear();
    memo[key] = hb;
    return hb;
}

}  // namespace tg
