// sm_103a kernels of the row-major FP32 GEMM C = A x B and their launchers.
//
// The method is the pages' shared-memory tiling ("03 CUDA Shared Memory:
// Tiling, Bank Conflicts, and Reduction", "Shared Memory와 Tiling"; PMPP ch. 5
// notes §5.3-§5.5), rebuilt for Blackwell:
//  * a CTA owns one output tile and walks K in phases; the tiles of A and B of
//    a phase are staged in shared memory by TMA instead of by the threads;
//  * out-of-range parts of a tile are the pages' ghost elements: TMA fills
//    them with zeros, and only the final store is range-checked;
//  * the pages' two __syncthreads() per phase (one so the tile is complete
//    before it is read, one so nobody overwrites a tile still being read)
//    become two mbarriers per pipeline stage, "full" and "empty", so several
//    phases are in flight at once;
//  * the loading threads are one producer warp; the math warps never load
//    from global memory (warp-uniform role split by warp index, as in the
//    pages' divergence-free branching by warp number).
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>
#include <nvtx3/nvToolsExt.h>

#include <cstdint>
#include <cstdlib>
#include <cstring>
#include <mutex>
#include <utility>

#include "tg_internal.h"
#include "tg_ptx.cuh"

namespace tg {

// Per-device error word: 0, or the site code of the first bounded wait that
// gave up.  Shared by every kernel and stream of this library on the device.
__device__ unsigned int g_error_word;

enum : uint32_t {
    kSiteFfmaProducer = 0x101,
    kSiteFfmaConsumer = 0x102,
    kSiteTfProducer = 0x201,
    kSiteTfMmaSmem = 0x202,
    kSiteTfMmaTmem = 0x203,
    kSiteTfEpilogue = 0x204,
    kSiteTfSplit = 0x205,
    kSiteSelftest = 0x301,
};

// ------------------------------------------------------------ shared bits

struct GemmArgs {
    int M, N, K;
    int tiles_m, tiles_n;    // tiles_m counts rows of `pair` tiles
    int pair;                // CTAs per cluster sharing a B tile (1 or 2)
    int split, nkb;
    long long units;
    float* out;              // C (split == 1) or the first K-slice partial
    // 3xTF32: the operands' split copies as 16 KiB tiles (see the pre-pass)
    const float* a_tiles;
    const float* b_tiles;
    int kbs;                 // K blocks per tile row of tiles
    long long ldo;           // row stride of `out`
    long long slice_stride;  // elements between K-slice partials
    int vec_out;             // rows of `out` start on 16-byte boundaries
    // balanced last round: the tail_units tile units after full_units are
    // shared out over tail_lanes lanes (see work_item).  tail_kx == 0: runs
    // of the units laid end to end, pieces to partial slot 2*lane (a lane's
    // first piece) or 2*lane + 1 (its last); tail_kx > 0: unit q's first
    // tail_kx K blocks on lane q (slot q*tail_slots), the rest of every unit
    // over the other lanes (slots q*tail_slots + 1 + i).  Slots are
    // [pair*BM][BN] floats of `tail`.
    long long full_units, tail_units;
    int tail_lanes, tail_kx, tail_slots;
    float* tail;
    // C = alpha * op(A) op(B) + beta * C, applied where C is written (scaled
    // = 0: a plain store of the product; beta == 0: C is not read)
    float alpha, beta;
    int scaled;
    uint64_t timeout_ns;
};

struct Unit {
    int m0, n0, kb0, kb1;
    float* out;
    long long ldo;
    bool direct;  // writes C itself (not a partial)
};

// Work unit u -> (K slice, output tile).  With pair = 2 a unit is two
// vertically adjacent tiles; the CTA of cluster rank `rank` takes tile row
// 2*row + rank.  Units below full_units cover their whole K range (or one of
// `split` K slices).
__device__ __forceinline__ Unit decode_unit(const GemmArgs& a, long long u, int rank, int BM, int BN) {
    const long long tiles = (long long)a.tiles_m * a.tiles_n;
    Unit x;
    int tm, tn;
    const int s = (int)(u / tiles);
    unit_tile(a.tiles_m, a.tiles_n, u - (long long)s * tiles, &tm, &tn);
    x.m0 = (tm * a.pair + rank) * BM;
    x.n0 = tn * BN;
    x.kb0 = (int)((long long)s * a.nkb / a.split);
    x.kb1 = (int)((long long)(s + 1) * a.nkb / a.split);
    x.out = a.out + (long long)s * a.slice_stride;
    x.ldo = a.ldo;
    x.direct = a.split == 1;
    return x;
}

// Stream-K tail arithmetic.  The tail's T = tail_units * nkb K blocks are laid
// end to end (tail unit q holds blocks [q*nkb, (q+1)*nkb)); lane v of the
// tail_lanes runs blocks [v*T/tail_lanes, (v+1)*T/tail_lanes).
__host__ __device__ __forceinline__ long long tail_run_begin(long long v, long long T, long long lanes) {
    return v * T / lanes;
}
// The lane whose run holds K block x of the tail (the last v with begin <= x).
__host__ __device__ __forceinline__ long long tail_lane_of(long long x, long long T, long long lanes) {
    return ((x + 1) * lanes + T - 1) / T - 1;
}

// Work item j of one lane (a CTA, or a CTA pair) of `lanes`, in the order
// the lane runs them: first the whole units lane, lane + lanes, ... below
// full_units; then, for each tail lane v = lane, lane + lanes, ..., the
// pieces of v's run, one per tail unit it meets.  Returns false past the last
// item.  Every role of the CTA walks j = 0, 1, ... and so sees the same
// sequence; only j is carried between items.
// kSplitPoint: the kernel may run a split-point tail (3xTF32); kOut: fill
// out/ldo/direct too (the roles that store; the copy and MMA threads only
// need the tile and its K range).
template <bool kSplitPoint, bool kOut = true>
__device__ __forceinline__ bool work_item(const GemmArgs& a, long long lane, long long lanes, long long j,
                                          int rank, int BM, int BN, Unit* x) {
    const long long nfull = a.full_units > lane ? (a.full_units - lane + lanes - 1) / lanes : 0;
    if (j < nfull) {
        *x = decode_unit(a, lane + j * lanes, rank, BM, BN);
        return true;
    }
    j -= nfull;
    const long long blk = (long long)a.pair * BM * BN;
    int tm, tn;
    if (kSplitPoint && a.tail_kx > 0) {  // split point: lockstep first parts, the rest spread out
        const long long U = a.tail_units, E = a.tail_lanes - U, rl = a.nkb - a.tail_kx, R = U * rl;
        for (long long v = lane; v < a.tail_lanes; v += lanes) {
            if (v < U) {
                if (j > 0) {
                    --j;
                    continue;
                }
                unit_tile(a.tiles_m, a.tiles_n, a.full_units + v, &tm, &tn);
                x->m0 = (tm * a.pair + rank) * BM;
                x->n0 = tn * BN;
                x->kb0 = 0;
                x->kb1 = a.tail_kx;
                if (kOut) {
                    x->direct = false;
                    x->out = a.tail + v * a.tail_slots * blk - (long long)tm * blk - x->n0;
                    x->ldo = BN;
                }
                return true;
            }
            const long long e = v - U;
            const long long s = tail_run_begin(e, R, E), t = tail_run_begin(e + 1, R, E);
            if (s >= t) continue;
            const long long q0 = s / rl, pieces = (t - 1) / rl - q0 + 1;
            if (j >= pieces) {
                j -= pieces;
                continue;
            }
            const long long q = q0 + j, b0 = q * rl;
            unit_tile(a.tiles_m, a.tiles_n, a.full_units + q, &tm, &tn);
            x->m0 = (tm * a.pair + rank) * BM;
            x->n0 = tn * BN;
            x->kb0 = a.tail_kx + (int)((s > b0 ? s : b0) - b0);
            x->kb1 = a.tail_kx + (int)((t < b0 + rl ? t : b0 + rl) - b0);
            if (kOut) {
                x->direct = false;
                const long long slot = q * a.tail_slots + 1 + (e - tail_lane_of(b0, R, E));
                x->out = a.tail + slot * blk - (long long)tm * blk - x->n0;
                x->ldo = BN;
            }
            return true;
        }
        return false;
    }
    const long long T = a.tail_units * a.nkb;
    for (long long v = lane; v < a.tail_lanes; v += lanes) {
        const long long s = tail_run_begin(v, T, a.tail_lanes);
        const long long e = tail_run_begin(v + 1, T, a.tail_lanes);
        if (s >= e) continue;
        const long long q0 = s / a.nkb, pieces = (e - 1) / a.nkb - q0 + 1;
        if (j >= pieces) {
            j -= pieces;
            continue;
        }
        const long long q = q0 + j, b0 = q * a.nkb;
        unit_tile(a.tiles_m, a.tiles_n, a.full_units + q, &tm, &tn);
        x->m0 = (tm * a.pair + rank) * BM;
        x->n0 = tn * BN;
        x->kb0 = (int)((s > b0 ? s : b0) - b0);
        x->kb1 = (int)((e < b0 + a.nkb ? e : b0 + a.nkb) - b0);
        if (kOut) {
            x->direct = x->kb0 == 0 && x->kb1 == a.nkb;
            if (x->direct) {  // the run holds the whole unit: C itself
                x->out = a.out;
                x->ldo = a.ldo;
            } else {  // this slot's [pair*BM][BN] block, addressed with global row/column
                const long long slot = 2 * v + (j == 0 ? 0 : 1);
                x->out = a.tail + slot * blk - (long long)tm * blk - x->n0;
                x->ldo = BN;
            }
        }
        return true;
    }
    return false;
}

// Store 4 consecutive values of one output row starting at column `col`,
// range-checked against N (the pages' guarded final store).
__device__ __forceinline__ void store_row4(float* row, int col, int N, float4 v, bool vec) {
    if (vec && col + 3 < N) {
        *reinterpret_cast<float4*>(row + col) = v;
    } else {
        if (col < N) row[col] = v.x;
        if (col + 1 < N) row[col + 1] = v.y;
        if (col + 2 < N) row[col + 2] = v.z;
        if (col + 3 < N) row[col + 3] = v.w;
    }
}

// The 4 values of C at row[col..col+3] (guarded like store_row4; zero past N).
__device__ __forceinline__ float4 load_row4_c(const float* row, int col, int N, bool vec) {
    if (vec && col + 3 < N) return *reinterpret_cast<const float4*>(row + col);
    return make_float4(col < N ? row[col] : 0.0f, col + 1 < N ? row[col + 1] : 0.0f,
                       col + 2 < N ? row[col + 2] : 0.0f, col + 3 < N ? row[col + 3] : 0.0f);
}

// alpha * v + beta * c (c ignored when beta == 0, so C may hold anything).
__device__ __forceinline__ float4 scale4(float4 v, float4 c, float alpha, float beta) {
    if (beta != 0.0f)
        return make_float4(fmaf(alpha, v.x, beta * c.x), fmaf(alpha, v.y, beta * c.y), fmaf(alpha, v.z, beta * c.z),
                           fmaf(alpha, v.w, beta * c.w));
    return make_float4(alpha * v.x, alpha * v.y, alpha * v.z, alpha * v.w);
}

// The final value alpha * v + beta * C of 4 consecutive outputs (C read only
// when beta != 0), then the guarded store.
__device__ __forceinline__ void store_row4_scaled(float* row, int col, int N, float4 v, bool vec,
                                                  float alpha, float beta) {
    const float4 c = beta != 0.0f ? load_row4_c(row, col, N, vec) : make_float4(0.f, 0.f, 0.f, 0.f);
    store_row4(row, col, N, scale4(v, c, alpha, beta), vec);
}

__device__ __forceinline__ uint8_t* align_smem_1024(uint8_t* raw) {
    const uint32_t a = smem_addr(raw);
    return raw + ((1024u - (a & 1023u)) & 1023u);
}

// ---------------------------------------------------------------- FFMA path
//
// CTA tile 128 x 256, K phase 32, 384 threads = 3 warpgroups.  Warpgroup 0
// is the producer (one thread issues the TMA loads); warpgroups 1-2 (math
// warps 0-7) do the math.  Each math thread keeps an 8 x 16 block of C in registers
// (register tiling: "Occupancy와 Block 크기" and PMPP ch. 6 coarsening): per
// k it reads 8 values of A and 16 of B from shared memory and performs 128
// FMAs as 64 packed fma.rn.f32x2 (two lanes of fp32 per instruction, same
// rounding as fmaf), which leaves issue slots for the shared-memory loads.
//
// Shared-memory layouts and banks ("Bank Conflict" section):
//  * A tile [128 rows][32 k] arrives with the 128-byte TMA swizzle: the 16-byte
//    chunk c of row r sits at chunk position c ^ (r % 8) -- the pages' XOR
//    swizzle applied to 16-byte words.  A thread's 8 rows are r0 + 4i, so the
//    4 lanes of a warp that read different rows in one instruction read 4
//    consecutive rows -> 4 different chunk positions -> no bank conflict.
//    Lanes sharing a row read the same address (broadcast).
//  * B tile [32 k][256 columns], no swizzle: 8 lanes read 8 consecutive
//    16-byte words of one row (conflict-free), the other lanes broadcast.

// Register budget: launched at kFfmaLaunchRegs per thread (the most 384
// threads may have), the producer warpgroup drops to kFfmaProducerRegs and the
// math warpgroups rise to kFfmaMathRegs; the pool balances exactly:
// 4*32*40 + 8*32*232 = 384*168.  The host refuses to launch a build whose
// register count differs, since an unbalanced raise would wait for ever.
constexpr int kFfmaThreads = 384;
constexpr int kFfmaLaunchRegs = 168, kFfmaProducerRegs = 40, kFfmaMathRegs = 232;
static_assert(4 * 32 * kFfmaProducerRegs + 8 * 32 * kFfmaMathRegs == kFfmaThreads * kFfmaLaunchRegs,
              "setmaxnreg split must balance the launch allocation");
constexpr uint32_t kFfmaAStage = kFfmaBM * kFfmaBK * 4;  // 16 KiB
constexpr uint32_t kFfmaBStage = kFfmaBK * kFfmaBN * 4;  // 32 KiB
constexpr uint32_t kFfmaStageBytes = kFfmaAStage + kFfmaBStage;
constexpr size_t kFfmaSmemBytes = 1024 + (size_t)kFfmaStages * kFfmaStageBytes + 2 * kFfmaStages * 8;

__device__ __forceinline__ float lanef(const float4& v, int i) {
    return i == 0 ? v.x : (i == 1 ? v.y : (i == 2 ? v.z : v.w));
}

__global__ void __launch_bounds__(kFfmaThreads, 1)
    ffma_gemm_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                     GemmArgs args) {
    constexpr int BM = kFfmaBM, BN = kFfmaBN, BK = kFfmaBK, ST = kFfmaStages;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = align_smem_1024(smem_raw);
    float* sA = reinterpret_cast<float*>(smem);
    float* sB = reinterpret_cast<float*>(smem + ST * kFfmaAStage);
    uint64_t* full = reinterpret_cast<uint64_t*>(smem + ST * kFfmaStageBytes);
    uint64_t* empty = full + ST;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const WaitCtl wc{&g_error_word, args.timeout_ns};

    if (threadIdx.x == 0) {
        for (int s = 0; s < ST; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], 8);
        }
        fence_barrier_init();
    }
    __syncthreads();
    grid_dep_wait();  // the operands (or their packed copies) are complete
    grid_dep_launch();

    if (warp < 4) {  // ---------------------------------------- producer
        regs_dec<kFfmaProducerRegs>();
        if (warp == 0 && lane == 0) {
            tma_prefetch_desc(&tmA);
            tma_prefetch_desc(&tmB);
            int stage = 0;
            uint32_t phase = 0, issued = 0, last_par = 0;
            bool ok = true;
            Unit t;
            for (long long j = 0; ok && work_item<false, false>(args, blockIdx.x, gridDim.x, j, 0, BM, BN, &t); ++j) {
                for (int kb = t.kb0; kb < t.kb1; ++kb) {
                    if (!mbar_wait(&empty[stage], phase ^ 1u, wc, kSiteFfmaProducer)) {
                        ok = false;
                        break;
                    }
                    mbar_arrive_expect_tx(&full[stage], kFfmaStageBytes);
                    tma_load_2d(sA + stage * BM * BK, &tmA, &full[stage], kb * BK, t.m0);
                    tma_load_2d(sB + stage * BK * BN, &tmB, &full[stage], t.n0, kb * BK);
                    issued |= 1u << stage;
                    last_par = (last_par & ~(1u << stage)) | (phase << stage);
                    if (++stage == ST) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
            }
            // every copy issued must land before the CTA may exit
            for (int s = 0; s < ST; ++s)
                if ((issued >> s) & 1u) mbar_drain(&full[s], (last_par >> s) & 1u, args.timeout_ns);
        }
        return;
    }

    // ------------------------------------------------------------- math
    regs_inc<kFfmaMathRegs>();
    const int mw = warp - 4;                  // math warp 0..7
    const int wm = mw & 3, wn = mw >> 2;      // warp tile: rows 32*wm.., columns 128*wn..
    const int lm = lane & 3, ln = lane >> 2;  // thread rows wm*32 + lm + 4i, columns 32j + 4ln + q
    int stage = 0;
    uint32_t phase = 0;
    Unit t;
    for (long long j = 0; work_item<false>(args, blockIdx.x, gridDim.x, j, 0, BM, BN, &t); ++j) {
        // acc[i][p] holds columns 32*(p/2) + 4ln + 2*(p%2) + {0, 1} of row i
        unsigned long long acc[8][8];
#pragma unroll
        for (int i = 0; i < 8; ++i)
#pragma unroll
            for (int j = 0; j < 8; ++j) acc[i][j] = 0ull;

        bool ok = true;
        for (int kb = t.kb0; kb < t.kb1; ++kb) {
            const bool got = mbar_wait(&full[stage], phase, wc, kSiteFfmaConsumer);
            if (!__all_sync(0xffffffffu, got)) {
                ok = false;
                break;
            }
            const float* a = sA + stage * BM * BK;
            const float* b = sB + stage * BK * BN + wn * 128 + 4 * ln;
#pragma unroll 1
            for (int kk = 0; kk < BK; kk += 4) {
                float4 av[8];
#pragma unroll
                for (int i = 0; i < 8; ++i) {
                    const int r = wm * 32 + lm + 4 * i;
                    const int chunk = (kk >> 2) ^ (r & 7);
                    av[i] = *reinterpret_cast<const float4*>(a + r * BK + chunk * 4);
                }
                // B as packed pairs: bv[j].x = columns (0,1), .y = (2,3) of chunk j;
                // the next k's fragment is loaded while this k's FMAs run
                ulonglong2 bnext[4];
#pragma unroll
                for (int j = 0; j < 4; ++j) bnext[j] = *reinterpret_cast<const ulonglong2*>(b + kk * BN + 32 * j);
#pragma unroll
                for (int k4 = 0; k4 < 4; ++k4) {
                    ulonglong2 bv[4];
#pragma unroll
                    for (int j = 0; j < 4; ++j) bv[j] = bnext[j];
                    if (k4 < 3) {
#pragma unroll
                        for (int j = 0; j < 4; ++j)
                            bnext[j] = *reinterpret_cast<const ulonglong2*>(b + (kk + k4 + 1) * BN + 32 * j);
                    }
                    // all eight broadcasts first, so no FMA waits on its own splat
                    unsigned long long x2[8];
#pragma unroll
                    for (int i = 0; i < 8; ++i) x2[i] = f32x2_splat(lanef(av[i], k4));
#pragma unroll
                    for (int i = 0; i < 8; ++i) {
#pragma unroll
                        for (int j = 0; j < 4; ++j) {
                            fma_f32x2(acc[i][2 * j], x2[i], bv[j].x);
                            fma_f32x2(acc[i][2 * j + 1], x2[i], bv[j].y);
                        }
                    }
                }
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(&empty[stage]);
            if (++stage == ST) {
                stage = 0;
                phase ^= 1u;
            }
        }
        if (!ok) break;

        // guarded store: 4 rows x 128 contiguous bytes per warp instruction
        const bool vec = args.vec_out != 0;
        const bool scale = args.scaled != 0 && t.direct;
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const int r = t.m0 + wm * 32 + lm + 4 * i;
            if (r < args.M) {
                float* row = t.out + (long long)r * t.ldo;
                // with beta != 0 the row's four old C groups are loaded before
                // any store, so their loads overlap instead of each store
                // waiting for its own load
                const bool read_c = scale && args.beta != 0.0f;
                float4 old[4];
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    const int c = t.n0 + wn * 128 + 32 * j + 4 * ln;
                    old[j] = read_c ? load_row4_c(row, c, args.N, vec) : make_float4(0.f, 0.f, 0.f, 0.f);
                }
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    const int c = t.n0 + wn * 128 + 32 * j + 4 * ln;
                    const float2 lo = f32x2_unpack(acc[i][2 * j]), hi = f32x2_unpack(acc[i][2 * j + 1]);
                    const float4 v = make_float4(lo.x, lo.y, hi.x, hi.y);
                    store_row4(row, c, args.N, scale ? scale4(v, old[j], args.alpha, args.beta) : v, vec);
                }
            }
        }
    }
}

// -------------------------------------------------------------- 3xTF32 path
//
// Operands come from the split pre-pass as 16 KiB tiles: 128 rows of A (or
// of B transposed) x one 16-wide K block, each row 16 hi values then the same
// 16 lo values (128 bytes), already in the 128-byte-swizzled order of the
// tensor core's K-major layout.  A stage is then one copy per 128-row tile
// rather than a TMA box of 128 or 256 separate rows.  Measured on GB300 with
// cycle counters: four boxes of 64-byte rows per stage left the MMA thread
// waiting for data 19 % of the time, two boxes of 128-byte rows 12 %.
// Within a stage the hi slice ks (8 values) starts ks * 32 bytes into each
// row and the lo slice 64 bytes after it.
//
// Two forms.  Pair MMA (the default for CTA pairs): the pair's first CTA
// issues M = 256 products (tcgen05.mma.cta_group::2) whose A rows and B rows
// (N) are split between the two CTAs' shared memory, each CTA holding its A
// tile and its half of B (32 KiB a stage, 6 stages), loaded by 2-D
// tensor-map copies that complete on the first CTA's barrier; each CTA's
// tensor memory holds its 128 rows of the accumulator.  Per-CTA MMA (single
// CTAs, or pairs with the pair MMA off): each CTA issues M = 128 products
// on its A tile and the whole B tile (48 KiB a stage, 4 stages), fetching
// both halves of B itself with plain bulk copies; the two CTAs of a pair
// then share nothing but their cluster rank.
//
// Per 8-wide K slice the MMA thread issues
//     D += A_hi B_lo;  D += A_hi B_hi;  D += A_lo B_hi
// (A_lo B_lo, of relative size 2^-22, is dropped).  In the per-CTA form the
// first two share A_hi, which the tensor core keeps in its A collector
// buffer, so each slice reads A_hi from shared memory once.
//
// Accumulation precision.  The tensor core's fp32 accumulation loses about
// one unit in the last place towards zero per MMA instead of rounding to
// nearest, so an error accumulated over all of K grows linearly with K (about
// 7e-9 * K relative, measured on this part).  The kernel therefore lets the
// tensor core accumulate only kTfChunkKB K blocks (256 values of K) into a
// tensor-memory buffer; the epilogue warps add each finished chunk into an
// fp32 register accumulator with ordinary round-to-nearest additions, and
// store the tile after its last chunk.  The remaining error is about
// 7e-9 * 256 ~ 2e-6 relative, independent of K.
//
// Warp roles (384 threads, 3 warpgroups): warp 0 = copy producer, warp 1 =
// tensor-memory owner and MMA issuer (one thread; with the pair MMA only in
// the pair's first CTA), warps 2-3 idle; warps 4-11 = epilogue.  Epilogue
// warp e reads tensor-memory lanes 32*(e%4).. (a warp may only touch the lane
// quarter of its warp index modulo 4) and columns 128*(e/4)..+127, so each
// thread owns 128 accumulators of one output row.
// Two chunk buffers of 256 columns (all 512 tensor-memory columns) let the
// epilogue drain one chunk while the MMAs fill the next.

constexpr int kTfThreads = 384;
constexpr int kTfLaunchRegs = 168, kTfIssueRegs = 72, kTfEpiRegs = 216;
static_assert(4 * 32 * kTfIssueRegs + 8 * 32 * kTfEpiRegs == kTfThreads * kTfLaunchRegs,
              "setmaxnreg split must balance the launch allocation");
constexpr int kTfChunkKB = 16;                                     // K blocks per chunk (256 of K)
constexpr uint32_t kTfRowBytes = 2 * kTf32BK * 4;                  // hi + lo of one K block: 128 bytes
constexpr uint32_t kTfAStage = kTf32BM * kTfRowBytes;              // 16 KiB
constexpr uint32_t kTfBStage = kTf32BN * kTfRowBytes;              // 32 KiB
constexpr uint32_t kTfStageBytes = kTfAStage + kTfBStage;          // 48 KiB
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kSwRowGroupBytes = 8 * kTfRowBytes;  // 8 rows of the 128-byte swizzle atom
constexpr long long kTileFloats = kTfAStage / 4;        // one 128-row tile: 4096 floats
constexpr uint32_t kDescSwizzle128 = 2;
static_assert(kTfRowBytes == 128, "one K block of hi and lo must fill one 128-byte swizzle row");
// one 32 x 32 fp32 staging block per epilogue warp for the coalesced C store
constexpr uint32_t kTfOutStageBytes = 8 * 32 * 32 * 4;
constexpr uint32_t kTfBarBytes = 256;  // mbarriers and the tensor-memory slot

// Stage ring of the two forms of the kernel.  Per-CTA tensor-core issue
// (kPairMma false): a stage holds the A tile and the whole B tile, 48 KiB, 4
// stages.  Pair MMA (cta_group::2, the pair's first CTA issuing M = 256
// products for both): a CTA holds its A tile and its half of B, 32 KiB, so 6
// stages fit.
template <bool kPairMma>
struct TfRing {
    static constexpr int kStages = kPairMma ? 6 : kTf32Stages;
    static constexpr uint32_t kStageBytes = kPairMma ? 2 * kTfAStage : kTfStageBytes;
    static constexpr int kBars = 3 * kStages + 5;
    static constexpr size_t kSmemBytes = 1024 + (size_t)kStages * kStageBytes + kTfBarBytes + kTfOutStageBytes;
    static_assert(kBars * 8 + 16 <= (int)kTfBarBytes, "barriers and the tensor-memory slot fit");
    static_assert(kSmemBytes <= 232448, "fits the 227 KiB of shared memory a block may opt in to");
};
constexpr size_t kTfSmemBytes = TfRing<false>::kSmemBytes;
constexpr size_t kTfSmemBytesPairMma = TfRing<true>::kSmemBytes;

// Raw operands (split in the kernel, pair-MMA form only).  An operand stored
// K-major (A as M x K, B as N x K) is copied by TMA straight from the
// caller's buffer: one box of 16 K values x 128 rows (8 KiB, 64-byte rows,
// 64-byte swizzle: the tensor core's K-major SW64 layout), rows and K past
// the matrix read as zeros (the ghost elements).  The raw fp32 value is the
// hi operand as it stands: kind::tf32 reads only its sign, exponent and top
// 10 mantissa bits, i.e. hi = x truncated to tf32 (verified on this GPU).
// Two warps of each CTA then write lo = tf32(x - trunc(x)) (x - trunc(x) is
// exact in fp32) beside it, in the same layout 8 KiB further on, so the 16
// KiB region of the operand in a stage holds [raw | lo] instead of the
// pre-pass's 16 KiB hi/lo tile.  The split is elementwise, so it needs no
// knowledge of the swizzle.
constexpr uint32_t kRawTileBytes = kTf32BM * kTf32BK * 4;  // 8 KiB
constexpr uint32_t kSwRowGroupBytes64 = 8 * 64;            // 8 rows of the 64-byte swizzle atom
constexpr uint32_t kDescSwizzle64 = 4;
static_assert(2 * kRawTileBytes == kTfAStage, "raw tile + lo fill one operand region of a stage");

// x rounded to bf16 (nearest even), truncated where that would overflow.
__device__ __forceinline__ uint32_t bf16_bits(float x) {
    const __nv_bfloat16 b = __float2bfloat16_rn(x);
    return __bfloat16_as_ushort((__hisinf(b) && !isinf(x)) ? __float2bfloat16_rz(x) : b);
}

__device__ __forceinline__ uint2 to_bf16x4(float a, float b, float c, float d) {
    return make_uint2(bf16_bits(a) | (bf16_bits(b) << 16), bf16_bits(c) | (bf16_bits(d) << 16));
}

// bf16 of four values (round to nearest even; a finite value beyond the
// largest bf16 becomes the largest, as bf16_bits does), two per instruction:
// the low half of each word holds the earlier value.
__device__ __forceinline__ uint2 to_bf16x4_fast(float a, float b, float c, float d) {
    uint32_t lo, hi;
    asm("cvt.rn.satfinite.bf16x2.f32 %0, %1, %2;" : "=r"(lo) : "f"(b), "f"(a));
    asm("cvt.rn.satfinite.bf16x2.f32 %0, %1, %2;" : "=r"(hi) : "f"(d), "f"(c));
    return make_uint2(lo, hi);
}

// lo = tf32(x - trunc_tf32(x)) of four values.
__device__ __forceinline__ float4 split_lo4(float4 x) {
    auto lo = [](float v) {
        return to_tf32(v - __uint_as_float(__float_as_uint(v) & 0xffffe000u));
    };
    return make_float4(lo(x.x), lo(x.y), lo(x.z), lo(x.w));
}

// The 64 threads t = 0..63 of the split warps write the lo half of one raw
// operand region (512 16-byte groups, 8 per thread; consecutive threads take
// consecutive groups, so every warp access is conflict-free).
__device__ __forceinline__ void split_raw_tile(uint8_t* region, int t) {
    const float4* src = reinterpret_cast<const float4*>(region);
    float4* dst = reinterpret_cast<float4*>(region + kRawTileBytes);
#pragma unroll
    for (int h = 0; h < 2; ++h) {
        float4 v[4];
#pragma unroll
        for (int u = 0; u < 4; ++u) v[u] = src[t + 64 * (4 * h + u)];
#pragma unroll
        for (int u = 0; u < 4; ++u) dst[t + 64 * (4 * h + u)] = split_lo4(v[u]);
    }
}

// The tf32 + bf16 variant with a raw A: the split warps write bf16(hi) and
// bf16(lo) of the raw tile (hi = x truncated to tf32, which is how the tensor
// core reads the raw value in the hi x hi product; lo = x - hi, exact) into
// the region's second 8 KiB: 128 rows of 64 bytes in the 64-byte swizzle,
// 16-byte group j of row r at position j ^ ((r / 2) % 4), groups 0 / 1 holding
// bf16(hi) of K 0-7 / 8-15 and groups 2 / 3 bf16(lo) of the same, so that one
// K = 16 bf16 product reads hi at +0 and lo at +32 bytes of each row.  Raw
// group i (16 bytes) holds row i / 4, K values 4c..4c+3 with c = (i % 4) ^
// ((row / 2) % 4).
//
// Thread t (warp w = t / 32, lane l) takes, in each of its 8 rounds u, the
// 8-row group g = w + 2u: lanes 0-15 rows {0, 1, 4, 5} of the group, lanes
// 16-31 rows {2, 3, 6, 7}, four lanes per row (16-byte position l % 4).  The
// 8-byte stores are served per half-warp; with four consecutive rows in a
// half-warp, rows r and r + 2 (same row parity, swizzle keys 2k and 2k + 1)
// hit the same banks, while rows {0, 1, 4, 5} and {2, 3, 6, 7} fill all 16
// eight-byte slots of a 128-byte bank row (measured: 13.7 M store bank
// conflicts per 4096^3 launch with four consecutive rows per half-warp).
// Every quarter-warp's 16-byte loads still cover 8 different bank groups.
__device__ __forceinline__ void split_raw_tile_bf16(uint8_t* region, int t) {
    const float4* src = reinterpret_cast<const float4*>(region);
    uint8_t* dst = region + kRawTileBytes;
    const int lane = t & 31, w = t >> 5, q = lane & 15;
    const int rig = ((lane >> 4) << 1) + ((q >> 3) << 2) + ((q >> 2) & 1);  // {0,1,4,5} / {2,3,6,7}
    auto trunc = [](float x) { return __uint_as_float(__float_as_uint(x) & 0xffffe000u); };
#pragma unroll
    for (int h = 0; h < 2; ++h) {
        float4 v[4];
        int rr[4];
#pragma unroll
        for (int u = 0; u < 4; ++u) {
            rr[u] = 8 * (w + 2 * (4 * h + u)) + rig;
            v[u] = src[4 * rr[u] + (q & 3)];
        }
#pragma unroll
        for (int u = 0; u < 4; ++u) {
            const int r = rr[u], key = (r >> 1) & 3, c = (q & 3) ^ key;
            const float4 hi = make_float4(trunc(v[u].x), trunc(v[u].y), trunc(v[u].z), trunc(v[u].w));
            const int at = 64 * r + 8 * (c & 1);
            *reinterpret_cast<uint2*>(dst + at + 16 * ((c >> 1) ^ key)) = to_bf16x4_fast(hi.x, hi.y, hi.z, hi.w);
            *reinterpret_cast<uint2*>(dst + at + 16 * ((2 + (c >> 1)) ^ key)) =
                to_bf16x4_fast(v[u].x - hi.x, v[u].y - hi.y, v[u].z - hi.z, v[u].w - hi.w);
        }
    }
}

// kMixed: the operand tiles hold tf32 hi and bf16 hi / lo (the pre-pass's
// kSplitBf16 layout; with a raw A, the kSplitBf16H layout and the split
// above) and each 16-wide K block takes two tf32 hi x hi products and two
// bf16 cross products (hi x lo, lo x hi) instead of six tf32 ones.
// kRawA (pair MMA, 3xTF32): A is staged raw and split in the kernel (see
// kRawTileBytes); tmA then maps the caller's matrix, and B's split tiles come
// in the pre-pass's kSplitTf32H layout, so both operands are read with the
// 64-byte-swizzle descriptors.  (B is never split here: with both operands
// raw the two split warps held the kernel at 320-325 against 374 TFLOP/s at
// 8192^3, more than the pre-pass of B costs.)
template <int kPair, bool kPairMma, bool kMixed = false, bool kRawA = false>
__global__ void __launch_bounds__(kTfThreads, 1)
    tf32x3_gemm_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                       GemmArgs args) {
    static_assert(!kPairMma || kPair == 2, "the pair MMA needs a CTA pair");
    constexpr bool kRaw = kRawA;
    static_assert(!kRaw || kPairMma, "raw A: pair-MMA form only");
    constexpr int BM = kTf32BM, BN = kTf32BN, BK = kTf32BK;
    constexpr int ST = TfRing<kPairMma>::kStages;
    constexpr uint32_t kStageBytes = TfRing<kPairMma>::kStageBytes;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = align_smem_1024(smem_raw);
    uint64_t* full = reinterpret_cast<uint64_t*>(smem + ST * kStageBytes);
    uint64_t* empty = full + ST;
    uint64_t* tfull = empty + ST;  // [2] chunk accumulated
    uint64_t* tempty = tfull + 2;  // [2] chunk drained by the epilogue
    uint64_t* drain = tempty + 2;  // every MMA of this CTA completed
    uint64_t* rfull = drain + 1;   // [ST] this CTA's raw A tile landed
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(rfull + ST);
    float* out_stage = reinterpret_cast<float*>(smem + ST * kStageBytes + kTfBarBytes);  // [8 warps][32 x 32]

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const WaitCtl wc{&g_error_word, args.timeout_ns};
    // cluster of kPair CTAs: CTA `rank` computes tile row 2*row + rank (with
    // the pair MMA it also loads rank's half of the pair's B tile)
    const int rank = kPair > 1 ? (int)cluster_ctarank() : 0;
    const long long first_unit = blockIdx.x / kPair, unit_stride = gridDim.x / kPair;
    constexpr uint16_t kPairMask = (uint16_t)((1u << kPair) - 1u);
    // pair MMA: the first CTA's barriers gather both CTAs' copies (full) and
    // both CTAs' chunk drains (tempty)
    const bool issuer = !kPairMma || rank == 0;

    if (threadIdx.x == 0) {
        for (int s = 0; s < ST; ++s) {
            // the first CTA's copy thread, plus, with raw operands, the two
            // split warps of each CTA of the pair
            mbar_init(&full[s], kRaw ? 1 + 2 * kPair : 1);
            // one MMA commit: this CTA's own, or the pair MMA's (which arrives in both CTAs)
            mbar_init(&empty[s], 1);
            mbar_init(&rfull[s], 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(&tfull[b], 1);
            mbar_init(&tempty[b], kPairMma ? 16 : 8);
        }
        mbar_init(drain, 1);
        fence_barrier_init();
    }
    if (warp == 1) {
        if (kPairMma) {
            tmem_alloc_pair(tmem_slot, kTmemCols);
            tmem_relinquish_pair();
        } else {
            tmem_alloc(tmem_slot, kTmemCols);
            tmem_relinquish();
        }
    }
    tc_fence_before_sync();
    __syncthreads();
    if (kPairMma) cluster_sync_all();  // the peer's barriers exist before any remote arrive
    tc_fence_after_sync();
    const uint32_t tmem_base = *tmem_slot;
    // the set-up above overlaps the end of the pre-pass; its output is read below
    grid_dep_wait();
    grid_dep_launch();

    if (warp < 4) {
        regs_dec<kTfIssueRegs>();
        if (warp == 0 && lane == 0) {  // ------------------------- producer
            int stage = 0;
            uint32_t phase = 0, issued = 0, last_par = 0;
            bool ok = true;
            Unit t;
            for (long long j = 0; ok && work_item<true, false>(args, first_unit, unit_stride, j, rank, BM, BN, &t); ++j) {
                for (int kb = t.kb0; kb < t.kb1; ++kb) {
                    // pair MMA: "empty" completes when the pair's products
                    // that read this stage in both CTAs are done
                    if (!mbar_wait(&empty[stage], phase ^ 1u, wc, kSiteTfProducer)) {
                        ok = false;
                        break;
                    }
                    uint8_t* st = smem + stage * kStageBytes;
                    // odd work items walk K backwards: this lane's next item
                    // (in the next round) usually has the same A rows, and
                    // starting where this one ended finds them still in L2
                    const int kq = (j & 1) ? t.kb0 + t.kb1 - 1 - kb : kb;
                    if (kPairMma) {
                        // this CTA's A tile and B half into its own ring.  Both
                        // CTAs' split-tile copies complete on the first CTA's
                        // "full"; a raw A tile completes on this CTA's "rfull",
                        // where the split warps pick it up
                        constexpr uint32_t kPairTx = 2 * ((kRawA ? 0 : kTfAStage) + kTfAStage);
                        if (kRawA) mbar_arrive_expect_tx(&rfull[stage], kRawTileBytes);
                        if (rank == 0) mbar_arrive_expect_tx(&full[stage], kPairTx);
                        const uint32_t bar0 = cluster_addr(&full[stage], 0);
                        if (kRawA)
                            tma_load_2d(st, &tmA, &rfull[stage], kq * BK, t.m0);
                        else
                            tma_load_2d_pair(st, &tmA, bar0, 0, ((t.m0 >> 7) * args.kbs + kq) * 128);
                        tma_load_2d_pair(st + kTfAStage, &tmB, bar0, 0, (((t.n0 >> 7) + rank) * args.kbs + kq) * 128);
                        issued |= 1u << stage;
                        last_par = (last_par & ~(1u << stage)) | (phase << stage);
                        if (++stage == ST) {
                            stage = 0;
                            phase ^= 1u;
                        }
                        continue;
                    }
                    // this CTA's A tile and the whole B tile (48 KiB), each
                    // 128-row tile one bulk copy into this CTA's own ring
                    mbar_arrive_expect_tx(&full[stage], kTfStageBytes);
                    const float* a_src = args.a_tiles + ((long long)(t.m0 >> 7) * args.kbs + kq) * kTileFloats;
                    const float* b_src = args.b_tiles + ((long long)(t.n0 >> 7) * args.kbs + kq) * kTileFloats;
                    bulk_load(st, a_src, kTfAStage, &full[stage]);
                    bulk_load(st + kTfAStage, b_src, kTfAStage, &full[stage]);
                    bulk_load(st + 2 * kTfAStage, b_src + (long long)args.kbs * kTileFloats, kTfAStage, &full[stage]);
                    issued |= 1u << stage;
                    last_par = (last_par & ~(1u << stage)) | (phase << stage);
                    if (++stage == ST) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
            }
            // every copy must land before the CTA may exit.  Pair MMA: the
            // first CTA's "full" barriers count both CTAs' bytes; the second
            // CTA waits instead until the products have consumed its last
            // stages ("empty" completes only after the copies landed).
            for (int s = 0; s < ST; ++s) {
                if (!((issued >> s) & 1u)) continue;
                if (kRaw) mbar_drain(&rfull[s], (last_par >> s) & 1u, args.timeout_ns);
                if (issuer)
                    mbar_drain(&full[s], (last_par >> s) & 1u, args.timeout_ns);
                else
                    mbar_drain(&empty[s], (last_par >> s) & 1u, args.timeout_ns);
            }
        } else if (kRaw && (warp == 2 || warp == 3)) {  // ------------- split of raw A tiles
            // per stage: wait for this CTA's raw A tile, write its lo half,
            // publish them to the tensor core (async proxy) and arrive on the
            // first CTA's "full" barrier, where the MMA thread waits
            const int t64 = threadIdx.x - 64;
            int stage = 0;
            uint32_t phase = 0;
            bool ok = true;
            Unit t;
            for (long long j = 0; ok && work_item<true, false>(args, first_unit, unit_stride, j, rank, BM, BN, &t); ++j) {
                for (int kb = t.kb0; kb < t.kb1; ++kb) {
                    const bool got = mbar_wait(&rfull[stage], phase, wc, kSiteTfSplit);
                    if (!__all_sync(0xffffffffu, got)) {
                        ok = false;
                        break;
                    }
                    if (kMixed)
                        split_raw_tile_bf16(smem + stage * kStageBytes, t64);
                    else
                        split_raw_tile(smem + stage * kStageBytes, t64);
                    fence_proxy_async_smem();
                    __syncwarp();
                    if (lane == 0) mbar_arrive_cluster(cluster_addr(&full[stage], 0));
                    if (++stage == ST) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
            }
        } else if (warp == 1 && lane == 0 && issuer) {  // ---------------- MMA issuer
            constexpr uint32_t idesc = idesc_tf32(kPairMma ? 2 * BM : BM, BN);
            constexpr uint32_t idesc_x = idesc_bf16(kPairMma ? 2 * BM : BM, BN);
            static_assert(BK == 16 && kTfRowBytes == 128, "the issue loop below is written for two 8-wide slices");
            const uint64_t desc_stage0 = smem_desc_kmajor(smem_addr(smem), kSwRowGroupBytes, kDescSwizzle128);
            // operand descriptors of stage 0 and the offset (16-byte units) of
            // the lo halves: a kSplitTf32 tile holds hi and lo in one 128-byte
            // swizzled row (lo +64 bytes); with raw operands every operand
            // region holds hi (or the raw tile) in 64-byte swizzled rows and
            // lo 8 KiB on.  The second 8-wide K slice is +32 bytes either way.
            constexpr uint32_t kLo = kRaw ? kRawTileBytes >> 4 : 4;
            const uint64_t desc_a0 =
                kRaw ? smem_desc_kmajor(smem_addr(smem), kSwRowGroupBytes64, kDescSwizzle64) : desc_stage0;
            const uint64_t desc_b0 = desc_a0 + (kTfAStage >> 4);
            int stage = 0;
            uint32_t phase = 0, chunk = 0;
            bool ok = true;
            Unit t;
            for (long long j = 0; ok && work_item<true, false>(args, first_unit, unit_stride, j, rank, BM, BN, &t); ++j) {
                for (int c0 = t.kb0; ok && c0 < t.kb1; c0 += kTfChunkKB, ++chunk) {
                    const int c1 = min(c0 + kTfChunkKB, t.kb1);
                    const uint32_t buf = chunk & 1u, par = (chunk >> 1) & 1u;
                    if (!mbar_wait(&tempty[buf], par ^ 1u, wc, kSiteTfMmaTmem)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after_sync();
                    const uint32_t d_tmem = tmem_base + buf * BN;
                    for (int kb = c0; kb < c1; ++kb) {
                        // raw operands: the split warps of both CTAs arrive
                        // after writing shared memory the products read
                        if (!(kRaw ? mbar_wait_cluster(&full[stage], phase, wc, kSiteTfMmaSmem)
                                   : mbar_wait(&full[stage], phase, wc, kSiteTfMmaSmem))) {
                            ok = false;
                            break;
                        }
                        tc_fence_after_sync();
                        // descriptors of this stage's tiles; their address field
                        // counts 16-byte units, so the lo half of each 128-byte row
                        // is +4 and the second 8-wide K slice +2
                        const uint64_t da = desc_stage0 + (uint64_t)stage * (kStageBytes >> 4);
                        const uint64_t db = da + (kTfAStage >> 4);
                        if (kMixed) {
                            // bf16 hi at +4 (K 0-15 in one 32-byte slice), bf16 lo at +6
                            const uint32_t acc = kb > c0 ? 1u : 0u;
                            if (kRaw) {
                                // every operand in 64-byte-swizzle rows: tf32 hi
                                // (the raw A) at +0 / +32 bytes per slice, the bf16
                                // tile 8 KiB on with hi at +0 and lo at +32 bytes
                                constexpr uint32_t kX = kRawTileBytes >> 4;
                                const uint64_t pa = desc_a0 + (uint64_t)stage * (kStageBytes >> 4);
                                const uint64_t pb = desc_b0 + (uint64_t)stage * (kStageBytes >> 4);
                                mma_f16_ss_pair(d_tmem, pa + kX, pb + kX + 2, idesc_x, acc);
                                mma_f16_ss_pair(d_tmem, pa + kX + 2, pb + kX, idesc_x, 1u);
                                mma_tf32_ss_pair(d_tmem, pa, pb, idesc, 1u);
                                mma_tf32_ss_pair(d_tmem, pa + 2, pb + 2, idesc, 1u);
                                mma_commit_pair(&empty[stage], kPairMask);
                            } else if (kPairMma) {
                                mma_f16_ss_pair(d_tmem, da + 4, db + 6, idesc_x, acc);
                                mma_f16_ss_pair(d_tmem, da + 6, db + 4, idesc_x, 1u);
                                mma_tf32_ss_pair(d_tmem, da, db, idesc, 1u);
                                mma_tf32_ss_pair(d_tmem, da + 2, db + 2, idesc, 1u);
                                mma_commit_pair(&empty[stage], kPairMask);
                            } else {
                                mma_f16_ss(d_tmem, da + 4, db + 6, idesc_x, acc);
                                mma_f16_ss(d_tmem, da + 6, db + 4, idesc_x, 1u);
                                mma_tf32_ss(d_tmem, da, db, idesc, 1u);
                                mma_tf32_ss(d_tmem, da + 2, db + 2, idesc, 1u);
                                mma_commit(&empty[stage]);
                            }
                            if (++stage == ST) {
                                stage = 0;
                                phase ^= 1u;
                            }
                            continue;
                        }
                        if (kPairMma) {  // M = 256 over the pair: each CTA's A rows and B half
                            const uint32_t acc = kb > c0 ? 1u : 0u;
                            const uint64_t pa = desc_a0 + (uint64_t)stage * (kStageBytes >> 4);
                            const uint64_t pb = desc_b0 + (uint64_t)stage * (kStageBytes >> 4);
                            mma_tf32_ss_pair(d_tmem, pa, pb + kLo, idesc, acc);
                            mma_tf32_ss_pair(d_tmem, pa, pb, idesc, 1u);
                            mma_tf32_ss_pair(d_tmem, pa + kLo, pb, idesc, 1u);
                            mma_tf32_ss_pair(d_tmem, pa + 2, pb + kLo + 2, idesc, 1u);
                            mma_tf32_ss_pair(d_tmem, pa + 2, pb + 2, idesc, 1u);
                            mma_tf32_ss_pair(d_tmem, pa + kLo + 2, pb + 2, idesc, 1u);
                            mma_commit_pair(&empty[stage], kPairMask);
                            if (++stage == ST) {
                                stage = 0;
                                phase ^= 1u;
                            }
                            continue;
                        }
                        // A_hi is read from shared memory once per slice and kept in
                        // the tensor core's A collector for its second product.  The
                        // chunk's first K block starts the accumulator.  No branch
                        // separates the MMAs: a branch in the issue sequence cost
                        // the single issuing thread about 10 % of its rate
                        // (measured), a flag computed per block does not.
                        const uint32_t acc = kb > c0 ? 1u : 0u;
                        mma_tf32_ss_fill_a(d_tmem, da, db + 4, idesc, acc);
                        mma_tf32_ss_lastuse_a(d_tmem, da, db, idesc, 1u);
                        mma_tf32_ss(d_tmem, da + 4, db, idesc, 1u);
                        mma_tf32_ss_fill_a(d_tmem, da + 2, db + 6, idesc, 1u);
                        mma_tf32_ss_lastuse_a(d_tmem, da + 2, db + 2, idesc, 1u);
                        mma_tf32_ss(d_tmem, da + 6, db + 2, idesc, 1u);
                        // frees the stage once these MMAs are done
                        mma_commit(&empty[stage]);
                        if (++stage == ST) {
                            stage = 0;
                            phase ^= 1u;
                        }
                    }
                    if (ok) {
                        if (kPairMma)
                            mma_commit_pair(&tfull[buf], kPairMask);
                        else
                            mma_commit(&tfull[buf]);
                    }
                }
            }
            // no tensor-memory access may be in flight when the CTA frees it
            if (kPairMma)
                mma_commit_pair(drain, kPairMask);
            else
                mma_commit(drain);
            mbar_drain(drain, 0, args.timeout_ns);
        }
    } else {  // ---------------------------------------------------- epilogue
        regs_inc<kTfEpiRegs>();
        const int e = warp - 4;
        const int q = warp & 3;        // tensor-memory lanes 32q..32q+31 = tile rows
        const int h = e >> 2;          // tile columns 128h..128h+127
        uint32_t chunk = 0;
        bool ok = true;
        Unit t;
        for (long long j = 0; ok && work_item<true>(args, first_unit, unit_stride, j, rank, BM, BN, &t); ++j) {
            float acc[128];
#pragma unroll
            for (int i = 0; i < 128; ++i) acc[i] = 0.0f;
            for (int c0 = t.kb0; c0 < t.kb1; c0 += kTfChunkKB, ++chunk) {
                const uint32_t buf = chunk & 1u, par = (chunk >> 1) & 1u;
                const bool got = mbar_wait(&tfull[buf], par, wc, kSiteTfEpilogue);
                if (!__all_sync(0xffffffffu, got)) {
                    ok = false;
                    break;
                }
                tc_fence_after_sync();
                const uint32_t taddr = tmem_base + ((uint32_t)(q * 32) << 16) + buf * BN + h * 128;
#pragma unroll
                for (int c = 0; c < 4; ++c) {
                    uint32_t r[32];
                    tmem_ld_32x32b_x32(taddr + c * 32, r);
                    tmem_ld_wait(r);
#pragma unroll
                    for (int i = 0; i < 32; ++i)
                        acc[c * 32 + i] += __uint_as_float(r[i]);
                }
                tc_fence_before_sync();
                __syncwarp();
                if (lane == 0) {  // chunk buffer may be refilled
                    if (kPairMma)
                        mbar_arrive_cluster(cluster_addr(&tempty[buf], 0));
                    else
                        mbar_arrive(&tempty[buf]);
                }
            }
            if (!ok) break;
            // Guarded store of the warp's 32 rows x 128 columns, coalesced: each
            // 32 x 32 block goes through the warp's shared-memory buffer (lane
            // = row on the way in, lane = column on the way out) and leaves one
            // row per instruction, 128 contiguous bytes.  Storing each thread's
            // row directly sent 32 separate 16-byte pieces per instruction, and
            // the burst of requests at every unit's end held up the next unit's
            // operand copies (measured: 2-6 % of the kernel, more for short K).
            // The 4-value group g of row r sits at r*32 + 4*(g ^ (r & 7)): the
            // 16-byte writes of 8 lanes (one row each) and the 4-byte reads of
            // a warp (one column each) both touch 32 different banks.
            float* stg = out_stage + e * 1024;
            const bool scaled = args.scaled != 0 && t.direct;
            const int row0 = t.m0 + q * 32;
            float4* stg_row = reinterpret_cast<float4*>(stg + lane * 32);
            const int rsw = lane & 7;
            const int rows = min(32, args.M - row0);
#pragma unroll
            for (int cb = 0; cb < 4; ++cb) {
#pragma unroll
                for (int g = 0; g < 8; ++g)
                    stg_row[g ^ rsw] = make_float4(acc[cb * 32 + 4 * g], acc[cb * 32 + 4 * g + 1],
                                                   acc[cb * 32 + 4 * g + 2], acc[cb * 32 + 4 * g + 3]);
                __syncwarp();
                const int col = t.n0 + h * 128 + cb * 32 + lane;
                // 16-byte stores (lanes 8k..8k+7 take the 8 groups of row k +
                // 4i, four 128-byte rows per instruction) where rows start on
                // 16 bytes and no split-point tail runs: measured against the
                // one-row-per-instruction form below, 2048^3 83.5 vs 85.3 us,
                // 777 x 1029 x 513 26.5 vs 27.5 us, 4096^3 kernel 373.5 vs 369.5
                // TFLOP/s, 8192^3 equal; with a split point (2048 x 2048 x
                // 16384) the pieces' 16-byte stores slowed the kernel ~1 %.
                // 3xTF32 pair forms only: the mixed instantiation spilled
                const bool vec4 = t.direct ? args.vec_out != 0 : true;
                if (kPairMma && !kMixed && args.tail_kx == 0 && vec4 && !(scaled && args.beta != 0.0f)) {
                    const int g = lane & 7;
                    const int colg = t.n0 + h * 128 + cb * 32 + 4 * g;
#pragma unroll
                    for (int i = 0; i < 8; ++i) {
                        const int r = (lane >> 3) + 4 * i;
                        if (r < rows) {
                            // group g of row r sits at r*32 + 4*(g ^ (r & 7))
                            float4 v = *reinterpret_cast<const float4*>(stg + r * 32 + 4 * (g ^ (r & 7)));
                            if (scaled)
                                v = make_float4(args.alpha * v.x, args.alpha * v.y, args.alpha * v.z, args.alpha * v.w);
                            store_row4(t.out + (long long)(row0 + r) * t.ldo, colg, args.N, v, true);
                        }
                    }
                } else if (col < args.N) {
                    // (r, lane) sits at r*32 + (lane ^ 4*(r & 7))
                    float* dst = t.out + (long long)row0 * t.ldo + col;
                    if (scaled && args.beta != 0.0f) {
                        // C's old values first, all 32 loads in flight at once:
                        // one load per store, each waited for in turn, held
                        // the epilogue up long enough to stall the next unit's
                        // MMAs (8192^3 kernel 317 against 384 TFLOP/s)
                        float old[32];
                        const float* src = dst;
#pragma unroll
                        for (int r = 0; r < 32; ++r, src += t.ldo) old[r] = r < rows ? *src : 0.0f;
#pragma unroll
                        for (int r = 0; r < 32; ++r, dst += t.ldo)
                            if (r < rows)
                                *dst = fmaf(args.alpha, stg[r * 32 + (lane ^ ((r & 7) << 2))], args.beta * old[r]);
                    } else {
#pragma unroll 1
                        for (int r = 0; r < rows; ++r, dst += t.ldo) {
                            const float v = stg[r * 32 + (lane ^ ((r & 7) << 2))];
                            *dst = scaled ? args.alpha * v : v;
                        }
                    }
                }
                __syncwarp();
            }
        }
    }

    __syncthreads();
    // pair MMA: the first CTA's products write both CTAs' tensor memory, and
    // its MMA thread has seen them all complete before it gets here
    if (kPairMma) cluster_sync_all();
    if (warp == 1) {
        __syncwarp();
        tc_fence_after_sync();
        if (kPairMma)
            tmem_dealloc_pair(tmem_base, kTmemCols);
        else
            tmem_dealloc(tmem_base, kTmemCols);
    }
    // pair MMA: neither CTA may exit while the other can still arrive on its
    // barriers or have products read its shared memory
    if (kPairMma) cluster_sync_all();
}

// ------------------------------------------------------------ pre-pass
//
// Lays each operand out K-major for the GEMM kernels, zero-padding columns
// past the valid extent (ghost elements):
//   SPLIT (3xTF32): op(A) and op(B)^T as 16 KiB tiles of 128 rows x one
//     16-wide K block, [row tile][K block], with rows padded to whole tiles
//     (zeros).  Tile row r holds 16 hi then 16 lo values, each 4-value group
//     (16 bytes) j of the 8 stored at position j ^ (r % 8): the 128-byte
//     swizzle.  hi = tf32(x), lo = tf32(x - hi) (x - hi is exact in fp32).
//   PACK (FFMA, operand not TMA-legal or transposed): op(A) -> [M][k4],
//     op(B) -> [K][n4].
// Each operand is either copied row by row (its stored rows already run along
// the destination rows) or transposed.  Memory-bound: the row-wise pass moves
// 4 values per item with 16-byte stores (and 16-byte loads when the source
// rows are 16-byte aligned), eight items in flight per thread; the transpose
// runs on 64 x 64 tiles through a [64][65] shared tile, 16 values per thread
// in flight, the next tile's loads overlapping the current tile's stores;
// the padded row makes the column read conflict-free ("Bank Conflict",
// padding: gcd(65, 32) = 1).  Loads and stores are row-coalesced.

struct OperandPass {
    const float* src;
    long long ld;    // source row stride (elements)
    int rows;        // destination rows written (SPLIT: padded to whole tiles)
    int rows_valid;  // destination rows that exist in the source (the rest are zeros)
    int cols;        // valid destination columns (source extent)
    int pitch;       // padded destination columns (multiple of 16 for SPLIT, of 4 for PACK)
    int trans;       // 1: dst[r][c] = src[c*ld + r]; 0: dst[r][c] = src[r*ld + c]
    int vec;         // row-wise only: source rows start on 16-byte boundaries
    float* d0;       // destination (nullptr = operand not needed)
    long long items; // row-wise: rows * pitch/4; transpose: 64x64 tiles
    int tiles_c;     // transpose: 64-wide tiles along the destination columns
};

struct PrepassArgs {
    OperandPass op[2];  // A, then B
};

__device__ __forceinline__ float4 load_row4(const float* src, long long ld, int row, int col,
                                            int cols, bool vec) {
    const float* p = src + (long long)row * ld + col;
    if (vec && col + 3 < cols) return *reinterpret_cast<const float4*>(p);
    float4 v;
    v.x = col < cols ? p[0] : 0.0f;
    v.y = col + 1 < cols ? p[1] : 0.0f;
    v.z = col + 2 < cols ? p[2] : 0.0f;
    v.w = col + 3 < cols ? p[3] : 0.0f;
    return v;
}

// Pre-pass modes: kPack copies (FFMA: op(A) -> [M][k4], op(B) -> [K][n4]);
// kSplitTf32 writes hi = tf32(x) and lo = tf32(x - hi) (3xTF32); kSplitBf16
// writes hi = tf32(x) and the bf16 roundings of hi and of x - hi (the
// bf16-cross-product path).  Both fill 128-byte tile rows of eight 16-byte
// groups, group g of row r stored at position g ^ (r % 8) (128-byte swizzle):
// kSplitTf32: groups 0-3 hi of K values 4g..4g+3, groups 4-7 their lo;
// kSplitBf16: groups 0-3 hi (tf32), group 4 / 5 bf16(hi) of K values 0-7 /
// 8-15, group 6 / 7 bf16(lo) of the same.
// kSplitTf32H writes the same hi and lo as kSplitTf32 in the layout of a raw
// operand region of the fused kernel: the tile's first 8 KiB hold hi, 64-byte
// rows of 16 K values with the 64-byte swizzle (group g of row r at position
// g ^ ((r / 2) % 4)), the second 8 KiB lo in the same places.  The pair MMA
// reads both operands of a product in one swizzle mode (measured on GB300: an
// A tile in the 64-byte and a B tile in the 128-byte swizzle gave wrong
// products in the cta_group::2 form, though not with one CTA), so a product
// whose other operand is split in the kernel takes this layout.
// kSplitBf16H: the kSplitBf16 values for a product whose A the kernel splits:
// tf32 hi in the first 8 KiB as in kSplitTf32H, and the second 8 KiB as 128
// rows of 64 bytes, 16-byte group j of row r at position j ^ ((r / 2) % 4),
// groups 0 / 1 bf16(hi) of K 0-7 / 8-15, groups 2 / 3 bf16(lo) (the layout
// the split warps write for A, see split_raw_tile_bf16).
constexpr int kPack = 0, kSplitTf32 = 1, kSplitBf16 = 2, kSplitTf32H = 3, kSplitBf16H = 4;

// Offset of destination element (r, c): hi in its swizzled tile (split
// modes) or the plain padded row (kPack).
template <int MODE>
__device__ __forceinline__ long long dst_offset(int pitch, int r, int c) {
    const long long tile = ((long long)(r >> 7) * (pitch >> 4) + (c >> 4)) * 4096;
    if (MODE == kSplitTf32H || MODE == kSplitBf16H)
        return tile + (r & 127) * 16 + ((((c & 15) >> 2) ^ ((r >> 1) & 3)) << 2) + (c & 3);
    if (MODE != kPack)
        return tile + (r & 127) * 32 + ((((c & 15) >> 2) ^ (r & 7)) << 2) + (c & 3);
    return (long long)r * pitch + c;
}

// kSplitBf16: float offset of the 4 bf16 values (8 bytes) that belong to the
// hi group at offset o, in logical group `first` (4: bf16 hi, 6: bf16 lo).
// o encodes the row (bits 5-11, swizzle key bits 5-7) and the stored group
// position (bits 2-4), so the logical group j follows from o alone.
__device__ __forceinline__ long long bf16_offset(long long o, int first) {
    const int key = (int)(o >> 5) & 7, j = ((int)(o >> 2) & 7) ^ key;
    return (o & ~31ll) + (((first + (j >> 1)) ^ key) << 2) + ((j & 1) << 1);
}

// hi of the split: x rounded to tf32 (nearest, ties away), or truncated where
// that rounding would carry one of the largest finite values to infinity.
__device__ __forceinline__ float split_hi(float x) {
    const float h = to_tf32(x);
    return (isinf(h) && !isinf(x)) ? __uint_as_float(__float_as_uint(x) & 0xffffe000u) : h;
}

// Store destination columns c..c+3 of row r (c a multiple of 4: one 16-byte
// group) at offset o.
template <int MODE>
__device__ __forceinline__ void store_split4(float* d0, long long o, float4 x) {
    if (MODE == kPack) {
        *reinterpret_cast<float4*>(d0 + o) = x;
        return;
    }
    const float4 hi = make_float4(split_hi(x.x), split_hi(x.y), split_hi(x.z), split_hi(x.w));
    *reinterpret_cast<float4*>(d0 + o) = hi;
    if (MODE == kSplitTf32H) {
        *reinterpret_cast<float4*>(d0 + o + 2048) =
            make_float4(to_tf32(x.x - hi.x), to_tf32(x.y - hi.y), to_tf32(x.z - hi.z), to_tf32(x.w - hi.w));
    } else if (MODE == kSplitBf16H) {
        // o = tile + 16 row + 4 (c ^ key) with key = (row / 2) % 4, c = (K % 16) / 4
        const long long tile = o & ~4095ll;
        const int row = (int)(o >> 4) & 127, key = (row >> 1) & 3, c = ((int)(o >> 2) & 3) ^ key;
        float* b = d0 + tile + 2048 + 16 * row + 2 * (c & 1);
        *reinterpret_cast<uint2*>(b + 4 * ((c >> 1) ^ key)) = to_bf16x4(hi.x, hi.y, hi.z, hi.w);
        *reinterpret_cast<uint2*>(b + 4 * ((2 + (c >> 1)) ^ key)) =
            to_bf16x4(x.x - hi.x, x.y - hi.y, x.z - hi.z, x.w - hi.w);
    } else if (MODE == kSplitTf32) {
        *reinterpret_cast<float4*>(d0 + (o ^ 16)) =
            make_float4(to_tf32(x.x - hi.x), to_tf32(x.y - hi.y), to_tf32(x.z - hi.z), to_tf32(x.w - hi.w));
    } else {
        *reinterpret_cast<uint2*>(d0 + bf16_offset(o, 4)) = to_bf16x4(hi.x, hi.y, hi.z, hi.w);
        *reinterpret_cast<uint2*>(d0 + bf16_offset(o, 6)) =
            to_bf16x4(x.x - hi.x, x.y - hi.y, x.z - hi.z, x.w - hi.w);
    }
}

template <int MODE>
__device__ __forceinline__ void rowwise_pass(const OperandPass& p) {
    constexpr int kInFlight = 8;  // 16-byte loads issued before the first store
    const long long stride = (long long)gridDim.x * blockDim.x;
    const int groups = p.pitch / 4;
    for (long long i = blockIdx.x * (long long)blockDim.x + threadIdx.x; i < p.items; i += kInFlight * stride) {
        float4 v[kInFlight];
        long long o[kInFlight];
#pragma unroll
        for (int u = 0; u < kInFlight; ++u) {
            const long long it = i + u * stride;
            o[u] = -1;
            if (it < p.items) {
                const int r = (int)(it / groups), c = (int)(it % groups) * 4;
                v[u] = r < p.rows_valid ? load_row4(p.src, p.ld, r, c, p.cols, p.vec != 0)
                                        : make_float4(0.f, 0.f, 0.f, 0.f);
                o[u] = dst_offset<MODE>(p.pitch, r, c);
            }
        }
#pragma unroll
        for (int u = 0; u < kInFlight; ++u)
            if (o[u] >= 0) store_split4<MODE>(p.d0, o[u], v[u]);
    }
}

// Source tile (r0, c0) of a transpose: this thread's 16 values, rows c0 + ty
// + 4j of the source (destination columns), column r0 + tx (coalesced).
__device__ __forceinline__ void transpose_load(const OperandPass& p, long long t, int tx, int ty, float* v) {
    const int r0 = (int)(t / p.tiles_c) * 64, c0 = (int)(t % p.tiles_c) * 64;
#pragma unroll
    for (int j = 0; j < 16; ++j) {
        const int c = c0 + ty + 4 * j, r = r0 + tx;
        v[j] = (c < p.cols && r < p.rows_valid) ? p.src[(long long)c * p.ld + r] : 0.0f;
    }
}

// The tiles are software-pipelined: the loads of a block's next tile are
// issued before the stores of the current one, so reads stay in flight while
// the block writes.
template <int MODE>
__device__ __forceinline__ void transpose_pass(const OperandPass& p, float (*tile)[65]) {
    const int tx = threadIdx.x & 63, ty = threadIdx.x >> 6;  // 64 x 4 threads
    long long t = blockIdx.x;
    if (t >= p.items) return;
    float v[16];
    transpose_load(p, t, tx, ty, v);
    for (; t < p.items; t += gridDim.x) {
        const int r0 = (int)(t / p.tiles_c) * 64, c0 = (int)(t % p.tiles_c) * 64;
#pragma unroll
        for (int j = 0; j < 16; ++j) tile[ty + 4 * j][tx] = v[j];
        __syncthreads();
        if (t + gridDim.x < p.items) transpose_load(p, t + gridDim.x, tx, ty, v);
        // one 16-byte group (destination columns c..c+3) of row r per store;
        // 16 threads cover a row's 64 columns
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            const int g = threadIdx.x + 256 * q, rl = g >> 4, cl = (g & 15) * 4;
            const int r = r0 + rl, c = c0 + cl;
            if (r < p.rows && c < p.pitch)  // pitch is a multiple of 4: the whole group is in range
                store_split4<MODE>(p.d0, dst_offset<MODE>(p.pitch, r, c),
                                   make_float4(tile[cl][rl], tile[cl + 1][rl], tile[cl + 2][rl], tile[cl + 3][rl]));
        }
        __syncthreads();
    }
}

template <int MODE>
__global__ void __launch_bounds__(256) prepass_kernel(PrepassArgs a) {
    __shared__ float tile[64][65];
    grid_dep_launch();  // the GEMM may start its set-up as this pass drains
    // A, then B (constant indices: the arguments stay in parameter space)
    if (a.op[0].d0 != nullptr) {
        if (a.op[0].trans)
            transpose_pass<MODE>(a.op[0], tile);
        else
            rowwise_pass<MODE>(a.op[0]);
    }
    if (a.op[1].d0 != nullptr) {
        if (a.op[1].trans)
            transpose_pass<MODE>(a.op[1], tile);
        else
            rowwise_pass<MODE>(a.op[1]);
    }
}

// ------------------------------------------------------ split-K reduce
// C = sum_{s=0}^{S-1} partial_s, always in slice order s = 0, 1, ... so the
// result does not depend on scheduling (float atomics would: "Reduction",
// the atomicAdd variant).  Memory-bound; float4 loads of the 16-byte-pitched
// partials.
__global__ void __launch_bounds__(256)
    splitk_reduce_kernel(const float* __restrict__ part, long long ldp, long long slice, int S,
                         float* C, long long ldc, int M, int N, int vec_c, int scaled, float alpha,
                         float beta) {
    grid_dep_wait();  // every partial is written
    const int n4g = (N + 3) / 4;
    const long long total = (long long)M * n4g;
    for (long long i = blockIdx.x * (long long)blockDim.x + threadIdx.x; i < total;
         i += (long long)gridDim.x * blockDim.x) {
        const int m = (int)(i / n4g), c = (int)(i % n4g) * 4;
        const float* p = part + (long long)m * ldp + c;
        float4 s = *reinterpret_cast<const float4*>(p);
        for (int t = 1; t < S; ++t) {
            const float4 v = *reinterpret_cast<const float4*>(p + t * slice);
            s.x += v.x;
            s.y += v.y;
            s.z += v.z;
            s.w += v.w;
        }
        if (scaled)
            store_row4_scaled(C + (long long)m * ldc, c, N, s, vec_c != 0, alpha, beta);
        else
            store_row4(C + (long long)m * ldc, c, N, s, vec_c != 0);
    }
}

// Balanced last round: every tail unit that more than one lane ran is the
// sum of its pieces' partials, added in a fixed order (deterministic).
// Stream-K runs: lane order; a unit run whole by one lane was stored by the
// GEMM kernel.  Split point: the unit's first part, then the pieces of its
// remainder in lane order.  A block takes a band of rows of one unit at a
// time (4 rows of 16-byte groups per thread, blockDim / (BN / 4) rows per
// pass), so the unit's lanes and slots are worked out once per band, not for
// every element: with the 64-bit divisions they need, per element they made
// the kernel instruction-bound (20 us for a 2048 x 2048 split-point tail).
__global__ void __launch_bounds__(256)
    tail_reduce_kernel(GemmArgs a, float* C, long long ldc, int BM, int BN, int vec_c) {
    grid_dep_wait();  // every partial is written
    constexpr int kRowsPerThread = 4;
    const int rows = a.pair * BM, q4 = BN / 4;
    const int rstep = blockDim.x / q4, band = kRowsPerThread * rstep;
    const int bands = (rows + band - 1) / band;
    const long long block = (long long)rows * BN;
    const long long items = a.tail_units * bands;
    const int tr = threadIdx.x / q4, c = (threadIdx.x % q4) * 4;
    for (long long b = blockIdx.x; b < items; b += gridDim.x) {
        const long long q = b / bands;
        const int r0 = (int)(b - q * bands) * band + tr;
        long long v0, v1, T, lanes, first;
        if (a.tail_kx > 0) {
            const long long rl = a.nkb - a.tail_kx;
            T = a.tail_units * rl;
            lanes = a.tail_lanes - a.tail_units;
            v0 = tail_lane_of(q * rl, T, lanes);
            v1 = tail_lane_of((q + 1) * rl - 1, T, lanes);
            first = q * a.tail_slots;  // the unit's first part
        } else {
            T = a.tail_units * a.nkb;
            lanes = a.tail_lanes;
            v0 = tail_lane_of(q * a.nkb, T, lanes);
            v1 = tail_lane_of((q + 1) * a.nkb - 1, T, lanes);
            if (v0 == v1) continue;
            first = 2 * v0 + (tail_run_begin(v0, T, lanes) / a.nkb == q ? 0 : 1);
        }
        int tm, tn;
        unit_tile(a.tiles_m, a.tiles_n, a.full_units + q, &tm, &tn);
        const int n = tn * BN + c;
        bool ok[kRowsPerThread];
        float4 s[kRowsPerThread];
        const float* tile = a.tail + (long long)r0 * BN + c;
#pragma unroll
        for (int u = 0; u < kRowsPerThread; ++u) {
            const int r = r0 + u * rstep;
            ok[u] = r < rows && tm * rows + r < a.M && n < a.N;
            s[u] = ok[u] ? *reinterpret_cast<const float4*>(tile + first * block + (long long)u * rstep * BN)
                         : make_float4(0.f, 0.f, 0.f, 0.f);
        }
        for (long long v = a.tail_kx > 0 ? v0 : v0 + 1; v <= v1; ++v) {
            // stream-K: slot 2v holds lane v's first piece, 2v + 1 its last;
            // split point: slot first + 1 + (v - v0)
            long long slot;
            if (a.tail_kx > 0)
                slot = first + 1 + (v - v0);
            else
                slot = 2 * v + (tail_run_begin(v, T, lanes) / a.nkb == q ? 0 : 1);
#pragma unroll
            for (int u = 0; u < kRowsPerThread; ++u) {
                if (!ok[u]) continue;
                const float4 x = *reinterpret_cast<const float4*>(tile + slot * block + (long long)u * rstep * BN);
                s[u].x += x.x;
                s[u].y += x.y;
                s[u].z += x.z;
                s[u].w += x.w;
            }
        }
#pragma unroll
        for (int u = 0; u < kRowsPerThread; ++u) {
            if (!ok[u]) continue;
            float* row = C + (long long)(tm * rows + r0 + u * rstep) * ldc;
            if (a.scaled)
                store_row4_scaled(row, n, a.N, s[u], vec_c != 0, a.alpha, a.beta);
            else
                store_row4(row, n, a.N, s[u], vec_c != 0);
        }
    }
}

// ------------------------------------------------------------ tiled path
//
// Small products, where launch count and latency dominate: no pre-pass.  The
// shared-memory tiling of the pages ("Shared Memory와 Tiling"; PMPP ch. 5
// notes §5.4-§5.5) with register blocking: a 64 x 64 output tile per
// 256-thread block, K staged 16 at a time in shared memory (A transposed to
// [k][row], B as [k][col]), each thread accumulating a 4 x 4 block in fp32
// with fused multiply-adds, the next K stage loaded into registers while the
// current one is used (double buffer).  Out-of-range elements load as zeros
// (ghost elements) and the store is guarded.  Either operand may be stored
// transposed; alpha and beta are applied at the store.  With few tiles K is
// split over a cluster of S blocks per tile (S <= 8): block rank s runs K
// slice s (zeros past the slice's end) and leaves its partial tile in its
// shared memory; after a cluster barrier each block adds its share of the
// tile's 16-byte groups over all S partials, read from the other blocks'
// shared memory, in slice order 0, 1, ... (deterministic), and stores them.
// One launch, no workspace.  (A 4-stage cp.async version of the tile was
// measured slower on small products: 18.2 vs 15.9 us at 256^3.)
constexpr int kTiledThreads = 256;  // tile shape kTiledBM x kTiledBN, K stage kTiledBK (tg_internal.h)
constexpr int kTiledPitch = kTiledBM + 4;  // [k][row] rows padded: 16-byte aligned, 2-way store conflicts at most

struct TiledArgs {
    const float* A;
    const float* B;
    float* C;
    long long lda, ldb, ldc;
    int M, N, K;
    int op_a, op_b;
    float alpha, beta;
    int scaled, vec_c;
    int split, nkb;  // K slices (blocks of a cluster per tile); K blocks of kTiledBK
};

// This thread's 4 values of the A stage at K offset k0: op N: 4 consecutive k
// of row r (r = tid / 4, k = 4 * (tid % 4)); op T (stored K x M): row
// r = tid % 64 at k = 4 * (tid / 64) + q, consecutive threads reading
// consecutive rows.
__device__ __forceinline__ void tiled_load_a(const TiledArgs& a, int row0, int k0, int kend, float (&v)[4], int& r,
                                             int& k) {
    const int tid = threadIdx.x;
    if (a.op_a == TG_OP_N) {
        r = tid >> 2;
        k = (tid & 3) * 4;
    } else {
        r = tid & 63;
        k = (tid >> 6) * 4;
    }
    const int gi = row0 + r;
#pragma unroll
    for (int q = 0; q < 4; ++q) {
        const int gk = k0 + k + q;
        const bool in = gi < a.M && gk < kend;
        v[q] = in ? (a.op_a == TG_OP_N ? a.A[(long long)gi * a.lda + gk] : a.A[(long long)gk * a.lda + gi]) : 0.0f;
    }
}

// This thread's 4 values of the B stage: op N: 4 consecutive columns of row
// k (k = tid / 16, c = 4 * (tid % 16)); op T (stored N x K): column
// c = tid / 4, 4 consecutive k from 4 * (tid % 4).
__device__ __forceinline__ void tiled_load_b(const TiledArgs& a, int col0, int k0, int kend, float (&v)[4], int& c,
                                             int& k) {
    const int tid = threadIdx.x;
    if (a.op_b == TG_OP_N) {
        k = tid >> 4;
        c = (tid & 15) * 4;
    } else {
        c = tid >> 2;
        k = (tid & 3) * 4;
    }
#pragma unroll
    for (int q = 0; q < 4; ++q) {
        const int gk = k0 + k + (a.op_b == TG_OP_N ? 0 : q);
        const int gj = col0 + c + (a.op_b == TG_OP_N ? q : 0);
        const bool in = gj < a.N && gk < kend;
        v[q] = in ? (a.op_b == TG_OP_N ? a.B[(long long)gk * a.ldb + gj] : a.B[(long long)gj * a.ldb + gk]) : 0.0f;
    }
}

__global__ void __launch_bounds__(kTiledThreads) tiled_gemm_kernel(TiledArgs a) {
    __shared__ __align__(16) float As[2][kTiledBK][kTiledPitch];
    __shared__ __align__(16) float Bs[2][kTiledBK][kTiledPitch];
    __shared__ __align__(16) float part[kTiledBM][kTiledBN];  // this K slice's partial tile (split > 1)
    const int tid = threadIdx.x, tx = tid & 15, ty = tid >> 4;
    const int tiles_n = (a.N + kTiledBN - 1) / kTiledBN;
    // a cluster of `split` consecutive blocks per tile, block s of it on K slice s
    const int tile = (int)(blockIdx.x / a.split), s = (int)(blockIdx.x % a.split);
    const int row0 = (tile / tiles_n) * kTiledBM, col0 = (tile % tiles_n) * kTiledBN;
    // this slice's K range: whole 16-wide blocks, the last one clipped to K
    const int kbeg = (int)((long long)s * a.nkb / a.split) * kTiledBK;
    const int kend = min(a.K, (int)((long long)(s + 1) * a.nkb / a.split) * kTiledBK);
    grid_dep_wait();  // operands written by the previous kernel of the stream
    float acc[4][4];
#pragma unroll
    for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) acc[i][j] = 0.0f;

    float va[4], vb[4];
    int ar, ak, bc, bk;
    tiled_load_a(a, row0, kbeg, kend, va, ar, ak);
    tiled_load_b(a, col0, kbeg, kend, vb, bc, bk);
    int buf = 0;
    for (int k0 = kbeg; k0 < kend; k0 += kTiledBK) {
#pragma unroll
        for (int q = 0; q < 4; ++q) As[buf][ak + q][ar] = va[q];
        if (a.op_b == TG_OP_N) {
#pragma unroll
            for (int q = 0; q < 4; ++q) Bs[buf][bk][bc + q] = vb[q];
        } else {
#pragma unroll
            for (int q = 0; q < 4; ++q) Bs[buf][bk + q][bc] = vb[q];
        }
        __syncthreads();
        if (k0 + kTiledBK < kend) {  // the next stage's loads overlap this stage's math
            tiled_load_a(a, row0, k0 + kTiledBK, kend, va, ar, ak);
            tiled_load_b(a, col0, k0 + kTiledBK, kend, vb, bc, bk);
        }
#pragma unroll
        for (int k = 0; k < kTiledBK; ++k) {
            const float4 x = *reinterpret_cast<const float4*>(&As[buf][k][ty * 4]);
            const float4 y = *reinterpret_cast<const float4*>(&Bs[buf][k][tx * 4]);
            const float xa[4] = {x.x, x.y, x.z, x.w}, yb[4] = {y.x, y.y, y.z, y.w};
#pragma unroll
            for (int i = 0; i < 4; ++i)
#pragma unroll
                for (int j = 0; j < 4; ++j) acc[i][j] = fmaf(xa[i], yb[j], acc[i][j]);
        }
        // the other buffer is free: every thread passed this stage's barrier
        // after its last reads of it
        buf ^= 1;
    }
    grid_dep_launch();
    if (a.split > 1) {
        // partials into shared memory; the cluster barrier (release / acquire
        // at cluster scope) makes every block's partial visible to the others
#pragma unroll
        for (int i = 0; i < 4; ++i)
            *reinterpret_cast<float4*>(&part[ty * 4 + i][tx * 4]) =
                make_float4(acc[i][0], acc[i][1], acc[i][2], acc[i][3]);
        cluster_sync_all();
        // 16-byte group g of the tile (row g / 16, columns 4 (g % 16)..) for
        // g = s, s + split, ...: the sum over the slices in order
        for (int g = s + a.split * tid; g < kTiledBM * kTiledBN / 4; g += a.split * kTiledThreads) {
            const int rl = g >> 4, cl = (g & 15) * 4;
            // every slice's group first (the remote loads overlap), then the
            // sum in slice order
            float4 x[kTiledMaxSplit];
#pragma unroll
            for (int j = 0; j < kTiledMaxSplit; ++j)
                if (j < a.split) x[j] = ld_shared_cluster_f4(cluster_addr(&part[rl][cl], (uint32_t)j));
            float4 v = x[0];
#pragma unroll
            for (int j = 1; j < kTiledMaxSplit; ++j) {
                if (j < a.split) {
                    v.x += x[j].x;
                    v.y += x[j].y;
                    v.z += x[j].z;
                    v.w += x[j].w;
                }
            }
            const int r = row0 + rl;
            if (r < a.M) {
                float* row = a.C + (long long)r * a.ldc;
                if (a.scaled)
                    store_row4_scaled(row, col0 + cl, a.N, v, a.vec_c != 0, a.alpha, a.beta);
                else
                    store_row4(row, col0 + cl, a.N, v, a.vec_c != 0);
            }
        }
        cluster_sync_all();  // no block leaves while others may still read its partial
        return;
    }
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const int r = row0 + ty * 4 + i;
        if (r >= a.M) continue;
        float* row = a.C + (long long)r * a.ldc;
        const float4 v = make_float4(acc[i][0], acc[i][1], acc[i][2], acc[i][3]);
        if (a.scaled)
            store_row4_scaled(row, col0 + tx * 4, a.N, v, a.vec_c != 0, a.alpha, a.beta);
        else
            store_row4(row, col0 + tx * 4, a.N, v, a.vec_c != 0);
    }
}

// K == 0: the empty sum, so C = beta * C (C not read when beta == 0).
__global__ void __launch_bounds__(256) scale_c_kernel(float* C, long long ldc, int M, int N, float beta) {
    const long long total = (long long)M * N;
    for (long long i = blockIdx.x * (long long)blockDim.x + threadIdx.x; i < total;
         i += (long long)gridDim.x * blockDim.x) {
        float* c = C + (i / N) * ldc + (i % N);
        *c = beta != 0.0f ? beta * *c : 0.0f;
    }
}

// Waits on an mbarrier that nothing arrives on; the bounded wait gives up,
// records kSiteSelftest and the kernel returns normally.
__global__ void wait_selftest_kernel(uint64_t timeout_ns) {
    __shared__ uint64_t bar;
    if (threadIdx.x == 0) {
        mbar_init(&bar, 1);
        fence_barrier_init();
    }
    __syncthreads();
    if (threadIdx.x == 0) {
        const WaitCtl wc{&g_error_word, timeout_ns};
        (void)mbar_wait(&bar, 0, wc, kSiteSelftest);
    }
}

// ------------------------------------------------------------------ host

namespace {

uint64_t default_timeout_ns() {
    static uint64_t ns = [] {
        const char* s = std::getenv("TG_WAIT_TIMEOUT_MS");
        long long ms = s ? std::atoll(s) : 0;
        if (ms <= 0) ms = 4000;
        return (uint64_t)ms * 1000000ull;
    }();
    return ns;
}

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                             &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    });
    return fn;
}

// 2-D fp32 tensor map: `inner` elements per row (the valid extent; anything
// beyond reads as zero), `outer` rows, `row_bytes` between rows.
bool make_map(CUtensorMap* m, const void* base, uint64_t inner, uint64_t outer, uint64_t row_bytes,
              uint32_t box_inner, uint32_t box_outer, CUtensorMapSwizzle sw) {
    auto fn = encode_fn();
    if (!fn) return false;
    const cuuint64_t dims[2] = {inner, outer};
    const cuuint64_t strides[1] = {row_bytes};
    const cuuint32_t box[2] = {box_inner, box_outer};
    const cuuint32_t estr[2] = {1, 1};
    return fn(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, const_cast<void*>(base), dims, strides, box,
              estr, CU_TENSOR_MAP_INTERLEAVE_NONE, sw, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

int elementwise_grid(long long work, int per_block) {
    long long g = (work + per_block - 1) / per_block;
    if (g < 1) g = 1;
    if (g > 4096) g = 4096;
    return (int)g;
}

tg_status last_launch_status() {
    return cudaGetLastError() == cudaSuccess ? TG_OK : TG_ERR_CUDA;
}

// Kernels after the first of a call are launched with programmatic stream
// serialization (programmatic dependent launch), so their launch and set-up
// overlap the end of the kernel before them; each waits (grid_dep_wait)
// before it reads that kernel's output.  TG_PDL=0 launches them plainly.
bool pdl_enabled() {
    static const bool on = [] {
        const char* e = std::getenv("TG_PDL");
        return !(e != nullptr && std::strcmp(e, "0") == 0);
    }();
    return on;
}

// NVTX ranges around the launches of one call (pre-pass, GEMM, reduce), so a
// profiler can select a phase (e.g. ncu --nvtx --nvtx-include "tg_gemm/").
// Off unless TG_NVTX=1: the ranges cost a little host time per call.  NVTX
// is header-only and does nothing unless a profiler has attached its
// injection library.
bool nvtx_enabled() {
    static const bool on = [] {
        const char* e = std::getenv("TG_NVTX");
        return e != nullptr && std::strcmp(e, "1") == 0;
    }();
    return on;
}

struct NvtxRange {
    bool on;
    explicit NvtxRange(const char* name) : on(nvtx_enabled()) {
        if (on) nvtxRangePushA(name);
    }
    ~NvtxRange() {
        if (on) nvtxRangePop();
    }
    NvtxRange(const NvtxRange&) = delete;
    NvtxRange& operator=(const NvtxRange&) = delete;
};

template <typename... KArgs, typename... Args>
tg_status launch_dependent(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t stream,
                           unsigned cluster, Args&&... args) {
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[2];
    unsigned n = 0;
    if (cluster > 1) {
        attr[n].id = cudaLaunchAttributeClusterDimension;
        attr[n].val.clusterDim.x = cluster;
        attr[n].val.clusterDim.y = 1;
        attr[n].val.clusterDim.z = 1;
        ++n;
    }
    if (pdl_enabled()) {
        attr[n].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[n].val.programmaticStreamSerializationAllowed = 1;
        ++n;
    }
    cfg.attrs = attr;
    cfg.numAttrs = n;
    if (cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...) != cudaSuccess) {
        cudaGetLastError();
        return TG_ERR_CUDA;
    }
    return TG_OK;
}

}  // namespace

// Resident 256-thread blocks per SM of the two pre-pass kernels (the grid is
// sized to exactly fill the GPU once).
int g_prepass_blocks_per_sm[5] = {4, 4, 4, 4, 4};
// CTA pairs of the 3xTF32 kernel resident at once (0 = unknown).
int g_tf32_pair_clusters = 0;

tg_status prepare_device_kernels() {
    int nb = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&nb, prepass_kernel<kPack>, 256, 0) == cudaSuccess && nb > 0)
        g_prepass_blocks_per_sm[kPack] = nb;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&nb, prepass_kernel<kSplitTf32>, 256, 0) == cudaSuccess &&
        nb > 0)
        g_prepass_blocks_per_sm[kSplitTf32] = nb;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&nb, prepass_kernel<kSplitBf16>, 256, 0) == cudaSuccess &&
        nb > 0)
        g_prepass_blocks_per_sm[kSplitBf16] = nb;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&nb, prepass_kernel<kSplitTf32H>, 256, 0) == cudaSuccess &&
        nb > 0)
        g_prepass_blocks_per_sm[kSplitTf32H] = nb;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&nb, prepass_kernel<kSplitBf16H>, 256, 0) == cudaSuccess &&
        nb > 0)
        g_prepass_blocks_per_sm[kSplitBf16H] = nb;
    // The warpgroup register splits of both GEMM kernels only balance when the
    // kernels are launched with exactly the register counts they were designed
    // for; refuse to run a build that differs.
    cudaFuncAttributes fa{};
    if (cudaFuncGetAttributes(&fa, ffma_gemm_kernel) != cudaSuccess) return TG_ERR_CUDA;
    if (fa.numRegs != kFfmaLaunchRegs) return TG_ERR_CUDA;
    if (cudaFuncSetAttribute(ffma_gemm_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)kFfmaSmemBytes) != cudaSuccess)
        return TG_ERR_CUDA;
    struct {
        void (*kern)(CUtensorMap, CUtensorMap, GemmArgs);
        size_t smem;
    } tf_kernels[] = {{tf32x3_gemm_kernel<1, false>, kTfSmemBytes},
                      {tf32x3_gemm_kernel<2, false>, kTfSmemBytes},
                      {tf32x3_gemm_kernel<2, true>, kTfSmemBytesPairMma},
                      {tf32x3_gemm_kernel<2, true, false, true>, kTfSmemBytesPairMma},
                      {tf32x3_gemm_kernel<2, true, true, true>, kTfSmemBytesPairMma},
                      {tf32x3_gemm_kernel<1, false, true>, kTfSmemBytes},
                      {tf32x3_gemm_kernel<2, false, true>, kTfSmemBytes},
                      {tf32x3_gemm_kernel<2, true, true>, kTfSmemBytesPairMma}};
    for (const auto& k : tf_kernels) {
        if (cudaFuncGetAttributes(&fa, k.kern) != cudaSuccess) return TG_ERR_CUDA;
        if (fa.numRegs != kTfLaunchRegs) return TG_ERR_CUDA;
        if (cudaFuncSetAttribute(k.kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)k.smem) != cudaSuccess)
            return TG_ERR_CUDA;
    }
    // how many CTA pairs the GPU holds at once (one CTA per SM)
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = dim3(2);
    cfg.blockDim = dim3(kTfThreads);
    cfg.dynamicSmemBytes = kTfSmemBytesPairMma;
    cudaLaunchAttribute attr{};
    attr.id = cudaLaunchAttributeClusterDimension;
    attr.val.clusterDim.x = 2;
    attr.val.clusterDim.y = 1;
    attr.val.clusterDim.z = 1;
    cfg.attrs = &attr;
    cfg.numAttrs = 1;
    int clusters = 0;
    if (cudaOccupancyMaxActiveClusters(&clusters, tf32x3_gemm_kernel<2, true>, &cfg) == cudaSuccess && clusters > 0)
        g_tf32_pair_clusters = clusters;
    else
        cudaGetLastError();
    return TG_OK;
}

tg_status launch_plan(const Plan& p, const float* A, const float* B, float* C, void* ws,
                      cudaStream_t stream, cudaEvent_t ev_begin, cudaEvent_t ev_end) {
    if (p.M == 0 || p.N == 0) return TG_OK;
    if (p.zero_fill) {  // K == 0: C = beta * C
        scale_c_kernel<<<elementwise_grid((long long)p.M * p.N, 256), 256, 0, stream>>>(C, p.ldc, p.M, p.N,
                                                                                       p.beta);
        return last_launch_status();
    }
    if (p.path == TG_PATH_TILED) {  // one launch, operands read in place
        TiledArgs ta{};
        ta.A = A;
        ta.B = B;
        ta.C = C;
        ta.lda = p.lda;
        ta.ldb = p.ldb;
        ta.ldc = p.ldc;
        ta.M = p.M;
        ta.N = p.N;
        ta.K = p.K;
        ta.op_a = p.op_a;
        ta.op_b = p.op_b;
        ta.alpha = p.alpha;
        ta.beta = p.beta;
        ta.scaled = (p.alpha != 1.0f || p.beta != 0.0f) ? 1 : 0;
        ta.vec_c = p.vec_c ? 1 : 0;
        ta.split = p.split;
        ta.nkb = p.nkb;
        if (ev_begin && cudaEventRecord(ev_begin, stream) != cudaSuccess) return TG_ERR_CUDA;
        {
            NvtxRange r("tg_gemm");
            // a cluster of split blocks per tile (one block each when K is not split)
            if (launch_dependent(tiled_gemm_kernel, dim3((unsigned)((long long)p.tiles_m * p.tiles_n * p.split)),
                                 dim3(kTiledThreads), 0, stream, (unsigned)p.split, ta) != TG_OK)
                return TG_ERR_CUDA;
        }
        if (ev_end && cudaEventRecord(ev_end, stream) != cudaSuccess) return TG_ERR_CUDA;
        return TG_OK;
    }
    uint8_t* w = static_cast<uint8_t*>(ws);
    GemmArgs ga{};
    ga.M = p.M;
    ga.N = p.N;
    ga.K = p.K;
    ga.pair = p.pair;
    ga.tiles_m = (p.tiles_m + p.pair - 1) / p.pair;
    ga.tiles_n = p.tiles_n;
    ga.split = p.split;
    ga.nkb = p.nkb;
    ga.units = p.units;
    ga.full_units = p.full_units;
    ga.tail_units = p.tail_units;
    ga.tail_lanes = p.tail_lanes;
    ga.tail_kx = p.tail_kx;
    ga.tail_slots = p.tail_slots;
    ga.tail = p.tail_lanes > 0 ? reinterpret_cast<float*>(w + p.off_tail) : nullptr;
    ga.alpha = p.alpha;
    ga.beta = p.beta;
    ga.scaled = (p.alpha != 1.0f || p.beta != 0.0f) ? 1 : 0;
    ga.timeout_ns = default_timeout_ns();
    if (p.split > 1) {
        ga.out = reinterpret_cast<float*>(w + p.off_part);
        ga.ldo = p.ldp;
        ga.slice_stride = p.part_stride;
        ga.vec_out = 1;
    } else {
        ga.out = C;
        ga.ldo = p.ldc;
        ga.slice_stride = 0;
        ga.vec_out = p.vec_c ? 1 : 0;
    }

    // Operand passes of the pre-pass.  A is stored M x K (op N) or K x M
    // (op T); B is stored K x N (op N) or N x K (op T).
    auto pass = [](const float* src, long long ld, int rows, int cols, int pitch, bool trans, float* d0,
                   int rows_out) {
        OperandPass o{};
        o.src = src;
        o.ld = ld;
        o.rows = rows_out;
        o.rows_valid = rows;
        o.cols = cols;
        o.pitch = pitch;
        o.trans = trans ? 1 : 0;
        o.vec = (reinterpret_cast<uintptr_t>(src) % 16 == 0 && ld % 4 == 0) ? 1 : 0;
        o.d0 = d0;
        o.tiles_c = (pitch + 63) / 64;
        o.items = trans ? (long long)((rows_out + 63) / 64) * o.tiles_c : (long long)rows_out * (pitch / 4);
        return o;
    };
    PrepassArgs pa{};
    // one full wave of resident blocks keeps HBM busy without a tail
    const bool mixed = p.path == TG_PATH_TF32_BF16;
    const int mode = mixed ? (p.raw_a ? kSplitBf16H : kSplitBf16)
                           : (p.path == TG_PATH_TF32X3 ? (p.raw_a ? kSplitTf32H : kSplitTf32) : kPack);
    const int prepass_grid = g_prepass_blocks_per_sm[mode] * p.num_sms;

    if (tensor_path(p.path)) {
        float* a_tiles = p.raw_a ? nullptr : (p.ext_a ? p.ext_a : reinterpret_cast<float*>(w + p.off_a0));
        float* b_tiles = p.ext_b ? p.ext_b : reinterpret_cast<float*>(w + p.off_b0);
        // split tiles: A [a_rows/128][k16/16] from op(A); B [b_rows/128][k16/16] from op(B)^T
        // (none for an operand the kernel splits itself)
        const bool need_a = !p.raw_a && !p.a_ready, need_b = !p.b_ready;
        pa.op[0] = pass(A, p.lda, p.M, p.K, p.k16, p.op_a == TG_OP_T, need_a ? a_tiles : nullptr, p.a_rows);
        pa.op[1] = pass(B, p.ldb, p.N, p.K, p.k16, p.op_b == TG_OP_N, need_b ? b_tiles : nullptr, p.b_rows);
        if (need_a || need_b) {
            NvtxRange r("tg_prepass");
            if (mode == kSplitBf16H)
                prepass_kernel<kSplitBf16H><<<prepass_grid, 256, 0, stream>>>(pa);
            else if (mixed)
                prepass_kernel<kSplitBf16><<<prepass_grid, 256, 0, stream>>>(pa);
            else if (mode == kSplitTf32H)
                prepass_kernel<kSplitTf32H><<<prepass_grid, 256, 0, stream>>>(pa);
            else
                prepass_kernel<kSplitTf32><<<prepass_grid, 256, 0, stream>>>(pa);
            if (last_launch_status() != TG_OK) return TG_ERR_CUDA;
        }
        ga.a_tiles = a_tiles;
        ga.b_tiles = b_tiles;
        ga.kbs = p.k16 / 16;
        if (ev_begin && cudaEventRecord(ev_begin, stream) != cudaSuccess) return TG_ERR_CUDA;
        // the pair-MMA form reads the split tiles through 2-D tensor maps: rows
        // of 32 floats (one tile row, hi and lo), boxes of one 128-row tile
        // (the plan keeps the per-CTA form when these 32-bit row coordinates
        // would overflow); a raw A through a map of the caller's matrix:
        // boxes of 16 K values x 128 rows, 64-byte swizzle, zeros past the
        // edges
        CUtensorMap mA{}, mB{};
        const bool pair_mma = p.pair_mma;
        if (pair_mma) {
            const bool ok_a =
                p.raw_a ? make_map(&mA, A, p.K, p.M, 4ull * p.lda, kTf32BK, kTf32BM, CU_TENSOR_MAP_SWIZZLE_64B)
                        : make_map(&mA, a_tiles, 32, (uint64_t)p.a_rows * ga.kbs, 128, 32, 128,
                                   CU_TENSOR_MAP_SWIZZLE_NONE);
            const bool ok_b =
                make_map(&mB, b_tiles, 32, (uint64_t)p.b_rows * ga.kbs, 128, 32, 128, CU_TENSOR_MAP_SWIZZLE_NONE);
            if (!ok_a || !ok_b) return TG_ERR_CUDA;
        }
        int clusters = p.grid / 2;
        if (g_tf32_pair_clusters > 0 && clusters > g_tf32_pair_clusters) clusters = g_tf32_pair_clusters;
        NvtxRange r("tg_gemm");
        void (*kern)(CUtensorMap, CUtensorMap, GemmArgs);
        if (p.pair == 2 && pair_mma && p.raw_a)
            kern = mixed ? tf32x3_gemm_kernel<2, true, true, true> : tf32x3_gemm_kernel<2, true, false, true>;
        else if (p.pair == 2)
            kern = pair_mma ? (mixed ? tf32x3_gemm_kernel<2, true, true> : tf32x3_gemm_kernel<2, true>)
                            : (mixed ? tf32x3_gemm_kernel<2, false, true> : tf32x3_gemm_kernel<2, false>);
        else
            kern = mixed ? tf32x3_gemm_kernel<1, false, true> : tf32x3_gemm_kernel<1, false>;
        if (launch_dependent(kern, dim3(p.pair == 2 ? 2 * clusters : p.grid), dim3(kTfThreads),
                             pair_mma ? kTfSmemBytesPairMma : kTfSmemBytes, stream, p.pair, mA, mB, ga) != TG_OK)
            return TG_ERR_CUDA;
        if (ev_end && cudaEventRecord(ev_end, stream) != cudaSuccess) return TG_ERR_CUDA;
    } else {
        const float* a_src = A;
        const float* b_src = B;
        long long a_row = p.lda, b_row = p.ldb;
        if (p.pack_a || p.pack_b) {
            // A_pack [M][k4] from op(A); B_pack [K][n4] from op(B)
            float* ap = p.pack_a ? reinterpret_cast<float*>(w + p.off_a0) : nullptr;
            float* bp = p.pack_b ? reinterpret_cast<float*>(w + p.off_b0) : nullptr;
            pa.op[0] = pass(A, p.lda, p.M, p.K, p.k4, p.op_a == TG_OP_T, ap, p.M);
            pa.op[1] = pass(B, p.ldb, p.K, p.N, p.n4, p.op_b == TG_OP_T, bp, p.K);
            NvtxRange r("tg_prepass");
            prepass_kernel<kPack><<<prepass_grid, 256, 0, stream>>>(pa);
            if (last_launch_status() != TG_OK) return TG_ERR_CUDA;
            if (p.pack_a) {
                a_src = ap;
                a_row = p.k4;
            }
            if (p.pack_b) {
                b_src = bp;
                b_row = p.n4;
            }
        }
        CUtensorMap mA, mB;
        if (!make_map(&mA, a_src, p.K, p.M, 4ull * a_row, kFfmaBK, kFfmaBM, CU_TENSOR_MAP_SWIZZLE_128B) ||
            !make_map(&mB, b_src, p.N, p.K, 4ull * b_row, kFfmaBN, kFfmaBK, CU_TENSOR_MAP_SWIZZLE_NONE))
            return TG_ERR_CUDA;
        if (ev_begin && cudaEventRecord(ev_begin, stream) != cudaSuccess) return TG_ERR_CUDA;
        NvtxRange r("tg_gemm");
        if (launch_dependent(ffma_gemm_kernel, dim3(p.grid), dim3(kFfmaThreads), kFfmaSmemBytes, stream, 1, mA, mB,
                             ga) != TG_OK)
            return TG_ERR_CUDA;
        if (ev_end && cudaEventRecord(ev_end, stream) != cudaSuccess) return TG_ERR_CUDA;
    }

    NvtxRange r("tg_reduce");
    if (p.tail_lanes > 0) {
        // bands of 4 rows x 256 threads' worth of 16-byte groups (see the kernel)
        static_assert(256 % (kTf32BN / 4) == 0 && 256 % (kFfmaBN / 4) == 0, "a pass covers whole rows");
        const long long work = p.tail_units * p.pair * p.bm * (p.bn / 4);
        if (launch_dependent(tail_reduce_kernel, dim3(elementwise_grid(work, 4 * 256)), dim3(256), 0, stream, 1, ga, C,
                             (long long)p.ldc, p.bm, p.bn, p.vec_c ? 1 : 0) != TG_OK)
            return TG_ERR_CUDA;
    }
    if (p.split > 1) {
        const long long work = (long long)p.M * ((p.N + 3) / 4);
        if (launch_dependent(splitk_reduce_kernel, dim3(elementwise_grid(work, 256)), dim3(256), 0, stream, 1,
                             (const float*)ga.out, p.ldp, p.part_stride, p.split, C, (long long)p.ldc, p.M, p.N,
                             p.vec_c ? 1 : 0, ga.scaled, p.alpha, p.beta) != TG_OK)
            return TG_ERR_CUDA;
    }
    return TG_OK;
}

tg_status read_error_word(cudaStream_t stream, bool clear, unsigned int* value) {
    unsigned int v = 0;
    if (cudaStreamSynchronize(stream) != cudaSuccess) return TG_ERR_CUDA;
    if (cudaMemcpyFromSymbol(&v, g_error_word, sizeof(v)) != cudaSuccess) return TG_ERR_CUDA;
    if (clear && v != 0) {
        const unsigned int zero = 0;
        if (cudaMemcpyToSymbol(g_error_word, &zero, sizeof(zero)) != cudaSuccess) return TG_ERR_CUDA;
    }
    *value = v;
    return TG_OK;
}

tg_status launch_wait_selftest(unsigned int timeout_us, cudaStream_t stream) {
    wait_selftest_kernel<<<1, 32, 0, stream>>>((uint64_t)timeout_us * 1000ull);
    return last_launch_status();
}

}  // namespace tg
