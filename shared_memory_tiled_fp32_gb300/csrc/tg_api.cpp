// C-ABI entry points of tg_sgemm.h: argument checks, per-device state
// (compute capability, SM count, kernel attributes, workspace memory pool),
// workspace handling and the host-buffer convenience call.
#include <cuda_runtime.h>

#include <algorithm>
#include <cstdint>
#include <cstdio>
#include <cstdlib>
#include <mutex>
#include <string>
#include <vector>

#include "tg_internal.h"

namespace tg {
namespace {

constexpr int kMaxDevices = 64;

struct DeviceState {
    bool ready = false;
    tg_status status = TG_OK;
    int num_sms = 0;
    cudaMemPool_t pool = nullptr;
};

std::mutex g_mutex;
DeviceState g_devices[kMaxDevices];

// Copy streams and events of the host-buffer entry point, per device: one
// event per copy in (8 row + 8 column blocks at most), one per output block
// (64 at most), and three for the start and the end of a call.
constexpr int kMaxHostEvents = 3 + 16 + 64;
struct HostPipe {
    bool ready = false;
    cudaStream_t s_in = nullptr, s_out = nullptr;
    cudaEvent_t ev[kMaxHostEvents] = {};
    std::mutex mu;
};
HostPipe g_host[kMaxDevices];

tg_status host_pipe(int dev, HostPipe** out) {
    std::lock_guard<std::mutex> lock(g_mutex);
    HostPipe& h = g_host[dev];
    if (!h.ready) {
        if (cudaStreamCreateWithFlags(&h.s_in, cudaStreamNonBlocking) != cudaSuccess ||
            cudaStreamCreateWithFlags(&h.s_out, cudaStreamNonBlocking) != cudaSuccess)
            return TG_ERR_CUDA;
        for (cudaEvent_t& e : h.ev)
            if (cudaEventCreateWithFlags(&e, cudaEventDisableTiming) != cudaSuccess) return TG_ERR_CUDA;
        h.ready = true;
    }
    *out = &h;
    return TG_OK;
}

// State of the current device, initialised on first use.
tg_status current_device(DeviceState** out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return TG_ERR_CUDA;
    if (dev < 0 || dev >= kMaxDevices) return TG_ERR_UNSUPPORTED_DEVICE;
    std::lock_guard<std::mutex> lock(g_mutex);
    DeviceState& d = g_devices[dev];
    if (!d.ready) {
        int major = 0, minor = 0, sms = 0;
        if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
            return TG_ERR_CUDA;
        d.ready = true;
        d.num_sms = sms;
        if (major != 10 || minor != 3) {
            d.status = TG_ERR_UNSUPPORTED_DEVICE;  // the kernels are built for sm_103a only
        } else {
            d.status = prepare_device_kernels();
            if (d.status == TG_OK) {
                // A private stream-ordered pool that keeps freed memory for reuse,
                // so repeated calls do not map and unmap their workspace.
                cudaMemPoolProps props{};
                props.allocType = cudaMemAllocationTypePinned;
                props.location.type = cudaMemLocationTypeDevice;
                props.location.id = dev;
                if (cudaMemPoolCreate(&d.pool, &props) != cudaSuccess) {
                    d.status = TG_ERR_CUDA;
                } else {
                    uint64_t keep = UINT64_MAX;
                    cudaMemPoolSetAttribute(d.pool, cudaMemPoolAttrReleaseThreshold, &keep);
                }
            }
        }
    }
    *out = &d;
    return d.status;
}

tg_sgemm_opts default_opts() {
    tg_sgemm_opts o{};
    o.path = TG_PATH_AUTO;
    return o;
}

void fill_info(const Plan& p, tg_plan_info* out) {
    out->path = p.path;
    out->split_k = p.split;
    out->block_m = p.bm;
    out->block_n = p.bn;
    out->block_k = p.bk;
    out->stages = p.stages;
    out->tiles_m = p.tiles_m;
    out->tiles_n = p.tiles_n;
    out->units = p.units;
    out->grid = p.grid;
    out->prepass = (tensor_path(p.path) && !p.zero_fill && p.M > 0 && p.N > 0) || p.pack_a || p.pack_b;
    out->launches = p.launches;
    out->workspace_bytes = p.ws_bytes;
    out->pair = p.pair;
    out->tail_units = p.tail_units;
    out->tail_lanes = p.tail_lanes;
    out->tail_kx = p.tail_kx;
    out->fused_split = p.raw_a ? 1 : 0;
}

}  // namespace

tg_status workspace_alloc(size_t bytes, cudaStream_t stream, void** out) {
    DeviceState* d = nullptr;
    const tg_status st = current_device(&d);
    if (st != TG_OK) return st;
    if (cudaMallocFromPoolAsync(out, bytes, d->pool, stream) != cudaSuccess) {
        cudaGetLastError();
        return TG_ERR_OUT_OF_MEMORY;
    }
    return TG_OK;
}

void workspace_free(void* p, cudaStream_t stream) { cudaFreeAsync(p, stream); }

}  // namespace tg

using namespace tg;

extern "C" {

const char* tg_status_string(tg_status s) {
    switch (s) {
        case TG_OK: return "TG_OK";
        case TG_ERR_INVALID_VALUE: return "TG_ERR_INVALID_VALUE: invalid argument";
        case TG_ERR_UNSUPPORTED_DEVICE: return "TG_ERR_UNSUPPORTED_DEVICE: needs a compute capability 10.3 (sm_103a) device";
        case TG_ERR_OUT_OF_MEMORY: return "TG_ERR_OUT_OF_MEMORY: workspace allocation failed";
        case TG_ERR_CUDA: return "TG_ERR_CUDA: a CUDA call or kernel launch failed";
        case TG_ERR_TIMEOUT: return "TG_ERR_TIMEOUT: a kernel gave up a bounded wait";
        case TG_ERR_WORKSPACE_TOO_SMALL: return "TG_ERR_WORKSPACE_TOO_SMALL: workspace smaller than required";
    }
    return "unknown tg_status";
}

int tg_sgemm_version(void) { return 103; }

tg_status tg_sgemm_plan_general(int op_a, int op_b, int M, int N, int K, const void* A, int lda,
                                const void* B, int ldb, const void* C, int ldc, int path,
                                int split_k, int num_sms, tg_plan_info* out) {
    if (out == nullptr) return TG_ERR_INVALID_VALUE;
    tg_status st = validate(op_a, op_b, M, N, K, A, lda, B, ldb, C, ldc, path, split_k, false);
    if (st != TG_OK) return st;
    if (num_sms <= 0) {
        DeviceState* d = nullptr;
        st = current_device(&d);
        if (d == nullptr) return st;
        num_sms = d->num_sms;
    }
    Plan p;
    make_plan(op_a, op_b, M, N, K, 1.0f, A, lda, B, ldb, 0.0f, C, ldc, path, split_k, num_sms, &p);
    fill_info(p, out);
    return TG_OK;
}

tg_status tg_sgemm_plan(int M, int N, int K, const void* A, int lda, const void* B, int ldb,
                        const void* C, int ldc, int path, int split_k, int num_sms,
                        tg_plan_info* out) {
    return tg_sgemm_plan_general(TG_OP_N, TG_OP_N, M, N, K, A, lda, B, ldb, C, ldc, path, split_k,
                                 num_sms, out);
}

size_t tg_sgemm_workspace_bytes(int M, int N, int K, const void* A, int lda, const void* B,
                                int ldb, const void* C, int ldc, int path, int split_k) {
    tg_plan_info info{};
    if (tg_sgemm_plan(M, N, K, A, lda, B, ldb, C, ldc, path, split_k, 0, &info) != TG_OK) return 0;
    return info.workspace_bytes;
}

tg_status tg_sgemm_general(int op_a, int op_b, int M, int N, int K, float alpha, const float* A,
                           int lda, const float* B, int ldb, float beta, float* C, int ldc,
                           cudaStream_t stream, const tg_sgemm_opts* opts) {
    const tg_sgemm_opts o = opts ? *opts : default_opts();
    tg_status st = validate(op_a, op_b, M, N, K, A, lda, B, ldb, C, ldc, o.path, o.split_k);
    if (st != TG_OK) return st;
    if (M == 0 || N == 0) return TG_OK;
    DeviceState* d = nullptr;
    st = current_device(&d);
    if (st != TG_OK) return st;

    Plan p;
    make_plan(op_a, op_b, M, N, K, alpha, A, lda, B, ldb, beta, C, ldc, o.path, o.split_k, d->num_sms, &p);
    void* ws = nullptr;
    bool owned = false;
    if (p.ws_bytes > 0) {
        if (o.workspace != nullptr) {
            if (o.workspace_bytes < p.ws_bytes) return TG_ERR_WORKSPACE_TOO_SMALL;
            if (reinterpret_cast<uintptr_t>(o.workspace) % kWsAlign != 0) return TG_ERR_INVALID_VALUE;
            ws = o.workspace;
        } else {
            if (cudaMallocFromPoolAsync(&ws, p.ws_bytes, d->pool, stream) != cudaSuccess) {
                cudaGetLastError();
                return TG_ERR_OUT_OF_MEMORY;
            }
            owned = true;
        }
    }
    st = launch_plan(p, A, B, C, ws, stream, o.main_begin, o.main_end);
    if (owned && cudaFreeAsync(ws, stream) != cudaSuccess && st == TG_OK) st = TG_ERR_CUDA;
    return st;
}

tg_status tg_sgemm_ex(int M, int N, int K, const float* A, int lda, const float* B, int ldb,
                      float* C, int ldc, cudaStream_t stream, const tg_sgemm_opts* opts) {
    return tg_sgemm_general(TG_OP_N, TG_OP_N, M, N, K, 1.0f, A, lda, B, ldb, 0.0f, C, ldc, stream, opts);
}

tg_status tg_sgemm(int M, int N, int K, const float* A, int lda, const float* B, int ldb,
                   float* C, int ldc, cudaStream_t stream) {
    return tg_sgemm_ex(M, N, K, A, lda, B, ldb, C, ldc, stream, nullptr);
}

namespace {

// TG_HOST_TRACE=1: tg_sgemm_host records a timing event after each copy in,
// around each product and after each copy out, and prints them (ms after the
// call's start) to stderr once the call has synchronised.
struct HostTrace {
    bool on = false;
    std::vector<std::pair<std::string, cudaEvent_t>> marks;
    explicit HostTrace(bool enable) : on(enable) {}
    void mark(const std::string& what, cudaStream_t s) {
        if (!on) return;
        cudaEvent_t e = nullptr;
        if (cudaEventCreate(&e) != cudaSuccess) return;
        cudaEventRecord(e, s);
        marks.emplace_back(what, e);
    }
    void print() {
        for (auto& m : marks) {
            float ms = 0.0f;
            if (on && cudaEventElapsedTime(&ms, marks.front().second, m.second) == cudaSuccess)
                std::fprintf(stderr, "tg_host_trace %8.3f ms %s\n", ms, m.first.c_str());
        }
    }
    ~HostTrace() {
        for (auto& m : marks) cudaEventDestroy(m.second);
    }
};

// Device memory of one host-buffer call: the 16-byte-pitched copies of A, B
// and C, the split tiles (all of B^T's, one A row block's) and the largest
// workspace any of its products needs.
struct HostBytes {
    size_t a = 0, b = 0, c = 0, b_split = 0, a_split = 0, ws_max = 0;
    size_t total() const { return a + b + c + b_split + a_split + ws_max; }
};

// Plan of product (i, j) of a host-buffer call.  The products share B's split
// tiles, written by the first row block's products, so their layout follows
// that row block: if its products split A in the kernel (which needs the
// fused kernel's tile layout for B), so may the others; a later row block
// that cannot (128 rows or fewer: no CTA pair) splits its own copy of B in
// its workspace instead of reading the shared one.  If the first row block
// cannot, no product does.
tg::Plan host_product_plan(const tg::HostBlocks& hb, int M, int N, int K, int i, int Nj, const void* Ai,
                           int lda, const void* Bj, int ldb, const void* Cij, int ldc, int path, int split_k,
                           int num_sms, bool* shared_b) {
    using namespace tg;
    const bool tf32 = tensor_path(path);
    Plan first;
    make_plan(TG_OP_N, TG_OP_N, hb.rows(0, M), Nj, K, 1.0f, Ai, lda, Bj, ldb, 0.0f, Cij, ldc, path, split_k,
              num_sms, &first, tf32, tf32);
    const bool fused_pipe = first.raw_a;
    Plan pl;
    make_plan(TG_OP_N, TG_OP_N, hb.rows(i, M), Nj, K, 1.0f, Ai, lda, Bj, ldb, 0.0f, Cij, ldc, path, split_k,
              num_sms, &pl, tf32, tf32, fused_pipe);
    *shared_b = tf32 && pl.raw_a == fused_pipe;
    if (tf32 && !*shared_b)  // its own split of B, in its workspace
        make_plan(TG_OP_N, TG_OP_N, hb.rows(i, M), Nj, K, 1.0f, Ai, lda, Bj, ldb, 0.0f, Cij, ldc, path,
                  split_k, num_sms, &pl, false, tf32, fused_pipe);
    return pl;
}

// The column offset and width of block j of row block i.
void host_block_cols(const tg::HostBlocks& hb, int N, int i, int j, int* j0, int* Nj) {
    if (hb.col_blocks(i) == 1) {
        *j0 = 0;
        *Nj = N;
    } else {
        *j0 = j * hb.nb;
        *Nj = std::min(hb.nb, N - *j0);
    }
}

HostBytes host_bytes(const tg::HostBlocks& hb, int M, int N, int K, int path, int split_k, int num_sms) {
    using namespace tg;
    const bool tf32 = tensor_path(path);
    const long long k4 = ((long long)std::max(K, 1) + 3) / 4 * 4, n4 = ((long long)N + 3) / 4 * 4;
    const long long k16 = ((long long)std::max(K, 1) + 15) / 16 * 16;
    auto align = [](size_t x) { return (x + kWsAlign - 1) / kWsAlign * kWsAlign; };
    HostBytes r;
    r.a = 4ull * M * k4;
    r.b = 4ull * (size_t)std::max(K, 1) * n4;
    r.c = 4ull * M * n4;
    const int mb_max = std::max(hb.first, hb.mb);
    r.b_split = tf32 ? align(8ull * ((N + 255) / 256 * 256) * k16) : 0;
    bool a_split = false;  // some row block's A is split by the pre-pass (not by the kernel)
    // placeholder pointers with the alignment the real ones will have
    const void* al = reinterpret_cast<const void*>(static_cast<uintptr_t>(1) << 20);
    // every product: a row block's shape (its rows, and column blocks or full
    // width) can differ from its neighbours' anywhere in the list
    for (int i = 0; i < hb.pm; ++i)
        for (int j = 0; j < hb.col_blocks(i); ++j) {
            int j0 = 0, Nj = 0;
            host_block_cols(hb, N, i, j, &j0, &Nj);
            bool shared_b = false;
            const Plan pl = host_product_plan(hb, M, N, K, i, Nj, al, (int)k4, al, (int)n4, al, (int)n4, path,
                                              split_k, num_sms, &shared_b);
            r.ws_max = std::max(r.ws_max, pl.ws_bytes);
            a_split = a_split || (tf32 && !pl.raw_a);
        }
    r.a_split = a_split ? align(8ull * ((mb_max + 255) / 256 * 256) * k16) : 0;
    return r;
}

}  // namespace

tg_status tg_sgemm_host(int M, int N, int K, const float* A, int lda, const float* B, int ldb,
                        float* C, int ldc, cudaStream_t stream, const tg_sgemm_opts* opts) {
    const tg_sgemm_opts o = opts ? *opts : default_opts();
    tg_status st = validate(TG_OP_N, TG_OP_N, M, N, K, A, lda, B, ldb, C, ldc, o.path, o.split_k);
    if (st != TG_OK) return st;
    if (M == 0 || N == 0) return TG_OK;
    DeviceState* d = nullptr;
    st = current_device(&d);
    if (st != TG_OK) return st;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return TG_ERR_CUDA;
    HostPipe* hp = nullptr;
    st = host_pipe(dev, &hp);
    if (st != TG_OK) return st;
    std::lock_guard<std::mutex> lock(hp->mu);  // one host-buffer call per device at a time

    const int path = o.path == TG_PATH_FFMA || o.path == TG_PATH_TF32_BF16 ? o.path : TG_PATH_TF32X3;
    const bool tf32 = tensor_path(path);
    const long long k4 = ((long long)std::max(K, 1) + 3) / 4 * 4, n4 = ((long long)N + 3) / 4 * 4;
    // Output blocks: C is cut into row blocks, the first ones also into
    // column blocks, so the first product needs only A_0 and B_0 on the
    // device; the copies of later blocks (in on s_in, out on s_out) overlap
    // the products of earlier ones.  Row blocks past hb.split are computed
    // full width once all of B is in.  A and B are split once, by the first
    // product that reads each block, into shared hi/lo regions.
    const HostBlocks hb = choose_host_blocks(M, N, K, path, d->num_sms);
    const int pm = hb.pm, pn = hb.pn, nb = hb.nb;
    auto block_cols = [&](int i, int j, int* j0, int* Nj) { host_block_cols(hb, N, i, j, j0, Nj); };
    // device copies: 16-byte row pitches, so TMA reads them in place
    const HostBytes hbytes = host_bytes(hb, M, N, K, path, o.split_k, d->num_sms);
    const size_t a_bytes = hbytes.a, b_bytes = hbytes.b, c_bytes = hbytes.c, b_split = hbytes.b_split,
                 a_split = hbytes.a_split;
    const long long k16 = ((long long)std::max(K, 1) + 15) / 16 * 16;
    const size_t ws_total = b_split + a_split + hbytes.ws_max;

    void *dA = nullptr, *dB = nullptr, *dC = nullptr, *W = nullptr;
    if (cudaMallocFromPoolAsync(&dA, a_bytes, d->pool, stream) != cudaSuccess ||
        cudaMallocFromPoolAsync(&dB, b_bytes, d->pool, stream) != cudaSuccess ||
        cudaMallocFromPoolAsync(&dC, c_bytes, d->pool, stream) != cudaSuccess ||
        (ws_total > 0 && cudaMallocFromPoolAsync(&W, ws_total, d->pool, stream) != cudaSuccess)) {
        cudaGetLastError();
        for (void* q : {dA, dB, dC, W})
            if (q) cudaFreeAsync(q, stream);
        cudaStreamSynchronize(stream);
        return TG_ERR_OUT_OF_MEMORY;
    }
    float* fA = static_cast<float*>(dA);
    float* fB = static_cast<float*>(dB);
    float* fC = static_cast<float*>(dC);
    uint8_t* w8 = static_cast<uint8_t*>(W);
    float* b_cat = reinterpret_cast<float*>(w8);
    float* a_cat = reinterpret_cast<float*>(w8 + b_split);
    uint8_t* wplan = w8 + b_split + a_split;
    // events: [0] start, [1] end of the copies in, [2] end of the copies
    // out, [3 + i] A_i in, [11 + j] B_j in, [19 + i*pn + j] C_ij computed
    cudaEvent_t* ev = hp->ev;
    const char* trace_env = std::getenv("TG_HOST_TRACE");
    HostTrace trace(trace_env != nullptr && trace_env[0] == '1');
    trace.mark("start", stream);
    bool ok = cudaEventRecord(ev[0], stream) == cudaSuccess &&
              cudaStreamWaitEvent(hp->s_in, ev[0], 0) == cudaSuccess &&
              cudaStreamWaitEvent(hp->s_out, ev[0], 0) == cudaSuccess;
    auto copy_a = [&](int i) {
        const int i0 = hb.row0(i), Mi = hb.rows(i, M);
        ok = ok &&
             cudaMemcpy2DAsync(fA + (size_t)i0 * k4, 4ull * k4, A + (size_t)i0 * lda, 4ull * lda, 4ull * K, Mi,
                               cudaMemcpyHostToDevice, hp->s_in) == cudaSuccess &&
             cudaEventRecord(ev[3 + i], hp->s_in) == cudaSuccess;
        trace.mark("in A" + std::to_string(i) + " rows " + std::to_string(Mi), hp->s_in);
    };
    auto copy_b = [&](int j) {
        const int j0 = j * nb, Nj = std::min(nb, N - j0);
        ok = ok &&
             cudaMemcpy2DAsync(fB + j0, 4ull * n4, B + j0, 4ull * ldb, 4ull * Nj, K, cudaMemcpyHostToDevice,
                               hp->s_in) == cudaSuccess &&
             cudaEventRecord(ev[11 + j], hp->s_in) == cudaSuccess;
        trace.mark("in B" + std::to_string(j) + " cols " + std::to_string(Nj), hp->s_in);
    };
    if (K > 0) {  // in the order the products first need them
        copy_a(0);
        for (int j = 0; j < pn; ++j) copy_b(j);
        for (int i = 1; i < pm; ++i) copy_a(i);
    }
    if (hb.defer_out)  // the copies out start once the copies in are done
        ok = ok && cudaEventRecord(ev[1], hp->s_in) == cudaSuccess &&
             cudaStreamWaitEvent(hp->s_out, ev[1], 0) == cudaSuccess;
    st = ok ? TG_OK : TG_ERR_CUDA;
    for (int i = 0; st == TG_OK && i < pm; ++i) {
        const int nc = hb.col_blocks(i);
        for (int j = 0; st == TG_OK && j < nc; ++j) {
            const int i0 = hb.row0(i), Mi = hb.rows(i, M);
            int j0 = 0, Nj = 0;
            block_cols(i, j, &j0, &Nj);
            // B_j's copy for the first row block; all of B for a full-width one
            const int b_event = nc == 1 ? 11 + pn - 1 : 11 + j;
            if (K > 0 && ((j == 0 && cudaStreamWaitEvent(stream, ev[3 + i], 0) != cudaSuccess) ||
                          ((i == 0 || nc == 1) && cudaStreamWaitEvent(stream, ev[b_event], 0) != cudaSuccess))) {
                st = TG_ERR_CUDA;
                break;
            }
            const float* Ai = fA + (size_t)i0 * k4;
            const float* Bj = fB + j0;
            float* Cij = fC + (size_t)i0 * n4 + j0;
            bool shared_b = false;
            Plan pl = host_product_plan(hb, M, N, K, i, Nj, Ai, (int)k4, Bj, (int)n4, Cij, (int)n4, path,
                                        o.split_k, d->num_sms, &shared_b);
            (void)Mi;
            if (tf32) {  // A_i split by its first product (j == 0), B_j by its first (i == 0);
                         // an A_i the kernel splits itself is read in place
                if (!pl.raw_a) {
                    pl.ext_a = a_cat;
                    pl.a_ready = j > 0;
                }
                if (shared_b) {
                    pl.ext_b = b_cat + (size_t)j0 * 2 * k16;
                    pl.b_ready = i > 0;
                }
            }
            const std::string blk = std::to_string(i) + "," + std::to_string(j) + " (" + std::to_string(Mi) +
                                    " x " + std::to_string(Nj) + ")";
            trace.mark("product " + blk + " begins", stream);
            st = launch_plan(pl, Ai, Bj, Cij, wplan, stream, nullptr, nullptr);
            if (st != TG_OK) break;
            trace.mark("product " + blk + " ends", stream);
            cudaEvent_t done = ev[19 + i * pn + j];
            if (cudaEventRecord(done, stream) != cudaSuccess || cudaStreamWaitEvent(hp->s_out, done, 0) != cudaSuccess ||
                cudaMemcpy2DAsync(C + (size_t)i0 * ldc + j0, 4ull * ldc, Cij, 4ull * n4, 4ull * Nj, Mi,
                                  cudaMemcpyDeviceToHost, hp->s_out) != cudaSuccess)
                st = TG_ERR_CUDA;
            trace.mark("out " + blk, hp->s_out);
        }
    }
    // the buffers are released on `stream` once both copy streams are done
    cudaEventRecord(ev[2], hp->s_out);
    cudaStreamWaitEvent(stream, ev[2], 0);
    cudaEventRecord(ev[1], hp->s_in);
    cudaStreamWaitEvent(stream, ev[1], 0);
    for (void* q : {dA, dB, dC, W})
        if (q) cudaFreeAsync(q, stream);
    if (cudaStreamSynchronize(stream) != cudaSuccess) return TG_ERR_CUDA;
    if (st != TG_OK) return st;
    trace.print();
    unsigned int word = 0;
    st = read_error_word(stream, true, &word);
    if (st != TG_OK) return st;
    return word != 0 ? TG_ERR_TIMEOUT : TG_OK;
}

tg_status tg_sgemm_host_device_bytes(int M, int N, int K, int path, int split_k, int num_sms, size_t* total,
                                     size_t* product_workspace) {
    using namespace tg;
    if (M < 0 || N < 0 || K < 0 || split_k < 0 || total == nullptr) return TG_ERR_INVALID_VALUE;
    if (path != TG_PATH_AUTO && path != TG_PATH_FFMA && path != TG_PATH_TF32X3 && path != TG_PATH_TF32_BF16)
        return TG_ERR_INVALID_VALUE;
    if (num_sms <= 0) {
        DeviceState* d = nullptr;
        const tg_status st = current_device(&d);
        if (st != TG_OK) return st;
        num_sms = d->num_sms;
    }
    *total = 0;
    if (product_workspace != nullptr) *product_workspace = 0;
    if (M == 0 || N == 0) return TG_OK;
    const int p = path == TG_PATH_FFMA || path == TG_PATH_TF32_BF16 ? path : TG_PATH_TF32X3;
    const HostBytes b = host_bytes(choose_host_blocks(M, N, K, p, num_sms), M, N, K, p, split_k, num_sms);
    *total = b.total();
    if (product_workspace != nullptr) *product_workspace = b.ws_max;
    return TG_OK;
}

tg_status tg_sgemm_host_blocks(int M, int N, int K, int path, int num_sms, tg_host_blocks_info* out) {
    using namespace tg;
    if (M < 0 || N < 0 || K < 0 || out == nullptr) return TG_ERR_INVALID_VALUE;
    if (path != TG_PATH_AUTO && path != TG_PATH_FFMA && path != TG_PATH_TF32X3 && path != TG_PATH_TF32_BF16)
        return TG_ERR_INVALID_VALUE;
    if (num_sms <= 0) {
        DeviceState* d = nullptr;
        const tg_status st = current_device(&d);
        if (st != TG_OK) return st;
        num_sms = d->num_sms;
    }
    const HostBlocks hb = choose_host_blocks(
        M, N, K, path == TG_PATH_FFMA || path == TG_PATH_TF32_BF16 ? path : TG_PATH_TF32X3, num_sms);
    out->row_blocks = hb.pm;
    out->col_blocks = hb.pn;
    out->first_block_rows = hb.first;
    out->block_rows = hb.mb;
    out->block_cols = hb.nb;
    out->split_row_blocks = hb.split;
    out->defer_copies_out = hb.defer_out ? 1 : 0;
    out->model_ms = hb.model_ms;
    return TG_OK;
}

tg_status tg_sgemm_sync_status(cudaStream_t stream) {
    unsigned int word = 0;
    tg_status st = read_error_word(stream, true, &word);
    if (st != TG_OK) return st;
    return word != 0 ? TG_ERR_TIMEOUT : TG_OK;
}

unsigned int tg_sgemm_error_site(cudaStream_t stream) {
    unsigned int word = 0;
    if (read_error_word(stream, false, &word) != TG_OK) return 0xFFFFFFFFu;
    return word;
}

tg_status tg_selftest_wait_timeout(unsigned int timeout_us, cudaStream_t stream) {
    if (timeout_us < 1 || timeout_us > 10000000u) return TG_ERR_INVALID_VALUE;
    DeviceState* d = nullptr;
    tg_status st = current_device(&d);
    if (st != TG_OK) return st;
    return launch_wait_selftest(timeout_us, stream);
}

}  // extern "C"
