// C-ABI entry points of tg_sgemm.h: argument checks, per-device state
// (compute capability, SM count, kernel attributes, workspace memory pool),
// workspace handling and the host-buffer convenience call.
#include <cuda_runtime.h>

#include <cstdint>
#include <mutex>

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
    out->prepass = (p.path == TG_PATH_TF32X3 && !p.zero_fill && p.M > 0 && p.N > 0) || p.pack_a || p.pack_b;
    out->launches = p.launches;
    out->workspace_bytes = p.ws_bytes;
    out->pair = p.pair;
    out->tail_units = p.tail_units;
    out->tail_split = p.tail_split;
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

int tg_sgemm_version(void) { return 100; }

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

tg_status tg_sgemm_host(int M, int N, int K, const float* A, int lda, const float* B, int ldb,
                        float* C, int ldc, cudaStream_t stream, const tg_sgemm_opts* opts) {
    const tg_sgemm_opts o = opts ? *opts : default_opts();
    tg_status st = validate(TG_OP_N, TG_OP_N, M, N, K, A, lda, B, ldb, C, ldc, o.path, o.split_k);
    if (st != TG_OK) return st;
    if (M == 0 || N == 0) return TG_OK;
    DeviceState* d = nullptr;
    st = current_device(&d);
    if (st != TG_OK) return st;

    const int dlda = K > 0 ? K : 1, dldb = N, dldc = N;
    void *dA = nullptr, *dB = nullptr, *dC = nullptr;
    const size_t a_bytes = 4ull * M * (size_t)(K > 0 ? K : 1);
    const size_t b_bytes = 4ull * (size_t)(K > 0 ? K : 1) * N;
    const size_t c_bytes = 4ull * M * N;
    if (cudaMallocFromPoolAsync(&dA, a_bytes, d->pool, stream) != cudaSuccess ||
        cudaMallocFromPoolAsync(&dB, b_bytes, d->pool, stream) != cudaSuccess ||
        cudaMallocFromPoolAsync(&dC, c_bytes, d->pool, stream) != cudaSuccess) {
        cudaGetLastError();
        if (dA) cudaFreeAsync(dA, stream);
        if (dB) cudaFreeAsync(dB, stream);
        if (dC) cudaFreeAsync(dC, stream);
        cudaStreamSynchronize(stream);
        return TG_ERR_OUT_OF_MEMORY;
    }
    bool ok = true;
    if (K > 0) {
        ok = ok && cudaMemcpy2DAsync(dA, 4ull * dlda, A, 4ull * lda, 4ull * K, M,
                                     cudaMemcpyHostToDevice, stream) == cudaSuccess;
        ok = ok && cudaMemcpy2DAsync(dB, 4ull * dldb, B, 4ull * ldb, 4ull * N, K,
                                     cudaMemcpyHostToDevice, stream) == cudaSuccess;
    }
    if (ok) {
        st = tg_sgemm_ex(M, N, K, static_cast<const float*>(dA), dlda, static_cast<const float*>(dB),
                         dldb, static_cast<float*>(dC), dldc, stream, &o);
        ok = st == TG_OK;
    } else {
        st = TG_ERR_CUDA;
    }
    if (ok && cudaMemcpy2DAsync(C, 4ull * ldc, dC, 4ull * dldc, 4ull * N, M, cudaMemcpyDeviceToHost,
                                stream) != cudaSuccess)
        st = TG_ERR_CUDA;
    cudaFreeAsync(dA, stream);
    cudaFreeAsync(dB, stream);
    cudaFreeAsync(dC, stream);
    if (cudaStreamSynchronize(stream) != cudaSuccess) return TG_ERR_CUDA;
    if (st != TG_OK) return st;
    unsigned int word = 0;
    st = read_error_word(stream, true, &word);
    if (st != TG_OK) return st;
    return word != 0 ? TG_ERR_TIMEOUT : TG_OK;
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
