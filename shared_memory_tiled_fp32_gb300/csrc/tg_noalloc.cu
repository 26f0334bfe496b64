// tg_sgemm_noalloc: the 3xTF32 product for callers that cannot allocate
// device memory at call time.
//
// tg_sgemm needs scratch memory (the hi/lo tf32 copies of B, and of A when
// the GEMM kernel cannot split A itself; the K-slice or balanced-tail
// partials when K is shared out) and normally takes it from a stream-ordered
// memory pool or from the caller.  Some callers can do neither: a host
// application that owns the whole device-memory budget through its own
// allocator and forbids libraries from allocating, a latency-critical loop
// that must never enter the CUDA allocator, or code that must not be able to
// fail with out-of-memory once it is running.  For them this file reserves a
// fixed scratch array in device memory when the library's module is loaded,
// and the entry point below runs the same pre-pass, GEMM and reduce kernels
// with their workspace placed in that array.  It calls no cudaMalloc,
// cudaFree or other allocating routine.
#include <cuda_runtime.h>

#include <mutex>

#include "tg_internal.h"

namespace tg {
namespace {

// The scratch.  Every GPU on which CUDA loads this file's device code (with
// lazy loading: at the first tg_sgemm_noalloc call there) holds these
// TG_SGEMM_NOALLOC_SCRATCH_BYTES bytes until the process exits.  In host
// code `g_noalloc_scratch` names a host-side stand-in, not device memory: its
// device address is fetched with cudaGetSymbolAddress below.
static __device__ __align__(256) unsigned char g_noalloc_scratch[TG_SGEMM_NOALLOC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;

struct NoallocDevice {
    bool ready = false;
    tg_status status = TG_OK;
    int num_sms = 0;
    void* scratch = nullptr;  // device address of g_noalloc_scratch on this device
};

std::mutex g_noalloc_mutex;
NoallocDevice g_noalloc_devices[kMaxDevices];

// One-time set-up of the current device: capability check, kernel
// attributes, and the device address of the scratch array.
tg_status noalloc_device(NoallocDevice** out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return TG_ERR_CUDA;
    if (dev < 0 || dev >= kMaxDevices) return TG_ERR_UNSUPPORTED_DEVICE;
    std::lock_guard<std::mutex> lock(g_noalloc_mutex);
    NoallocDevice& d = g_noalloc_devices[dev];
    if (!d.ready) {
        int major = 0, minor = 0, sms = 0;
        if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
            return TG_ERR_CUDA;
        d.num_sms = sms;
        if (major != 10 || minor != 3) {
            d.status = TG_ERR_UNSUPPORTED_DEVICE;
        } else {
            d.status = prepare_device_kernels();
            if (d.status == TG_OK) {
                void* p = nullptr;
                if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || p == nullptr)
                    d.status = TG_ERR_CUDA;
                else
                    d.scratch = p;
            }
        }
        d.ready = true;
    }
    *out = &d;
    return d.status;
}

}  // namespace
}  // namespace tg

extern "C" tg_status tg_sgemm_noalloc(int M, int N, int K, const float* A, int lda, const float* B,
                                      int ldb, float* C, int ldc, cudaStream_t stream) {
    using namespace tg;
    tg_status st = validate(TG_OP_N, TG_OP_N, M, N, K, A, lda, B, ldb, C, ldc, TG_PATH_TF32X3, 0);
    if (st != TG_OK) return st;
    if (M == 0 || N == 0) return TG_OK;
    NoallocDevice* d = nullptr;
    st = noalloc_device(&d);
    if (st != TG_OK) return st;

    Plan p;
    make_plan(TG_OP_N, TG_OP_N, M, N, K, 1.0f, A, lda, B, ldb, 0.0f, C, ldc, TG_PATH_TF32X3, 0,
              d->num_sms, &p);
    if (p.ws_bytes > TG_SGEMM_NOALLOC_SCRATCH_BYTES && (p.split > 1 || p.tail_lanes > 0))
        // drop the split and stream-K tail partials
        make_plan(TG_OP_N, TG_OP_N, M, N, K, 1.0f, A, lda, B, ldb, 0.0f, C, ldc, TG_PATH_TF32X3, 1,
                  d->num_sms, &p);
    if (p.ws_bytes > TG_SGEMM_NOALLOC_SCRATCH_BYTES) return TG_ERR_WORKSPACE_TOO_SMALL;
    // Nothing in the scratch has to start at zero: the pre-pass writes every
    // hi/lo element it later reads (padding included), and the reduce stores
    // only partial columns the GEMM wrote.  Stale bytes from an earlier call
    // are therefore harmless.
    return launch_plan(p, A, B, C, p.ws_bytes > 0 ? d->scratch : nullptr, stream, nullptr, nullptr);
}
