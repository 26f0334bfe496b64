// Peak probes: how fast this GPU runs the two math instruction mixes of the
// GEMM kernels when nothing else (no loads, no epilogue) is in the way.
//
//  * probe_tf32_mma_kernel: one CTA per SM, one thread issuing
//    tcgen05.mma.cta_group::1.kind::tf32 M=128, N=256, K=8 from operand tiles
//    that stay in shared memory, three per 8-wide K slice and a commit every
//    six -- the issue pattern of the 3xTF32 GEMM's main loop.
//    The same kernel with kind::f16 (M=128, N=256, K=16: the same 32 bytes
//    of each operand row per MMA, twice the products) measures the rate a
//    split into fp16 halves would run at.
//  * probe_ffma_kernel: 16 independent fp32 FMA chains per thread, 2048
//    threads per SM.
//
// The roofline "peak" in the bench stays the one derived from the measured
// copy/bf16 figures; these probes give the ceiling of the instruction mix for
// context.
#include <cuda_runtime.h>

#include <cstdint>

#include "../../include/tg_probes.h"
#include "tg_internal.h"
#include "tg_ptx.cuh"

namespace tg {
namespace {

constexpr int kProbeM = 128, kProbeN = 256, kProbeK = 8;
constexpr uint32_t kProbeA = kProbeM * 16 * 4;  // 128 rows x 64 bytes
constexpr uint32_t kProbeB = kProbeN * 16 * 4;  // 256 rows x 64 bytes
// large enough that one CTA occupies an SM
constexpr size_t kProbeSmem = 160 * 1024;

template <bool kF16>
__global__ void __launch_bounds__(128, 1) probe_mma_kernel(int iters, int use_collector,
                                                         uint64_t timeout_ns) {
    extern __shared__ uint8_t smem_raw[];
    const uint32_t a0 = smem_addr(smem_raw);
    uint8_t* smem = smem_raw + ((1024u - (a0 & 1023u)) & 1023u);
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + kProbeA + kProbeB);
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 2);
    const int warp = threadIdx.x >> 5;
    // operand tiles: zeros written by the threads, then made visible to the
    // tensor core (async proxy)
    for (uint32_t i = threadIdx.x; i < (kProbeA + kProbeB) / 16; i += blockDim.x)
        reinterpret_cast<uint4*>(smem)[i] = make_uint4(0, 0, 0, 0);
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    if (threadIdx.x == 0) {
        mbar_init(&bars[0], 1);
        mbar_init(&bars[1], 1);
        fence_barrier_init();
    }
    if (warp == 0) {
        tmem_alloc(tmem_slot, 256);
        tmem_relinquish();
    }
    tc_fence_before_sync();
    __syncthreads();
    tc_fence_after_sync();
    const uint32_t tmem = *tmem_slot;
    if (threadIdx.x == 0) {
        constexpr uint32_t idesc = kF16 ? idesc_f16(kProbeM, kProbeN) : idesc_tf32(kProbeM, kProbeN);
        const uint32_t sa = smem_addr(smem), sb = sa + kProbeA;
        // the MMA sequence inside the loop has no branch, as in the GEMM's
        // issue loop (a branch between MMAs costs the single issuing thread
        // about 10 % of the rate)
        if (kF16) {
            for (int it = 0; it < iters; ++it) {
#pragma unroll
                for (int ks = 0; ks < 2; ++ks) {
                    const uint64_t da = smem_desc_kmajor(sa + ks * 32, 512, 4);
                    const uint64_t db = smem_desc_kmajor(sb + ks * 32, 512, 4);
                    mma_f16_ss(tmem, da, db, idesc, (it > 0 || ks > 0) ? 1u : 0u);
                    mma_f16_ss(tmem, da, db, idesc, 1u);
                    mma_f16_ss(tmem, da, db, idesc, 1u);
                }
                mma_commit(&bars[0]);
            }
        } else if (use_collector) {
            for (int it = 0; it < iters; ++it) {
#pragma unroll
                for (int ks = 0; ks < 2; ++ks) {
                    const uint64_t da = smem_desc_kmajor(sa + ks * 32, 512, 4);
                    const uint64_t db = smem_desc_kmajor(sb + ks * 32, 512, 4);
                    mma_tf32_ss_fill_a(tmem, da, db, idesc, (it > 0 || ks > 0) ? 1u : 0u);
                    mma_tf32_ss_lastuse_a(tmem, da, db, idesc, 1u);
                    mma_tf32_ss(tmem, da, db, idesc, 1u);
                }
                mma_commit(&bars[0]);  // one commit per six MMAs, like the GEMM's stages
            }
        } else {
            for (int it = 0; it < iters; ++it) {
#pragma unroll
                for (int ks = 0; ks < 2; ++ks) {
                    const uint64_t da = smem_desc_kmajor(sa + ks * 32, 512, 4);
                    const uint64_t db = smem_desc_kmajor(sb + ks * 32, 512, 4);
                    mma_tf32_ss(tmem, da, db, idesc, (it > 0 || ks > 0) ? 1u : 0u);
                    mma_tf32_ss(tmem, da, db, idesc, 1u);
                    mma_tf32_ss(tmem, da, db, idesc, 1u);
                }
                mma_commit(&bars[0]);
            }
        }
        mma_commit(&bars[1]);
        mbar_drain(&bars[1], 0, timeout_ns);
    }
    __syncthreads();
    if (warp == 0) {
        tc_fence_after_sync();
        tmem_dealloc(tmem, 256);
    }
}

__global__ void __launch_bounds__(256) probe_ffma_kernel(int iters, float* sink) {
    float v[16];
#pragma unroll
    for (int j = 0; j < 16; ++j) v[j] = (float)(threadIdx.x + j) * 1e-3f;
    const float b = 0.999f, c = 1e-3f;
    for (int it = 0; it < iters; ++it) {
#pragma unroll
        for (int j = 0; j < 16; ++j) v[j] = fmaf(v[j], b, c);
    }
    float s = 0.0f;
#pragma unroll
    for (int j = 0; j < 16; ++j) s += v[j];
    if (s == -1.0f) *sink = s;  // never true; keeps the chains alive
}

int probe_sms() {
    int dev = 0, sms = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return 0;
    if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
    return sms;
}

bool probe_device_ok() {
    int dev = 0, major = 0, minor = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return false;
    cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev);
    cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev);
    return major == 10 && minor == 3;
}

}  // namespace
}  // namespace tg

extern "C" tg_status tg_probe_tf32_mma(int iters, int use_collector, cudaStream_t stream,
                                       double* tensor_flop) {
    using namespace tg;
    if (iters < 1 || tensor_flop == nullptr) return TG_ERR_INVALID_VALUE;
    if (!probe_device_ok()) return TG_ERR_UNSUPPORTED_DEVICE;
    const int sms = probe_sms();
    if (sms <= 0) return TG_ERR_CUDA;
    if (cudaFuncSetAttribute(probe_mma_kernel<false>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)kProbeSmem) != cudaSuccess)
        return TG_ERR_CUDA;
    probe_mma_kernel<false><<<sms, 128, kProbeSmem, stream>>>(iters, use_collector, 4000000000ull);
    if (cudaGetLastError() != cudaSuccess) return TG_ERR_CUDA;
    *tensor_flop = 2.0 * kProbeM * kProbeN * kProbeK * 6.0 * iters * sms;
    return TG_OK;
}

extern "C" tg_status tg_probe_f16_mma(int iters, cudaStream_t stream, double* tensor_flop) {
    using namespace tg;
    if (iters < 1 || tensor_flop == nullptr) return TG_ERR_INVALID_VALUE;
    if (!probe_device_ok()) return TG_ERR_UNSUPPORTED_DEVICE;
    const int sms = probe_sms();
    if (sms <= 0) return TG_ERR_CUDA;
    if (cudaFuncSetAttribute(probe_mma_kernel<true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)kProbeSmem) != cudaSuccess)
        return TG_ERR_CUDA;
    probe_mma_kernel<true><<<sms, 128, kProbeSmem, stream>>>(iters, 0, 4000000000ull);
    if (cudaGetLastError() != cudaSuccess) return TG_ERR_CUDA;
    *tensor_flop = 2.0 * kProbeM * kProbeN * (2 * kProbeK) * 6.0 * iters * sms;
    return TG_OK;
}

extern "C" tg_status tg_probe_ffma(int iters, float* sink, cudaStream_t stream, double* flop) {
    using namespace tg;
    if (iters < 1 || flop == nullptr || sink == nullptr) return TG_ERR_INVALID_VALUE;
    if (!probe_device_ok()) return TG_ERR_UNSUPPORTED_DEVICE;
    const int sms = probe_sms();
    if (sms <= 0) return TG_ERR_CUDA;
    const int blocks = 8 * sms;
    probe_ffma_kernel<<<blocks, 256, 0, stream>>>(iters, sink);
    if (cudaGetLastError() != cudaSuccess) return TG_ERR_CUDA;
    *flop = 2.0 * 16.0 * iters * 256.0 * blocks;
    return TG_OK;
}
