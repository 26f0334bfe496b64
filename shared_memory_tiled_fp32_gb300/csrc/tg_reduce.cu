// Sum reduction, five variants (include/tg_reduce.h).
//
// The four versions of the pages run as the pages lay them out: a block of
// 256 threads loads 256 consecutive values (one each) into shared memory and
// folds them; the block partials are folded again by the same kernel until
// one value is left.  Memory-bound (one add per 4-byte value), so the GB300
// form reads float4s in a grid-stride loop over one wave of resident blocks
// (four independent float4 accumulators per thread keep 64 bytes per thread
// in flight), folds each warp with shuffles and each block through one
// shared value per warp, and a single block folds the block partials in a
// fixed order.
#include <cuda_runtime.h>

#include <cstdint>

#include "../../include/tg_reduce.h"
#include "tg_internal.h"

namespace tg {
namespace {

constexpr int kRB = 256;           // threads (and values) per block of the pages' versions
constexpr int kFastBlocksPerSm = 4;  // TG_REDUCE_FAST: 4 x 256 threads per SM

template <int V>
__global__ void __launch_bounds__(kRB) block_fold_kernel(const float* __restrict__ in, long long n,
                                                         float* __restrict__ out) {
    __shared__ float buf[kRB];
    const int tid = threadIdx.x;
    const long long i = (long long)blockIdx.x * kRB + tid;
    buf[tid] = i < n ? in[i] : 0.0f;
    __syncthreads();
    if (V == TG_REDUCE_INTERLEAVED) {
        for (int s = 1; s < kRB; s *= 2) {
            if (tid % (2 * s) == 0) buf[tid] += buf[tid + s];
            __syncthreads();
        }
        if (tid == 0) out[blockIdx.x] = buf[0];
    } else if (V == TG_REDUCE_SEQUENTIAL) {
        for (int s = kRB / 2; s > 0; s >>= 1) {
            if (tid < s) buf[tid] += buf[tid + s];
            __syncthreads();
        }
        if (tid == 0) out[blockIdx.x] = buf[0];
    } else {  // SHUFFLE and ATOMIC
        for (int s = kRB / 2; s > 32; s >>= 1) {
            if (tid < s) buf[tid] += buf[tid + s];
            __syncthreads();
        }
        if (tid < 32) {
            float x = buf[tid] + buf[tid + 32];
            for (int off = 16; off > 0; off >>= 1) x += __shfl_down_sync(0xffffffffu, x, off);
            if (tid == 0) {
                if (V == TG_REDUCE_ATOMIC)
                    atomicAdd(out, x);
                else
                    out[blockIdx.x] = x;
            }
        }
    }
}

__global__ void set_zero_kernel(float* p) { *p = 0.0f; }

__device__ __forceinline__ float warp_fold(float x) {
    for (int off = 16; off > 0; off >>= 1) x += __shfl_down_sync(0xffffffffu, x, off);
    return x;
}

// Block sum of one value per thread, in a fixed order; valid in thread 0.
__device__ __forceinline__ float block_fold(float x, float* warp_sums) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    x = warp_fold(x);
    if (lane == 0) warp_sums[warp] = x;
    __syncthreads();
    float s = 0.0f;
    if (warp == 0) {
        s = lane < (int)(blockDim.x >> 5) ? warp_sums[lane] : 0.0f;
        s = warp_fold(s);
    }
    return s;
}

__global__ void __launch_bounds__(kRB) fast_partial_kernel(const float* __restrict__ x, long long n,
                                                           float* __restrict__ partials) {
    __shared__ float warp_sums[kRB / 32];
    // the float4 body starts at the first 16-byte boundary; the few values
    // before it and after the last whole float4 are added by thread 0 of block 0
    const long long head = (long long)((16u - (reinterpret_cast<uintptr_t>(x) & 15u)) & 15u) / 4;
    const long long h = head < n ? head : n;
    const long long n4 = (n - h) / 4;
    const float4* x4 = reinterpret_cast<const float4*>(x + h);
    const long long stride = (long long)gridDim.x * blockDim.x;
    float4 a0 = make_float4(0.f, 0.f, 0.f, 0.f), a1 = a0, a2 = a0, a3 = a0;
    long long i = blockIdx.x * (long long)blockDim.x + threadIdx.x;
    for (; i + 3 * stride < n4; i += 4 * stride) {
        const float4 v0 = x4[i], v1 = x4[i + stride], v2 = x4[i + 2 * stride], v3 = x4[i + 3 * stride];
        a0.x += v0.x; a0.y += v0.y; a0.z += v0.z; a0.w += v0.w;
        a1.x += v1.x; a1.y += v1.y; a1.z += v1.z; a1.w += v1.w;
        a2.x += v2.x; a2.y += v2.y; a2.z += v2.z; a2.w += v2.w;
        a3.x += v3.x; a3.y += v3.y; a3.z += v3.z; a3.w += v3.w;
    }
    for (; i < n4; i += stride) {
        const float4 v = x4[i];
        a0.x += v.x; a0.y += v.y; a0.z += v.z; a0.w += v.w;
    }
    float t = ((a0.x + a0.y) + (a0.z + a0.w)) + ((a1.x + a1.y) + (a1.z + a1.w)) +
              (((a2.x + a2.y) + (a2.z + a2.w)) + ((a3.x + a3.y) + (a3.z + a3.w)));
    if (blockIdx.x == 0 && threadIdx.x == 0) {
        for (long long j = 0; j < h; ++j) t += x[j];
        for (long long j = h + 4 * n4; j < n; ++j) t += x[j];
    }
    const float s = block_fold(t, warp_sums);
    if (threadIdx.x == 0) partials[blockIdx.x] = s;
}

__global__ void __launch_bounds__(kRB) fast_final_kernel(const float* __restrict__ partials, int count,
                                                         float* __restrict__ result) {
    __shared__ float warp_sums[kRB / 32];
    float t = 0.0f;
    for (int j = threadIdx.x; j < count; j += blockDim.x) t += partials[j];
    const float s = block_fold(t, warp_sums);
    if (threadIdx.x == 0) *result = s;
}

int plan_passes(int variant, long long n, int num_sms, long long* counts, size_t* ws) {
    int p = 0;
    size_t bytes = 0;
    if (variant == TG_REDUCE_FAST) {
        const long long grid = (long long)kFastBlocksPerSm * num_sms;
        counts[p++] = grid;
        counts[p++] = 1;
        bytes = 4ull * grid;
    } else if (variant == TG_REDUCE_ATOMIC) {
        counts[p++] = 1;  // the result, zeroed
        counts[p++] = 1;  // every block adds into it
    } else {
        long long m = n;
        do {
            m = (m + kRB - 1) / kRB;
            counts[p++] = m;
            if (m > 1) bytes += 4ull * m;
        } while (m > 1 && p < 8);
    }
    *ws = bytes;
    return p;
}

template <int V>
tg_status fold_passes(long long n, const float* x, float* result, float* ws, cudaStream_t stream) {
    const float* src = x;
    long long m = n;
    float* dst = ws;
    while (true) {
        const long long blocks = (m + kRB - 1) / kRB;
        float* out = blocks == 1 ? result : dst;
        block_fold_kernel<V><<<(unsigned)blocks, kRB, 0, stream>>>(src, m, out);
        if (cudaGetLastError() != cudaSuccess) return TG_ERR_CUDA;
        if (blocks == 1) return TG_OK;
        src = dst;
        dst += blocks;
        m = blocks;
    }
}

}  // namespace
}  // namespace tg

extern "C" tg_status tg_reduce_plan(int variant, long long n, int num_sms, int* passes, long long* counts,
                                    size_t* workspace_bytes) {
    using namespace tg;
    if (variant < TG_REDUCE_INTERLEAVED || variant > TG_REDUCE_FAST || n < 0 || passes == nullptr ||
        counts == nullptr || workspace_bytes == nullptr)
        return TG_ERR_INVALID_VALUE;
    if (num_sms <= 0) {
        int dev = 0;
        if (cudaGetDevice(&dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&num_sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
            return TG_ERR_CUDA;
    }
    *passes = plan_passes(variant, n, num_sms, counts, workspace_bytes);
    return TG_OK;
}

extern "C" tg_status tg_reduce_sum(int variant, long long n, const float* x, float* result, cudaStream_t stream) {
    using namespace tg;
    if (variant < TG_REDUCE_INTERLEAVED || variant > TG_REDUCE_FAST || n < 0 || result == nullptr)
        return TG_ERR_INVALID_VALUE;
    if (n > 0 && x == nullptr) return TG_ERR_INVALID_VALUE;
    int dev = 0, major = 0, minor = 0, sms = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return TG_ERR_CUDA;
    cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev);
    cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (major != 10 || minor != 3) return TG_ERR_UNSUPPORTED_DEVICE;
    if (n == 0) {
        set_zero_kernel<<<1, 1, 0, stream>>>(result);
        return cudaGetLastError() == cudaSuccess ? TG_OK : TG_ERR_CUDA;
    }
    long long counts[8];
    size_t bytes = 0;
    plan_passes(variant, n, sms, counts, &bytes);
    void* ws = nullptr;
    if (bytes > 0) {
        tg_status st = workspace_alloc(bytes, stream, &ws);
        if (st != TG_OK) return st;
    }
    float* w = static_cast<float*>(ws);
    tg_status st = TG_OK;
    switch (variant) {
        case TG_REDUCE_INTERLEAVED: st = fold_passes<TG_REDUCE_INTERLEAVED>(n, x, result, w, stream); break;
        case TG_REDUCE_SEQUENTIAL: st = fold_passes<TG_REDUCE_SEQUENTIAL>(n, x, result, w, stream); break;
        case TG_REDUCE_SHUFFLE: st = fold_passes<TG_REDUCE_SHUFFLE>(n, x, result, w, stream); break;
        case TG_REDUCE_ATOMIC: {
            set_zero_kernel<<<1, 1, 0, stream>>>(result);
            const long long blocks = (n + kRB - 1) / kRB;
            block_fold_kernel<TG_REDUCE_ATOMIC><<<(unsigned)blocks, kRB, 0, stream>>>(x, n, result);
            st = cudaGetLastError() == cudaSuccess ? TG_OK : TG_ERR_CUDA;
            break;
        }
        default: {
            const int grid = (int)counts[0];
            fast_partial_kernel<<<grid, kRB, 0, stream>>>(x, n, w);
            fast_final_kernel<<<1, kRB, 0, stream>>>(w, grid, result);
            st = cudaGetLastError() == cudaSuccess ? TG_OK : TG_ERR_CUDA;
        }
    }
    if (ws != nullptr) workspace_free(ws, stream);
    return st;
}
