// Tiled matrix transpose, four variants (include/tg_transpose.h).
//
// Memory-bound: every element is read once and written once (8 bytes per
// element against the copy-bandwidth roofline).  A 128-thread block (32 x 4)
// moves 32 x 32 tiles, 8 elements per thread, in a grid-stride loop over
// tiles with one full wave of resident blocks; each thread issues its 8 loads
// before its 8 stores, which keeps enough bytes in flight to cover HBM
// latency.  The shared tile layouts are the pages' three: plain
// [32][32] (column read = 32-way bank conflict), padded [32][33]
// (gcd(33, 32) = 1: conflict-free) and XOR-swizzled (column c of row r at
// c ^ r: conflict-free for rows and columns).  The direct variant skips
// shared memory: coalesced reads, and writes whose 32 lanes land in 32
// different rows of the output (the "stride >= 32 bytes" case of "Global
// Memory와 Coalescing": one sector per lane).
#include <cuda_runtime.h>

#include <cstdint>
#include <mutex>

#include "../../include/tg_transpose.h"
#include "tg_internal.h"

namespace tg {
namespace {

constexpr int kT = 32;        // tile edge
constexpr int kRowsPer = 4;   // thread rows: 32 x 4 threads, 8 elements each
constexpr int kPer = kT / kRowsPer;
constexpr int kThreads = 32 * kRowsPer;

template <int V>
__device__ __forceinline__ int tile_index(int r, int c) {
    if (V == TG_TRANSPOSE_PADDED) return r * (kT + 1) + c;
    if (V == TG_TRANSPOSE_SWIZZLED) return r * kT + (c ^ r);
    return r * kT + c;
}

template <int V>
__global__ void __launch_bounds__(kThreads) transpose_kernel(const float* __restrict__ in, long long ld_in,
                                                        float* __restrict__ out, long long ld_out,
                                                        int rows, int cols) {
    __shared__ float tile[kT * (kT + 1)];
    const int tx = threadIdx.x & 31, ty = threadIdx.x >> 5;
    const int tiles_c = (cols + kT - 1) / kT;
    const long long tiles = (long long)((rows + kT - 1) / kT) * tiles_c;
    for (long long t = blockIdx.x; t < tiles; t += gridDim.x) {
        const int r0 = (int)(t / tiles_c) * kT, c0 = (int)(t % tiles_c) * kT;
        if (V == TG_TRANSPOSE_DIRECT) {
            float v[kPer];
#pragma unroll
            for (int j = 0; j < kPer; ++j) {
                const int r = r0 + ty + kRowsPer * j, c = c0 + tx;
                v[j] = (r < rows && c < cols) ? in[(long long)r * ld_in + c] : 0.0f;
            }
#pragma unroll
            for (int j = 0; j < kPer; ++j) {
                const int r = r0 + ty + kRowsPer * j, c = c0 + tx;
                if (r < rows && c < cols) out[(long long)c * ld_out + r] = v[j];
            }
            continue;
        }
        float v[kPer];
#pragma unroll
        for (int j = 0; j < kPer; ++j) {  // read rows of the input tile (coalesced)
            const int r = r0 + ty + kRowsPer * j, c = c0 + tx;
            v[j] = (r < rows && c < cols) ? in[(long long)r * ld_in + c] : 0.0f;
        }
#pragma unroll
        for (int j = 0; j < kPer; ++j) tile[tile_index<V>(ty + kRowsPer * j, tx)] = v[j];
        __syncthreads();
#pragma unroll
        for (int j = 0; j < kPer; ++j) {  // write rows of the output = columns of the tile
            const int c = c0 + ty + kRowsPer * j, r = r0 + tx;
            v[j] = tile[tile_index<V>(tx, ty + kRowsPer * j)];
            if (r < rows && c < cols) out[(long long)c * ld_out + r] = v[j];
        }
        __syncthreads();
    }
}

int g_transpose_blocks_per_sm[4] = {0, 0, 0, 0};
std::mutex g_transpose_mutex;

template <int V>
tg_status launch(int rows, int cols, const float* in, long long ld_in, float* out, long long ld_out,
                 cudaStream_t stream) {
    int dev = 0, sms = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return TG_ERR_CUDA;
    if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return TG_ERR_CUDA;
    int per_sm;
    {
        std::lock_guard<std::mutex> lock(g_transpose_mutex);
        if (g_transpose_blocks_per_sm[V] == 0) {
            int nb = 0;
            if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&nb, transpose_kernel<V>, kThreads, 0) != cudaSuccess ||
                nb <= 0)
                nb = 4;
            g_transpose_blocks_per_sm[V] = nb;
        }
        per_sm = g_transpose_blocks_per_sm[V];
    }
    const long long tiles = (long long)((rows + kT - 1) / kT) * ((cols + kT - 1) / kT);
    long long grid = (long long)per_sm * sms;
    if (grid > tiles) grid = tiles;
    transpose_kernel<V><<<(int)grid, kThreads, 0, stream>>>(in, ld_in, out, ld_out, rows, cols);
    return cudaGetLastError() == cudaSuccess ? TG_OK : TG_ERR_CUDA;
}

}  // namespace
}  // namespace tg

extern "C" tg_status tg_transpose(int variant, int rows, int cols, const float* in, int ld_in, float* out,
                                  int ld_out, cudaStream_t stream) {
    using namespace tg;
    if (variant < TG_TRANSPOSE_DIRECT || variant > TG_TRANSPOSE_SWIZZLED) return TG_ERR_INVALID_VALUE;
    if (rows < 0 || cols < 0) return TG_ERR_INVALID_VALUE;
    if (ld_in < (cols > 1 ? cols : 1) || ld_out < (rows > 1 ? rows : 1)) return TG_ERR_INVALID_VALUE;
    if (rows == 0 || cols == 0) return TG_OK;
    if (in == nullptr || out == nullptr) return TG_ERR_INVALID_VALUE;
    const uintptr_t i0 = reinterpret_cast<uintptr_t>(in);
    const uintptr_t i1 = i0 + 4ull * ((unsigned long long)(rows - 1) * ld_in + cols);
    const uintptr_t o0 = reinterpret_cast<uintptr_t>(out);
    const uintptr_t o1 = o0 + 4ull * ((unsigned long long)(cols - 1) * ld_out + rows);
    if (i0 < o1 && o0 < i1) return TG_ERR_INVALID_VALUE;
    int dev = 0, major = 0, minor = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return TG_ERR_CUDA;
    cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev);
    cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev);
    if (major != 10 || minor != 3) return TG_ERR_UNSUPPORTED_DEVICE;
    switch (variant) {
        case TG_TRANSPOSE_DIRECT: return launch<TG_TRANSPOSE_DIRECT>(rows, cols, in, ld_in, out, ld_out, stream);
        case TG_TRANSPOSE_TILE32: return launch<TG_TRANSPOSE_TILE32>(rows, cols, in, ld_in, out, ld_out, stream);
        case TG_TRANSPOSE_PADDED: return launch<TG_TRANSPOSE_PADDED>(rows, cols, in, ld_in, out, ld_out, stream);
        default: return launch<TG_TRANSPOSE_SWIZZLED>(rows, cols, in, ld_in, out, ld_out, stream);
    }
}
