// Plain streaming read of a device buffer: the measurement aid behind moe_stream_read. One kernel
// reads [p, p + bytes) once, 16 bytes per load and eight loads in flight per thread, grid-strided
// so that consecutive threads read consecutive 16-byte words (every request a full line), and XORs
// every 32-bit word into one value per block, which the block XORs into *sink (one atomic per
// block, so the result does not depend on the order the blocks finish in).
//
// It computes nothing of the forward. The benchmark times it on the same number of bytes as a
// forward step, in the same way (L2 flushed, CUDA events around the launch), to give the read
// throughput that one kernel of that size reaches on the device: the size-dependent ceiling that
// the step's fraction of the HBM peak is read against.
#include "kernels.cuh"

namespace moe {

namespace {

constexpr int kReadThreads = 512;
constexpr int kReadUnroll = 8;

__device__ __forceinline__ uint32_t xor4(const uint4& v) { return v.x ^ v.y ^ v.z ^ v.w; }

__global__ void __launch_bounds__(kReadThreads) stream_read_kernel(const uint4* __restrict__ p, size_t n,
                                                                   uint32_t* sink) {
    __shared__ uint32_t red[kReadThreads / 32];
    const size_t stride = static_cast<size_t>(gridDim.x) * kReadThreads;
    size_t i = static_cast<size_t>(blockIdx.x) * kReadThreads + threadIdx.x;
    uint32_t acc = 0;
    for (; i + (kReadUnroll - 1) * stride < n; i += kReadUnroll * stride) {
        uint4 v[kReadUnroll];
#pragma unroll
        for (int k = 0; k < kReadUnroll; ++k) v[k] = __ldcs(p + i + k * stride);
#pragma unroll
        for (int k = 0; k < kReadUnroll; ++k) acc ^= xor4(v[k]);
    }
    for (; i < n; i += stride) acc ^= xor4(__ldcs(p + i));
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) acc ^= __shfl_xor_sync(0xffffffffu, acc, o);
    if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = acc;
    __syncthreads();
    if (threadIdx.x == 0) {
        uint32_t b = 0;
#pragma unroll
        for (int w = 0; w < kReadThreads / 32; ++w) b ^= red[w];
        atomicXor(sink, b);
    }
}

}  // namespace

cudaError_t launch_stream_read(const void* p, size_t bytes, uint32_t* sink, int sms, cudaStream_t stream) {
    // two blocks of 512 threads per SM: every SM's 2048 thread slots busy in one wave
    const size_t n = bytes / 16;
    const size_t want = (n + kReadThreads - 1) / kReadThreads;
    const int blocks = static_cast<int>(want < static_cast<size_t>(2 * sms) ? want : static_cast<size_t>(2 * sms));
    stream_read_kernel<<<blocks, kReadThreads, 0, stream>>>(static_cast<const uint4*>(p), n, sink);
    return cudaGetLastError();
}

}  // namespace moe
