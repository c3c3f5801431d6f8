// Streaming-read ceiling probe: read a device buffer once with 16-byte
// loads and fold it into one word per CTA.  It measures what a plain,
// well-formed read stream achieves on this device, the figure the aiter
// PR #5190 page compares its kernel with ("streaming-read ceiling").
#include "common.cuh"

namespace mtpattn {
namespace {

constexpr int kThreads = 512;
constexpr int kUnroll = 8;

__device__ __forceinline__ uint4 ld_stream(const uint4* ptr) {
  uint4 v;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];\n"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "l"(ptr));
  return v;
}

__global__ void __launch_bounds__(kThreads)
stream_read_kernel(const uint4* __restrict__ buf, size_t n16, uint32_t* __restrict__ sink) {
  uint32_t acc = 0;
  const size_t stride = static_cast<size_t>(gridDim.x) * kThreads;
  size_t i = static_cast<size_t>(blockIdx.x) * kThreads + threadIdx.x;
  for (; i + (kUnroll - 1) * stride < n16; i += kUnroll * stride) {
    uint4 v[kUnroll];
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) v[u] = ld_stream(buf + i + u * stride);
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) acc ^= v[u].x ^ v[u].y ^ v[u].z ^ v[u].w;
  }
  for (; i < n16; i += stride) {
    const uint4 v = ld_stream(buf + i);
    acc ^= v.x ^ v.y ^ v.z ^ v.w;
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) acc ^= __shfl_xor_sync(0xffffffffu, acc, o);
  __shared__ uint32_t part[kThreads / 32];
  if ((threadIdx.x & 31) == 0) part[threadIdx.x >> 5] = acc;
  __syncthreads();
  if (threadIdx.x == 0) {
    uint32_t a = 0;
    for (int w = 0; w < kThreads / 32; ++w) a ^= part[w];
    sink[blockIdx.x] = a;
  }
}

}  // namespace

cudaError_t launch_stream_read(const void* buf, size_t bytes, uint32_t* sink, int blocks,
                               cudaStream_t stream) {
  stream_read_kernel<<<blocks, kThreads, 0, stream>>>(static_cast<const uint4*>(buf), bytes / 16,
                                                       sink);
  return cudaGetLastError();
}

}  // namespace mtpattn
