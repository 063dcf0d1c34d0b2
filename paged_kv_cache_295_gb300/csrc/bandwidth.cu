// Bandwidth reference kernels: a 16-byte vector device-to-device copy and a
// 16-byte vector read-only reduction.  Timed next to the decode kernel, they
// give the HBM denominators of its roofline on the same device and clocks.
#include "common.cuh"

namespace pkv {
namespace {

constexpr int kBwThreads = 512;
constexpr int kBwBlocksPerSm = 4;
constexpr int kUnroll = 4;

__global__ void __launch_bounds__(kBwThreads) copy16_kernel(const uint4* __restrict__ src,
                                                            uint4* __restrict__ dst, int64_t n) {
  const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
  int64_t i = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x;
  for (; i + (kUnroll - 1) * stride < n; i += kUnroll * stride) {
    uint4 v[kUnroll];
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) v[u] = __ldcs(src + i + u * stride);
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) __stcs(dst + i + u * stride, v[u]);
  }
  for (; i < n; i += stride) __stcs(dst + i, __ldcs(src + i));
}

__global__ void __launch_bounds__(kBwThreads) read16_kernel(const uint4* __restrict__ src,
                                                            int64_t n, float* __restrict__ sink) {
  const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
  int64_t i = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x;
  uint32_t x = 0;
  for (; i + (kUnroll - 1) * stride < n; i += kUnroll * stride) {
    uint4 v[kUnroll];
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) v[u] = __ldcs(src + i + u * stride);
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) x ^= v[u].x ^ v[u].y ^ v[u].z ^ v[u].w;
  }
  for (; i < n; i += stride) {
    const uint4 v = __ldcs(src + i);
    x ^= v.x ^ v.y ^ v.z ^ v.w;
  }
  // Keep the loads live: fold the warp's words and let lane 0 of warp 0 write.
  for (int off = 16; off > 0; off >>= 1) x ^= __shfl_xor_sync(0xffffffffu, x, off);
  if (threadIdx.x == 0) sink[blockIdx.x] = __uint_as_float(x & 0x007FFFFFu);
}

int bw_grid() { return device_sm_count() * kBwBlocksPerSm; }

}  // namespace
}  // namespace pkv

extern "C" int32_t pkv_read_kernel_sink_floats(void) { return pkv::bw_grid(); }

extern "C" pkv_status pkv_copy_kernel(const void* src, void* dst, size_t bytes,
                                      pkv_stream_t stream) {
  using namespace pkv;
  if (bytes == 0) return PKV_OK;
  if (!src || !dst || bytes % 16 || !aligned16(src) || !aligned16(dst)) return PKV_ERR_INVALID_ARG;
  copy16_kernel<<<bw_grid(), kBwThreads, 0, reinterpret_cast<cudaStream_t>(stream)>>>(
      static_cast<const uint4*>(src), static_cast<uint4*>(dst), static_cast<int64_t>(bytes / 16));
  return cuda_status(cudaGetLastError());
}

extern "C" pkv_status pkv_read_kernel(const void* src, size_t bytes, float* sink,
                                      pkv_stream_t stream) {
  using namespace pkv;
  if (bytes == 0) return PKV_OK;
  if (!src || !sink || bytes % 16 || !aligned16(src)) return PKV_ERR_INVALID_ARG;
  read16_kernel<<<bw_grid(), kBwThreads, 0, reinterpret_cast<cudaStream_t>(stream)>>>(
      static_cast<const uint4*>(src), static_cast<int64_t>(bytes / 16), sink);
  return cuda_status(cudaGetLastError());
}
