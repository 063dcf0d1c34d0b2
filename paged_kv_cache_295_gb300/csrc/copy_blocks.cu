// copy_blocks: the device half of copy-on-write ("LLM inference tutorial"
// section 4.2, the class docstring: copy-on-write for beam search), and
// swap_blocks: the device half of swapping blocks to host memory and back
// ("ToPG framework" section 2.3).  One CTA per (pair, plane) moves one block
// of one plane with 16-byte loads and stores, four in flight per thread.  The
// copy is bound by HBM bandwidth; the swap by the host link (the kernel reads
// or writes page-locked host memory directly).
#include <cuda_runtime.h>

#include <cstdint>

#include "common.cuh"

namespace pkv {
namespace {

constexpr int kCopyThreads = 256;

__global__ void __launch_bounds__(kCopyThreads)
    copy_blocks_kernel(uint8_t* base, int32_t num_planes, int64_t plane_stride,
                       int64_t block_bytes, int64_t num_blocks, const int32_t* pairs,
                       int32_t* status) {
  const int64_t item = blockIdx.x;
  const int32_t k = static_cast<int32_t>(item / num_planes);
  const int32_t plane = static_cast<int32_t>(item % num_planes);
  const int32_t src = __ldg(pairs + 2 * k), dst = __ldg(pairs + 2 * k + 1);
  if (src < 0 || src >= num_blocks || dst < 0 || dst >= num_blocks) {
    if (plane == 0 && threadIdx.x == 0) flag_status(status, PKV_DEV_BAD_BLOCK);
    return;
  }
  if (src == dst) return;
  const uint4* s = reinterpret_cast<const uint4*>(base + plane * plane_stride + src * block_bytes);
  uint4* d = reinterpret_cast<uint4*>(base + plane * plane_stride + dst * block_bytes);
  const int64_t units = block_bytes / 16;
  int64_t u = threadIdx.x;
  for (; u + 3 * kCopyThreads < units; u += 4 * kCopyThreads) {
    const uint4 a = s[u], b = s[u + kCopyThreads], c = s[u + 2 * kCopyThreads],
                e = s[u + 3 * kCopyThreads];
    d[u] = a;
    d[u + kCopyThreads] = b;
    d[u + 2 * kCopyThreads] = c;
    d[u + 3 * kCopyThreads] = e;
  }
  for (; u < units; u += kCopyThreads) d[u] = s[u];
}

// One block of one plane between the pool and a host slot.
__global__ void __launch_bounds__(kCopyThreads)
    swap_blocks_kernel(uint8_t* base, uint8_t* host, int32_t num_planes, int64_t plane_stride,
                       int64_t block_bytes, int64_t num_blocks, int64_t num_host_blocks,
                       const int32_t* pairs, int32_t to_host, int32_t* status) {
  const int64_t item = blockIdx.x;
  const int32_t k = static_cast<int32_t>(item / num_planes);
  const int32_t plane = static_cast<int32_t>(item % num_planes);
  const int32_t a = __ldg(pairs + 2 * k), b = __ldg(pairs + 2 * k + 1);
  const int32_t dev = to_host ? a : b, slot = to_host ? b : a;
  if (dev < 0 || dev >= num_blocks || slot < 0 || slot >= num_host_blocks) {
    if (plane == 0 && threadIdx.x == 0) flag_status(status, PKV_DEV_BAD_BLOCK);
    return;
  }
  uint4* d = reinterpret_cast<uint4*>(base + plane * plane_stride + dev * block_bytes);
  uint4* h = reinterpret_cast<uint4*>(host + (static_cast<int64_t>(slot) * num_planes + plane) *
                                                 block_bytes);
  const uint4* s = to_host ? d : h;
  uint4* t = to_host ? h : d;
  const int64_t units = block_bytes / 16;
  int64_t u = threadIdx.x;
  for (; u + 3 * kCopyThreads < units; u += 4 * kCopyThreads) {
    const uint4 x0 = s[u], x1 = s[u + kCopyThreads], x2 = s[u + 2 * kCopyThreads],
                x3 = s[u + 3 * kCopyThreads];
    t[u] = x0;
    t[u + kCopyThreads] = x1;
    t[u + 2 * kCopyThreads] = x2;
    t[u + 3 * kCopyThreads] = x3;
  }
  for (; u < units; u += kCopyThreads) t[u] = s[u];
}

}  // namespace
}  // namespace pkv

extern "C" pkv_status swap_blocks(void* base, int32_t num_planes, int64_t plane_stride_bytes,
                                  int64_t block_bytes, int64_t num_blocks, void* host,
                                  int64_t num_host_blocks, const int32_t* pairs, int32_t n,
                                  int32_t to_host, int32_t* device_status, pkv_stream_t stream) {
  using namespace pkv;
  if (n < 0 || num_planes <= 0 || block_bytes <= 0 || num_blocks <= 0 || num_host_blocks <= 0 ||
      plane_stride_bytes < num_blocks * block_bytes || (to_host != 0 && to_host != 1))
    return PKV_ERR_INVALID_ARG;
  if (block_bytes % 16 || plane_stride_bytes % 16) return PKV_ERR_INVALID_ARG;
  if (n == 0) return PKV_OK;
  if (!base || !host || !pairs || !aligned16(base) || !aligned16(host) ||
      (reinterpret_cast<uintptr_t>(pairs) & 3u))
    return PKV_ERR_INVALID_ARG;
  void* hdev = nullptr;   // the device's address of the page-locked host area
  if (cudaHostGetDevicePointer(&hdev, host, 0) != cudaSuccess || !hdev) {
    cudaGetLastError();
    return PKV_ERR_INVALID_ARG;
  }
  const int64_t items = static_cast<int64_t>(n) * num_planes;
  if (items > 0x7fffffffLL) return PKV_ERR_UNSUPPORTED;
  swap_blocks_kernel<<<static_cast<unsigned>(items), kCopyThreads, 0,
                       reinterpret_cast<cudaStream_t>(stream)>>>(
      static_cast<uint8_t*>(base), static_cast<uint8_t*>(hdev), num_planes, plane_stride_bytes,
      block_bytes, num_blocks, num_host_blocks, pairs, to_host, device_status);
  return cudaGetLastError() == cudaSuccess ? PKV_OK : PKV_ERR_CUDA;
}

extern "C" pkv_status copy_blocks(void* base, int32_t num_planes, int64_t plane_stride_bytes,
                                  int64_t block_bytes, int64_t num_blocks, const int32_t* pairs,
                                  int32_t n, int32_t* device_status, pkv_stream_t stream) {
  using namespace pkv;
  if (n < 0 || num_planes <= 0 || block_bytes <= 0 || num_blocks <= 0 ||
      plane_stride_bytes < num_blocks * block_bytes)
    return PKV_ERR_INVALID_ARG;
  if (block_bytes % 16 || plane_stride_bytes % 16) return PKV_ERR_INVALID_ARG;
  if (n == 0) return PKV_OK;
  if (!base || !pairs || !aligned16(base) || (reinterpret_cast<uintptr_t>(pairs) & 3u))
    return PKV_ERR_INVALID_ARG;
  const int64_t items = static_cast<int64_t>(n) * num_planes;
  if (items > 0x7fffffffLL) return PKV_ERR_UNSUPPORTED;
  copy_blocks_kernel<<<static_cast<unsigned>(items), kCopyThreads, 0,
                       reinterpret_cast<cudaStream_t>(stream)>>>(
      static_cast<uint8_t*>(base), num_planes, plane_stride_bytes, block_bytes, num_blocks, pairs,
      device_status);
  return cudaGetLastError() == cudaSuccess ? PKV_OK : PKV_ERR_CUDA;
}
