// copy_blocks: the device half of copy-on-write ("LLM inference tutorial"
// section 4.2, the class docstring: copy-on-write for beam search).  One CTA
// per (pair, plane) moves one block of one plane with 16-byte loads and
// stores, four in flight per thread; the copy is bound by HBM bandwidth.
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

}  // namespace
}  // namespace pkv

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
