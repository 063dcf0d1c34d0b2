// Shared device helpers for the libpagedkv kernels (sm_103a).
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp8.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <array>
#include <mutex>
#include <unordered_map>
#include <utility>

#include "pagedkv.h"

namespace pkv {

constexpr int kElemBytes[4] = {4, 2, 1, 1};

inline int elem_bytes(int32_t dt) { return (dt >= 0 && dt <= 3) ? kElemBytes[dt] : 0; }

inline bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

inline pkv_status cuda_status(cudaError_t e) { return e == cudaSuccess ? PKV_OK : PKV_ERR_CUDA; }

// Programmatic dependent launch.  A kernel started by launch_pdl may begin
// while the kernel before it on the stream is still running (its CTAs are
// placed as soon as the earlier kernel's CTAs have all called
// allow_dependents() or exited), so it must call grid_dependency_wait() before
// it reads anything written by earlier work on the stream; the wait returns
// once that work has completed and its writes are visible (at once when the
// kernel was launched without the attribute).  This hides the launch and CTA
// placement of back-to-back kernels (append, decode, split-KV reduce).
__device__ __forceinline__ void grid_dependency_wait() {
  asm volatile("griddepcontrol.wait;\n" ::: "memory");
}
__device__ __forceinline__ void allow_dependents() {
  asm volatile("griddepcontrol.launch_dependents;\n" ::: "memory");
}

template <typename... KArgs, typename... Args>
inline cudaError_t launch_pdl(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem,
                              cudaStream_t stream, Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, std::forward<Args>(args)...);
}

// Number of SMs of the current device, cached per device.
int device_sm_count();

// Opts kernel `kern` into `bytes` of dynamic shared memory on the current
// device.  The attribute belongs to the function in each device's context, so
// the largest value set so far is remembered per (kernel, device).
inline bool opt_in_smem(const void* kern, int bytes) {
  static std::mutex mu;
  static std::unordered_map<const void*, std::array<int, 64>> done;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) {
    cudaGetLastError();
    dev = 0;
  }
  std::lock_guard<std::mutex> lock(mu);
  auto it = done.find(kern);
  if (it == done.end()) it = done.emplace(kern, std::array<int, 64>{}).first;
  int& have = it->second[dev];
  if (bytes <= have) return true;
  if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes) !=
      cudaSuccess)
    return false;
  have = bytes;
  return true;
}

__device__ __forceinline__ void flag_status(int32_t* status, int32_t bit) {
  if (status) atomicOr(status, bit);
}

// ---- element decoding into float (exact for bf16 / f32 / e4m3) ------------
__device__ __forceinline__ float bf16_lo(uint32_t u) { return __uint_as_float(u << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t u) { return __uint_as_float(u & 0xFFFF0000u); }

// Two E4M3 codes (low byte first) to two floats via the f16x2 conversion.
__device__ __forceinline__ float2 e4m3x2_to_float2(uint16_t two) {
  __half2_raw h = __nv_cvt_fp8x2_to_halfraw2(static_cast<__nv_fp8x2_storage_t>(two), __NV_E4M3);
  __half2 hh = *reinterpret_cast<__half2*>(&h);
  return __half22float2(hh);
}

// ---- 16-byte vector of one row segment, decoded to float ------------------
// KV element type tags.
struct F32 {
  static constexpr int kBytes = 4;
  static constexpr int kPerVec = 4;
};
struct BF16 {
  static constexpr int kBytes = 2;
  static constexpr int kPerVec = 8;
};
struct FP8 {
  static constexpr int kBytes = 1;
  static constexpr int kPerVec = 16;
};

struct INT8 {
  static constexpr int kBytes = 1;
  static constexpr int kPerVec = 16;
};

template <typename T>
__device__ __forceinline__ void decode16(const uint4& v, float* x);

template <>
__device__ __forceinline__ void decode16<F32>(const uint4& v, float* x) {
  x[0] = __uint_as_float(v.x);
  x[1] = __uint_as_float(v.y);
  x[2] = __uint_as_float(v.z);
  x[3] = __uint_as_float(v.w);
}

template <>
__device__ __forceinline__ void decode16<BF16>(const uint4& v, float* x) {
  x[0] = bf16_lo(v.x); x[1] = bf16_hi(v.x);
  x[2] = bf16_lo(v.y); x[3] = bf16_hi(v.y);
  x[4] = bf16_lo(v.z); x[5] = bf16_hi(v.z);
  x[6] = bf16_lo(v.w); x[7] = bf16_hi(v.w);
}

template <>
__device__ __forceinline__ void decode16<FP8>(const uint4& v, float* x) {
  const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    float2 a = e4m3x2_to_float2(static_cast<uint16_t>(w[i] & 0xFFFFu));
    float2 b = e4m3x2_to_float2(static_cast<uint16_t>(w[i] >> 16));
    x[4 * i + 0] = a.x; x[4 * i + 1] = a.y;
    x[4 * i + 2] = b.x; x[4 * i + 3] = b.y;
  }
}

template <>
__device__ __forceinline__ void decode16<INT8>(const uint4& v, float* x) {
  const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
#pragma unroll
    for (int b = 0; b < 4; ++b)
      x[4 * i + b] = static_cast<float>(static_cast<int8_t>((w[i] >> (8 * b)) & 0xFFu));
  }
}

}  // namespace pkv
