// Widening loads and 8-bit quantisation of new K/V rows, shared by the append
// kernel (reshape_and_cache) and the decode kernel's fused append, so both
// store the same bytes.  FP8: E4M3 of the IEEE float32 quotient x / scale,
// round to nearest even, saturating ("ToPG framework" section 3.3); INT8:
// clamp(round_half_even(x / scale), -128, 127) with NaN -> 0 ("LLM inference
// tutorial" section 3.1 symmetric quantisation, 8 bits).
#pragma once

#include "common.cuh"

namespace pkv {

template <typename Src>
__device__ __forceinline__ void load16(const Src* p, float* x);

template <>
__device__ __forceinline__ void load16<float>(const float* p, float* x) {
  const float4* v = reinterpret_cast<const float4*>(p);
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const float4 f = __ldg(v + i);
    x[4 * i + 0] = f.x; x[4 * i + 1] = f.y; x[4 * i + 2] = f.z; x[4 * i + 3] = f.w;
  }
}

template <>
__device__ __forceinline__ void load16<__nv_bfloat16>(const __nv_bfloat16* p, float* x) {
  const uint4* v = reinterpret_cast<const uint4*>(p);
#pragma unroll
  for (int i = 0; i < 2; ++i) {
    float y[8];
    decode16<BF16>(__ldg(v + i), y);
#pragma unroll
    for (int k = 0; k < 8; ++k) x[8 * i + k] = y[k];
  }
}

// Four float32 quotients -> four cache bytes (low byte first).
template <typename Q>
__device__ __forceinline__ uint32_t quant4(const float* q);

template <>
__device__ __forceinline__ uint32_t quant4<FP8>(const float* q) {   // E4M3, RNE, saturating
  const uint32_t lo = __nv_cvt_float2_to_fp8x2(make_float2(q[0], q[1]), __NV_SATFINITE, __NV_E4M3);
  const uint32_t hi = __nv_cvt_float2_to_fp8x2(make_float2(q[2], q[3]), __NV_SATFINITE, __NV_E4M3);
  return (lo & 0xFFFFu) | (hi << 16);
}

template <>
__device__ __forceinline__ uint32_t quant4<INT8>(const float* q) {   // RNE, clamp, NaN -> 0
  uint32_t w = 0;
#pragma unroll
  for (int b = 0; b < 4; ++b) {
    int v = __float2int_rn(q[b]);   // round half to even; NaN -> 0, +-inf saturate
    v = v < -128 ? -128 : (v > 127 ? 127 : v);
    w |= (static_cast<uint32_t>(v) & 0xFFu) << (8 * b);
  }
  return w;
}

// 16 source elements -> 16 cache bytes: each divided by `scale` (IEEE
// float32 division), then the 8-bit code.
template <typename Src, typename Q>
__device__ __forceinline__ uint4 quant16(const Src* src, float scale) {
  float x[16];
  load16<Src>(src, x);
  uint32_t w[4];
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    float q[4];
#pragma unroll
    for (int e = 0; e < 4; ++e) q[e] = __fdiv_rn(x[4 * k + e], scale);
    w[k] = quant4<Q>(q);
  }
  return make_uint4(w[0], w[1], w[2], w[3]);
}

}  // namespace pkv
