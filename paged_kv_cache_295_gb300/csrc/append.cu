// reshape_and_cache: write the new tokens' K and V rows into one layer's
// paged cache at their slots ("LLM inference tutorial" section 4.2,
// append_token: physical block slot / block_size, offset slot % block_size).
// The FP8 variant stores E4M3(float(x) / scale[head]) ("ToPG framework"
// section 3.3 compressed FP8 cache; the tutorial's section 3.1 symmetric
// x / scale rule); the INT8 variant stores clamp(round(x / scale[head]),
// -128, 127) with round half to even (the tutorial's section 3.1
// symmetric_quantize with bits = 8), a NaN quotient as 0.
//
// One thread writes one 16-byte segment of one destination row, so a warp
// covers whole rows with coalesced 16-byte stores.  The work is tiny next to
// the attention read, so the kernel is a plain grid-stride loop.
#include "common.cuh"
#include "quant.cuh"

namespace pkv {
namespace {

// Copy kernel: same element type in source and cache.
__global__ void append_copy_kernel(const uint4* __restrict__ k_new, const uint4* __restrict__ v_new,
                                   const int64_t* __restrict__ slots, uint4* __restrict__ k_cache,
                                   uint4* __restrict__ v_cache, int32_t num_tokens,
                                   int32_t num_kv_heads, int32_t segs, int64_t num_slots,
                                   int32_t* status) {
  grid_dependency_wait();   // launched with launch_pdl: earlier work on the stream is done
  allow_dependents();
  const int64_t per_kv = static_cast<int64_t>(num_tokens) * num_kv_heads * segs;
  const int64_t total = 2 * per_kv;
  for (int64_t i = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; i < total;
       i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const bool is_v = i >= per_kv;
    const int64_t j = is_v ? i - per_kv : i;
    const int32_t seg = static_cast<int32_t>(j % segs);
    const int64_t th = j / segs;                       // token * heads + head
    const int32_t head = static_cast<int32_t>(th % num_kv_heads);
    const int64_t tok = th / num_kv_heads;
    const int64_t slot = slots[tok];
    if (slot < 0) continue;
    if (slot >= num_slots) {
      if (!is_v && head == 0 && seg == 0) flag_status(status, PKV_DEV_BAD_SLOT);
      continue;
    }
    const int64_t dst = (slot * num_kv_heads + head) * segs + seg;
    if (is_v)
      v_cache[dst] = __ldg(v_new + j);
    else
      k_cache[dst] = __ldg(k_new + j);
  }
}

// Quantising kernel: f32 / bf16 source -> 8-bit cache (Q = FP8 or INT8), per-head scale.
template <typename Src, typename Q>
__global__ void append_quant_kernel(const Src* __restrict__ k_new, const Src* __restrict__ v_new,
                                  const int64_t* __restrict__ slots, uint4* __restrict__ k_cache,
                                  uint4* __restrict__ v_cache, const float* __restrict__ k_scale,
                                  const float* __restrict__ v_scale, int32_t num_tokens,
                                  int32_t num_kv_heads, int32_t head_dim, int64_t num_slots,
                                  int32_t* status) {
  grid_dependency_wait();   // launched with launch_pdl: earlier work on the stream is done
  allow_dependents();
  const int32_t segs = head_dim / 16;
  const int64_t per_kv = static_cast<int64_t>(num_tokens) * num_kv_heads * segs;
  const int64_t total = 2 * per_kv;
  for (int64_t i = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; i < total;
       i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const bool is_v = i >= per_kv;
    const int64_t j = is_v ? i - per_kv : i;
    const int32_t seg = static_cast<int32_t>(j % segs);
    const int64_t th = j / segs;
    const int32_t head = static_cast<int32_t>(th % num_kv_heads);
    const int64_t tok = th / num_kv_heads;
    const int64_t slot = slots[tok];
    if (slot < 0) continue;
    if (slot >= num_slots) {
      if (!is_v && head == 0 && seg == 0) flag_status(status, PKV_DEV_BAD_SLOT);
      continue;
    }
    const float s = __ldg((is_v ? v_scale : k_scale) + head);
    const int64_t dst = (slot * num_kv_heads + head) * segs + seg;
    (is_v ? v_cache : k_cache)[dst] = quant16<Src, Q>((is_v ? v_new : k_new) + j * 16, s);
  }
}

int grid_for(int64_t work, int threads) {
  const int64_t want = (work + threads - 1) / threads;
  const int64_t cap = static_cast<int64_t>(device_sm_count()) * 16;
  return static_cast<int>(want < cap ? (want > 0 ? want : 1) : cap);
}

}  // namespace
}  // namespace pkv

extern "C" pkv_status reshape_and_cache(const void* k_new, const void* v_new,
                                        const int64_t* slot_mapping, void* k_cache, void* v_cache,
                                        int32_t num_tokens, int32_t num_kv_heads, int32_t head_dim,
                                        int32_t block_size, int64_t num_blocks, int32_t src_dtype,
                                        int32_t cache_dtype, const float* k_scale,
                                        const float* v_scale, int32_t* device_status,
                                        pkv_stream_t stream) {
  using namespace pkv;
  if (num_tokens < 0 || num_kv_heads <= 0 || head_dim <= 0 || block_size <= 0 || num_blocks <= 0)
    return PKV_ERR_INVALID_ARG;
  const int es_src = elem_bytes(src_dtype), es_dst = elem_bytes(cache_dtype);
  if (es_src == 0 || es_dst == 0) return PKV_ERR_UNSUPPORTED;
  if (num_tokens == 0) return PKV_OK;
  if (!k_new || !v_new || !slot_mapping || !k_cache || !v_cache) return PKV_ERR_INVALID_ARG;
  if (!aligned16(k_new) || !aligned16(v_new) || !aligned16(k_cache) || !aligned16(v_cache) ||
      (reinterpret_cast<uintptr_t>(slot_mapping) & 7u))
    return PKV_ERR_INVALID_ARG;
  if ((static_cast<int64_t>(head_dim) * es_dst) % 16 != 0 ||
      (static_cast<int64_t>(head_dim) * es_src) % 16 != 0)
    return PKV_ERR_UNSUPPORTED;
  const int64_t num_slots = num_blocks * block_size;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  constexpr int kThreads = 256;
  const bool quant = cache_dtype == PKV_FP8_E4M3 || cache_dtype == PKV_INT8;
  if (src_dtype == cache_dtype && !quant) {
    const int32_t segs = head_dim * es_dst / 16;
    const int64_t work = 2LL * num_tokens * num_kv_heads * segs;
    if (launch_pdl(append_copy_kernel, dim3(grid_for(work, kThreads)), dim3(kThreads), 0, st,
                   static_cast<const uint4*>(k_new), static_cast<const uint4*>(v_new),
                   slot_mapping, static_cast<uint4*>(k_cache), static_cast<uint4*>(v_cache),
                   num_tokens, num_kv_heads, segs, num_slots, device_status) != cudaSuccess)
      return PKV_ERR_CUDA;
  } else if (quant && (src_dtype == PKV_F32 || src_dtype == PKV_BF16)) {
    if (!k_scale || !v_scale) return PKV_ERR_INVALID_ARG;
    const int64_t work = 2LL * num_tokens * num_kv_heads * (head_dim / 16);
    const int grid = grid_for(work, kThreads);
    auto launch = [&](auto src_tag, auto q_tag) {
      using Src = decltype(src_tag);
      using Q = decltype(q_tag);
      return launch_pdl(append_quant_kernel<Src, Q>, dim3(grid), dim3(kThreads), 0, st,
                        static_cast<const Src*>(k_new), static_cast<const Src*>(v_new),
                        slot_mapping, static_cast<uint4*>(k_cache),
                        static_cast<uint4*>(v_cache), k_scale, v_scale, num_tokens,
                        num_kv_heads, head_dim, num_slots, device_status);
    };
    cudaError_t e;
    if (cache_dtype == PKV_FP8_E4M3)
      e = src_dtype == PKV_F32 ? launch(float{}, FP8{}) : launch(__nv_bfloat16{}, FP8{});
    else
      e = src_dtype == PKV_F32 ? launch(float{}, INT8{}) : launch(__nv_bfloat16{}, INT8{});
    if (e != cudaSuccess) return PKV_ERR_CUDA;
  } else {
    return PKV_ERR_UNSUPPORTED;
  }
  return cuda_status(cudaGetLastError());
}
