// paged_attention_prefill: argument checks, tensor maps and the launch of the
// tcgen05 prefill kernel.
#include <cmath>

#include "prefill_tc.cuh"
#include "tmap.cuh"

namespace pkv {
namespace {

bool pow2(int x) { return x > 0 && (x & (x - 1)) == 0; }
int ilog2(int x) {
  int l = 0;
  while ((1 << l) < x) ++l;
  return l;
}

}  // namespace
}  // namespace pkv

extern "C" pkv_status paged_attention_prefill(
    const void* q, const int32_t* query_start, const void* k_cache, const void* v_cache,
    const int32_t* block_tables, const int32_t* context_lens, int32_t num_seqs,
    int32_t num_tokens, int32_t max_query_len, int32_t num_q_heads, int32_t num_kv_heads,
    int32_t head_dim, int32_t block_size, int64_t num_blocks, int32_t max_blocks_per_seq,
    int32_t max_context_len, float scale, int32_t causal, int32_t q_dtype, int32_t kv_dtype,
    const float* k_scale, const float* v_scale, float* out, int32_t* device_status,
    pkv_stream_t stream) {
  using namespace pkv;
  if (num_seqs < 0 || num_tokens < 0 || max_query_len < 0 || num_q_heads <= 0 ||
      num_kv_heads <= 0 || num_blocks <= 0 || max_blocks_per_seq <= 0 || max_context_len < 0)
    return PKV_ERR_INVALID_ARG;
  if (num_q_heads % num_kv_heads != 0) return PKV_ERR_INVALID_ARG;
  if (causal != 0 && causal != 1) return PKV_ERR_INVALID_ARG;
  if (!std::isfinite(scale)) return PKV_ERR_INVALID_ARG;
  const int G = num_q_heads / num_kv_heads;
  const bool fp8 = kv_dtype == PKV_FP8_E4M3, i8 = kv_dtype == PKV_INT8;
  const bool codes8 = fp8 || i8;   // 8-bit caches: widened to fp16 in the kernel
  if (head_dim != kPfD || q_dtype != PKV_BF16 || (kv_dtype != PKV_BF16 && !codes8) || G > 16)
    return PKV_ERR_UNSUPPORTED;
  if (!pow2(block_size) || block_size < 8 || block_size > 4096) return PKV_ERR_UNSUPPORTED;
  if (num_blocks * block_size > 0x7fffffffLL) return PKV_ERR_UNSUPPORTED;
  if (static_cast<int64_t>(max_blocks_per_seq) * block_size > 0x7fffffffLL)
    return PKV_ERR_INVALID_ARG;
  if (static_cast<int64_t>(max_context_len) > static_cast<int64_t>(max_blocks_per_seq) * block_size)
    return PKV_ERR_INVALID_ARG;
  if (max_query_len > num_tokens) return PKV_ERR_INVALID_ARG;
  if (num_seqs == 0 || max_query_len == 0) return PKV_OK;
  if (!q || !query_start || !k_cache || !v_cache || !block_tables || !context_lens || !out)
    return PKV_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(k_cache) || !aligned16(v_cache) || !aligned16(out) ||
      (reinterpret_cast<uintptr_t>(query_start) & 3u) ||
      (reinterpret_cast<uintptr_t>(block_tables) & 3u) ||
      (reinterpret_cast<uintptr_t>(context_lens) & 3u))
    return PKV_ERR_INVALID_ARG;
  if (codes8 && (!k_scale || !v_scale)) return PKV_ERR_INVALID_ARG;
  if (num_seqs > 65535 || num_kv_heads > 65535) return PKV_ERR_UNSUPPORTED;
  if (!encode_fn()) return PKV_ERR_CUDA;

  PrefillParams p{};
  p.q = static_cast<const __nv_bfloat16*>(q);
  p.query_start = query_start;
  p.block_tables = block_tables;
  p.context_lens = context_lens;
  p.out = out;
  p.status = device_status;
  p.num_blocks = num_blocks;
  p.num_q_heads = num_q_heads;
  p.num_kv_heads = num_kv_heads;
  p.max_blocks_per_seq = max_blocks_per_seq;
  p.bs_log2 = ilog2(block_size);
  p.box_rows = block_size < kPfKeys ? block_size : kPfKeys;
  p.tile_tokens = kPfRows / G;
  p.causal = causal;
  p.max_context_len = max_context_len;
  p.num_tokens = num_tokens;
  p.qk_scale_log2 = scale * 1.4426950408889634f;
  p.k_scale = codes8 ? k_scale : nullptr;
  p.v_scale = codes8 ? v_scale : nullptr;

  CUtensorMap tk, tv;
  const int64_t rows = num_blocks * block_size;
  if (!make_map(&tk, k_cache, kPfD, num_kv_heads, rows, p.box_rows, codes8) ||
      !make_map(&tv, v_cache, kPfD, num_kv_heads, rows, p.box_rows, codes8))
    return PKV_ERR_CUDA;

  const int pairs = (max_query_len + 2 * p.tile_tokens - 1) / (2 * p.tile_tokens);
  dim3 grid(pairs, num_kv_heads, num_seqs);
  auto launch = [&](auto kern, size_t smem) {
    if (!opt_in_smem(reinterpret_cast<const void*>(kern), static_cast<int>(smem)))
      return PKV_ERR_CUDA;
    kern<<<grid, kPfThreads, smem, reinterpret_cast<cudaStream_t>(stream)>>>(tk, tv, p);
    return cudaGetLastError() == cudaSuccess ? PKV_OK : PKV_ERR_CUDA;
  };
  if (fp8)
    return launch(paged_prefill_tc_kernel<kPfStagesFp8, 1>, PfLayout::bytes(kPfStagesFp8, true));
  if (i8)
    return launch(paged_prefill_tc_kernel<kPfStagesFp8, 2>, PfLayout::bytes(kPfStagesFp8, true));
  return launch(paged_prefill_tc_kernel<kPfStages, 0>, PfLayout::bytes(kPfStages, false));
}
