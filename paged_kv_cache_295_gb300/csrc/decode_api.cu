// Host entry points of the decode path: argument validation, split-KV
// partition choice, workspace layout and dispatch to the kernel instantiation
// for (KV type, head_dim, query-group size).
#include <atomic>
#include <cmath>

#include "decode_kernel.cuh"

namespace pkv {

int device_sm_count() {
  static int cached[64] = {0};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) {
    cudaGetLastError();
    return 152;   // GB300 has 152 SMs; used only when no device answers
  }
  if (cached[dev] == 0) {
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) {
      cudaGetLastError();
      n = 152;
    }
    cached[dev] = n;
  }
  return cached[dev];
}

namespace {

bool is_pow2(int64_t x) { return x > 0 && (x & (x - 1)) == 0; }

// Kernel choice.  By shape: the transposed mma.sync kernel (decode_mma2.cuh)
// for groups of up to 8 heads, the heads-as-rows mma.sync kernel
// (decode_mma.cuh) for groups of up to 16, else the CUDA-core kernel - the
// fastest measured order.  pkv_test_force_decode_kernel lets tests and
// profiles run the other kernels on the same inputs; the hot path reads that
// setting with one relaxed atomic load.
std::atomic<int32_t> g_forced_kernel{PKV_DECODE_KERNEL_AUTO};
int32_t forced_kernel() { return g_forced_kernel.load(std::memory_order_relaxed); }
// Bytes a test makes the next transposed-kernel launches wait for in vain
// (pkv_test_decode_stall); 0 otherwise.
std::atomic<uint32_t> g_stall_bytes{0};

int log2i(int64_t x) {
  int r = 0;
  while ((int64_t{1} << r) < x) ++r;
  return r;
}

// Split-KV partition length.  Aim for about 16 work items (CTAs that have
// tokens) per SM over the longest sequence, so the grid runs many waves and
// a ragged tail costs little; keep partitions between 256 and 4096 tokens so
// per-CTA set-up and the partial round trip stay a small share of the bytes.
// A partition writes G * (D + 2) floats of partials (and the reduce reads them
// back) per 2 * P * D cache elements it reads, so the partials' share of the
// traffic grows with the group size G: P is at least 256 * G, which keeps it
// near 0.4 % (GQA-8 on the 70B-shaped layer: 2048 instead of 1024, 2 % faster).
int32_t auto_partition(int32_t num_seqs, int32_t num_q_heads, int32_t num_kv_heads,
                       int32_t max_ctx) {
  const double work = static_cast<double>(num_seqs) * num_kv_heads * (max_ctx > 0 ? max_ctx : 1);
  const double items = 16.0 * device_sm_count();
  int64_t want = static_cast<int64_t>(work / items);
  const int64_t floor_g = 256LL * (num_q_heads / num_kv_heads);
  if (want < floor_g) want = floor_g;
  int64_t P = 256;
  while (P * 2 <= want && P < 4096) P *= 2;
  const int64_t slots = 3LL * device_sm_count();
  const int64_t ctx = max_ctx > 0 ? max_ctx : 1;
  const int64_t heads = static_cast<int64_t>(num_seqs) * num_kv_heads;
  // Long contexts: past 32 partitions per sequence the grid has CTAs to
  // spare, and fewer, longer partitions spend less on each CTA's start-up,
  // epilogue and partials.  P doubles (up to 4096) while a sequence still
  // has more than 32 partitions and the doubled grid keeps two waves of CTA
  // slots.  Measured on 8 sequences of 128K tokens, 8 KV heads (GQA-4):
  // 386.6 us per layer at 4096 against 391.8 at 2048; the 7B- and 70B-shaped
  // layers (2 to 8 partitions) keep 1024 and 2048, their best.
  while (P < 4096 && (ctx + P - 1) / P > 32 && heads * ((ctx + 2 * P - 1) / (2 * P)) >= 2 * slots)
    P *= 2;
  // Small batches: the rule above bottoms out at 256, but when the grid is
  // only a wave or two, each CTA's fixed start-up and epilogue dominate and
  // fewer, longer partitions finish sooner.  Up to 1024 tokens, P doubles
  // while the grid still fills one wave of CTA slots (three per SM).  Measured
  // in CUDA graphs on 32 heads, contexts U[256, 1024]: batch 8 runs 512
  // (19.0 us per layer against 21.0 at 256), batch 32 runs 1024 (63.7 against
  // 67.5), batch 2 keeps 256 (12.0 against 15.2 at 512).
  while (P < 1024 &&
         static_cast<int64_t>(num_seqs) * num_kv_heads * ((ctx + 2 * P - 1) / (2 * P)) >= slots)
    P *= 2;
  return static_cast<int32_t>(P);
}

int32_t resolve_partition(int32_t num_seqs, int32_t num_q_heads, int32_t num_kv_heads,
                          int32_t max_ctx, int32_t req) {
  if (req < 0 || (req > 0 && req % 64 != 0)) return 0;
  return req > 0 ? req : auto_partition(num_seqs, num_q_heads, num_kv_heads, max_ctx);
}

int32_t parts_for(int32_t max_ctx, int32_t P) {
  const int64_t n = (static_cast<int64_t>(max_ctx) + P - 1) / P;
  return static_cast<int32_t>(n > 0 ? n : 1);
}

using LaunchFn = pkv_status (*)(const DecodeLaunch&);

template <typename KV, int D>
LaunchFn pick_group(int G) {
  switch (G) {
    case 1: return launch_decode<KV, D, 1>;
    case 2: return launch_decode<KV, D, 2>;
    case 4: return launch_decode<KV, D, 4>;
    case 8: return launch_decode<KV, D, 8>;
    default: return nullptr;
  }
}

LaunchFn pick(int32_t kv_dtype, int D, int G) {
  switch (kv_dtype) {
    case PKV_F32:
      if (D == 64) return pick_group<F32, 64>(G);
      if (D == 128) return pick_group<F32, 128>(G);
      return nullptr;
    case PKV_BF16:
      if (D == 64) return pick_group<BF16, 64>(G);
      if (D == 128) return pick_group<BF16, 128>(G);
      if (D == 256) return pick_group<BF16, 256>(G);
      return nullptr;
    case PKV_INT8:
      if (D == 64) return pick_group<INT8, 64>(G);
      if (D == 128) return pick_group<INT8, 128>(G);
      if (D == 256) return pick_group<INT8, 256>(G);
      return nullptr;
    case PKV_FP8_E4M3:
      if (D == 64) return pick_group<FP8, 64>(G);
      if (D == 128) return pick_group<FP8, 128>(G);
      if (D == 256) return pick_group<FP8, 256>(G);
      return nullptr;
    default:
      return nullptr;
  }
}

}  // namespace
}  // namespace pkv

extern "C" int32_t paged_attention_partition_tokens(int32_t num_seqs, int32_t num_q_heads,
                                                    int32_t num_kv_heads,
                                                    int32_t max_context_len,
                                                    int32_t partition_tokens) {
  if (num_seqs < 0 || num_kv_heads <= 0 || num_q_heads <= 0 || num_q_heads % num_kv_heads != 0 ||
      max_context_len < 0)
    return 0;
  return pkv::resolve_partition(num_seqs, num_q_heads, num_kv_heads, max_context_len,
                                partition_tokens);
}

extern "C" size_t paged_attention_workspace_bytes(int32_t num_seqs, int32_t num_q_heads,
                                                  int32_t num_kv_heads, int32_t head_dim,
                                                  int32_t max_context_len,
                                                  int32_t partition_tokens) {
  if (num_seqs <= 0 || num_q_heads <= 0 || num_kv_heads <= 0 || head_dim <= 0 ||
      max_context_len < 0)
    return 0;
  const int32_t P = pkv::resolve_partition(num_seqs, num_q_heads, num_kv_heads, max_context_len,
                                           partition_tokens);
  if (P <= 0) return 0;
  const int32_t parts = pkv::parts_for(max_context_len, P);
  if (parts <= 1) return 0;
  return static_cast<size_t>(num_seqs) * num_q_heads * parts * (head_dim + 2) * sizeof(float);
}

namespace {

// The step's new token per sequence, appended by the decode call itself.
struct FusedAppend {
  const void* k_new;
  const void* v_new;
  const int64_t* slots;
  int32_t src_dtype;
};

pkv_status decode_impl(const void* q, const void* k_cache, const void* v_cache,
                       const int32_t* block_tables, const int32_t* context_lens, int32_t num_seqs,
                       int32_t num_q_heads, int32_t num_kv_heads, int32_t head_dim,
                       int32_t block_size, int64_t num_blocks, int32_t max_blocks_per_seq,
                       int32_t max_context_len, float scale, int32_t q_dtype, int32_t kv_dtype,
                       const float* k_scale, const float* v_scale, float* out, void* workspace,
                       size_t workspace_bytes, int32_t partition_tokens, int32_t* device_status,
                       pkv_stream_t stream, const FusedAppend* fa) {
  using namespace pkv;
  if (num_seqs < 0 || num_q_heads <= 0 || num_kv_heads <= 0 || head_dim <= 0 ||
      num_blocks <= 0 || num_blocks > INT32_MAX || max_blocks_per_seq <= 0 || max_context_len < 0)
    return PKV_ERR_INVALID_ARG;
  if (num_q_heads % num_kv_heads != 0) return PKV_ERR_INVALID_ARG;
  if (!is_pow2(block_size) || block_size > 4096) return PKV_ERR_UNSUPPORTED;
  if (q_dtype != PKV_F32 && q_dtype != PKV_BF16) return PKV_ERR_UNSUPPORTED;
  if (partition_tokens < 0 || partition_tokens % 64 != 0) return PKV_ERR_INVALID_ARG;
  if (static_cast<int64_t>(max_context_len) > static_cast<int64_t>(max_blocks_per_seq) * block_size)
    return PKV_ERR_INVALID_ARG;
  const int G = num_q_heads / num_kv_heads;
  const int32_t forced = forced_kernel();
  const bool use_mma2 = forced == PKV_DECODE_KERNEL_AUTO &&
                        mma2_path_supported(kv_dtype, head_dim, G, block_size, num_blocks);
  const bool use_mma = !use_mma2 && forced != PKV_DECODE_KERNEL_CUDA_CORE &&
                       mma_path_supported(kv_dtype, head_dim, G, block_size, num_blocks);
  LaunchFn fn = pick(kv_dtype, head_dim, G);
  if (!use_mma2 && !use_mma && !fn) return PKV_ERR_UNSUPPORTED;
  if (!std::isfinite(scale)) return PKV_ERR_INVALID_ARG;
  if (num_seqs == 0) return PKV_OK;
  if (!q || !k_cache || !v_cache || !block_tables || !context_lens || !out)
    return PKV_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(k_cache) || !aligned16(v_cache) || !aligned16(out) ||
      (reinterpret_cast<uintptr_t>(block_tables) & 3u) ||
      (reinterpret_cast<uintptr_t>(context_lens) & 3u))
    return PKV_ERR_INVALID_ARG;
  if ((kv_dtype == PKV_FP8_E4M3 || kv_dtype == PKV_INT8) && (!k_scale || !v_scale))
    return PKV_ERR_INVALID_ARG;

  int32_t P =
      resolve_partition(num_seqs, num_q_heads, num_kv_heads, max_context_len, partition_tokens);
  // 8-bit rows are half the bytes of 16-bit ones, so the automatic partition
  // (counted in tokens for 16-bit rows) doubles, at most 4096: each CTA then
  // moves the bytes it would for a bf16 cache and its fixed start-up and
  // epilogue weigh the same.  Measured on the 7B-shaped layer: FP8 114.6 ->
  // 112.1 us, INT8 116.6 -> 115.3.  The workspace this needs is never more
  // than paged_attention_workspace_bytes gives for partition_tokens = 0.
  if (partition_tokens == 0 && (kv_dtype == PKV_FP8_E4M3 || kv_dtype == PKV_INT8) && P < 4096)
    P *= 2;
  const int32_t parts = parts_for(max_context_len, P);
  const size_t need = paged_attention_workspace_bytes(num_seqs, num_q_heads, num_kv_heads,
                                                      head_dim, max_context_len, P);
  if (need > 0 && (!workspace || workspace_bytes < need || !aligned16(workspace)))
    return PKV_ERR_INVALID_ARG;
  if (static_cast<int64_t>(parts) > 65535) return PKV_ERR_UNSUPPORTED;
  if (num_seqs > 65535 || num_kv_heads > 65535) return PKV_ERR_UNSUPPORTED;

  DecodeLaunch a{};
  DecodeParams& p = a.p;
  p.q = q;
  p.k_cache = static_cast<const uint8_t*>(k_cache);
  p.v_cache = static_cast<const uint8_t*>(v_cache);
  p.block_tables = block_tables;
  p.context_lens = context_lens;
  p.k_scale = k_scale;
  p.v_scale = v_scale;
  p.out = out;
  float* ws = static_cast<float*>(workspace);
  p.part_ml = need > 0 ? ws : nullptr;
  p.part_o = need > 0 ? ws + static_cast<size_t>(num_seqs) * num_q_heads * parts * 2 : nullptr;
  p.status = device_status;
  p.num_kv_heads = num_kv_heads;
  p.num_q_heads = num_q_heads;
  p.bs_log2 = log2i(block_size);
  p.max_blocks_per_seq = max_blocks_per_seq;
  p.num_blocks = num_blocks;
  p.partition_tokens = P;
  p.max_parts = parts;
  p.q_is_bf16 = q_dtype == PKV_BF16;
  p.qk_scale_log2 = scale * 1.4426950408889634f;
  p.test_stall_bytes = g_stall_bytes.load(std::memory_order_relaxed);
  a.num_seqs = num_seqs;
  a.stream = reinterpret_cast<cudaStream_t>(stream);
  if (fa) {
    // The transposed kernel copies 16-bit rows itself.  8-bit caches keep the
    // append kernel: quantising in front of a warp's first copy cost more on
    // the ragged FP8 step (871.7 against 852.9 + the append, us per layer) and
    // was even on the INT8 layer.
    if (use_mma2 && kv_dtype == PKV_BF16) {
      p.k_new = fa->k_new;
      p.v_new = fa->v_new;
      p.new_slots = fa->slots;
      p.new_src_dtype = fa->src_dtype;
    } else {          // other kernels: the append kernel first, on the same stream
      const pkv_status st = reshape_and_cache(
          fa->k_new, fa->v_new, fa->slots, const_cast<void*>(k_cache),
          const_cast<void*>(v_cache), num_seqs, num_kv_heads, head_dim, block_size, num_blocks,
          fa->src_dtype, kv_dtype, k_scale, v_scale, device_status, stream);
      if (st != PKV_OK) return st;
    }
  }
  if (use_mma2)
    return launch_decode_mma2(a, k_cache, v_cache, head_dim, num_blocks, q_dtype == PKV_F32,
                              kv_dtype);
  if (use_mma)
    return launch_decode_mma(a, k_cache, v_cache, head_dim, num_blocks, q_dtype == PKV_F32,
                             kv_dtype == PKV_FP8_E4M3);
  return fn(a);
}

}  // namespace

extern "C" pkv_status paged_attention_decode(
    const void* q, const void* k_cache, const void* v_cache, const int32_t* block_tables,
    const int32_t* context_lens, int32_t num_seqs, int32_t num_q_heads, int32_t num_kv_heads,
    int32_t head_dim, int32_t block_size, int64_t num_blocks, int32_t max_blocks_per_seq,
    int32_t max_context_len, float scale, int32_t q_dtype, int32_t kv_dtype, const float* k_scale,
    const float* v_scale, float* out, void* workspace, size_t workspace_bytes,
    int32_t partition_tokens, int32_t* device_status, pkv_stream_t stream) {
  return decode_impl(q, k_cache, v_cache, block_tables, context_lens, num_seqs, num_q_heads,
                     num_kv_heads, head_dim, block_size, num_blocks, max_blocks_per_seq,
                     max_context_len, scale, q_dtype, kv_dtype, k_scale, v_scale, out, workspace,
                     workspace_bytes, partition_tokens, device_status, stream, nullptr);
}

extern "C" pkv_status paged_attention_decode_append(
    const void* q, const void* k_new, const void* v_new, const int64_t* slot_mapping,
    int32_t src_dtype, void* k_cache, void* v_cache, const int32_t* block_tables,
    const int32_t* context_lens, int32_t num_seqs, int32_t num_q_heads, int32_t num_kv_heads,
    int32_t head_dim, int32_t block_size, int64_t num_blocks, int32_t max_blocks_per_seq,
    int32_t max_context_len, float scale, int32_t q_dtype, int32_t kv_dtype, const float* k_scale,
    const float* v_scale, float* out, void* workspace, size_t workspace_bytes,
    int32_t partition_tokens, int32_t* device_status, pkv_stream_t stream) {
  using namespace pkv;
  const bool quant = kv_dtype == PKV_FP8_E4M3 || kv_dtype == PKV_INT8;
  const bool combo = quant ? (src_dtype == PKV_F32 || src_dtype == PKV_BF16)
                           : (src_dtype == kv_dtype && (kv_dtype == PKV_F32 || kv_dtype == PKV_BF16));
  if (!combo) return PKV_ERR_UNSUPPORTED;
  if (num_seqs > 0) {
    if (!k_new || !v_new || !slot_mapping) return PKV_ERR_INVALID_ARG;
    if (!aligned16(k_new) || !aligned16(v_new) ||
        (reinterpret_cast<uintptr_t>(slot_mapping) & 7u))
      return PKV_ERR_INVALID_ARG;
  }
  const FusedAppend fa{k_new, v_new, slot_mapping, src_dtype};
  return decode_impl(q, k_cache, v_cache, block_tables, context_lens, num_seqs, num_q_heads,
                     num_kv_heads, head_dim, block_size, num_blocks, max_blocks_per_seq,
                     max_context_len, scale, q_dtype, kv_dtype, k_scale, v_scale, out, workspace,
                     workspace_bytes, partition_tokens, device_status, stream, &fa);
}

extern "C" pkv_status pkv_test_force_decode_kernel(int32_t kernel) {
  if (kernel != PKV_DECODE_KERNEL_AUTO && kernel != PKV_DECODE_KERNEL_HEADS_AS_ROWS &&
      kernel != PKV_DECODE_KERNEL_CUDA_CORE)
    return PKV_ERR_INVALID_ARG;
  pkv::g_forced_kernel.store(kernel, std::memory_order_relaxed);
  return PKV_OK;
}

extern "C" pkv_status pkv_test_decode_stall(uint32_t bytes) {
  if (bytes % 16 != 0 || bytes > 65536) return PKV_ERR_INVALID_ARG;
  pkv::g_stall_bytes.store(bytes, std::memory_order_relaxed);
  return PKV_OK;
}
