// Host side of the tensor-core decode path: TMA tensor maps over the paged
// cache and the kernel launch for each (head_dim, q type, group rows) variant.
#include <cudaTypedefs.h>

#include <mutex>

#include "decode_mma.cuh"
#include "decode_mma_fp8.cuh"
#include "decode_mma2.cuh"
#include "tmap.cuh"

namespace pkv {

namespace {

template <int D>
struct MmaShape;
template <>
struct MmaShape<128> {
  static constexpr int NW = 4, STAGES = 3;
};
template <>
struct MmaShape<64> {
  static constexpr int NW = 4, STAGES = 6;
};

template <int D, bool QF32, bool ROWS16>
pkv_status launch(const CUtensorMap& tk, const CUtensorMap& tv, const MmaParams& mp, int num_seqs,
                  cudaStream_t stream) {
  constexpr int NW = MmaShape<D>::NW, STAGES = MmaShape<D>::STAGES;
  using SM = MmaSmem<D, NW, STAGES>;
  const int bs = 1 << mp.p.bs_log2;
  const int table_entries = (mp.p.partition_tokens + bs - 1) / bs + 2;
  const size_t smem = SM::bytes(table_entries);
  auto kern = paged_decode_mma_kernel<D, QF32, ROWS16, NW, STAGES>;
  if (!opt_in_smem(reinterpret_cast<const void*>(kern), static_cast<int>(smem)))
    return PKV_ERR_CUDA;
  dim3 grid(mp.p.num_kv_heads, mp.p.max_parts, num_seqs);
  kern<<<grid, NW * 32, smem, stream>>>(tk, tv, mp);
  if (cudaGetLastError() != cudaSuccess) return PKV_ERR_CUDA;
  return PKV_OK;
}

// FP8 caches (head_dim 128): 4 KiB stages, six deep, two CTAs per SM.
template <bool QF32, bool ROWS16>
pkv_status launch_fp8(const CUtensorMap& tk, const CUtensorMap& tv, const MmaParams& mp,
                      int num_seqs, cudaStream_t stream) {
  constexpr int NW = 4, STAGES = 6;
  using SM = MmaFp8Smem<NW, STAGES>;
  const int bs = 1 << mp.p.bs_log2;
  const int table_entries = (mp.p.partition_tokens + bs - 1) / bs + 2;
  const size_t smem = SM::bytes(table_entries);
  auto kern = paged_decode_mma_fp8_kernel<QF32, ROWS16, NW, STAGES>;
  if (!opt_in_smem(reinterpret_cast<const void*>(kern), static_cast<int>(smem)))
    return PKV_ERR_CUDA;
  dim3 grid(mp.p.num_kv_heads, mp.p.max_parts, num_seqs);
  kern<<<grid, NW * 32, smem, stream>>>(tk, tv, mp);
  if (cudaGetLastError() != cudaSuccess) return PKV_ERR_CUDA;
  return PKV_OK;
}

// Transposed mma.sync kernel with NW warps and STAGES-deep rings of CH-token
// chunks per warp.
template <typename KV, int D, bool QF32, int NW, int STAGES, int CH>
pkv_status launch_mma2_shape(const CUtensorMap& tk, const CUtensorMap& tv, const MmaParams& mp,
                             int num_seqs, cudaStream_t stream) {
  using SM = Mma2Smem<KV, D, NW, STAGES, CH>;
  const int bs = 1 << mp.p.bs_log2;
  const int table_entries = (mp.p.partition_tokens + bs - 1) / bs + 2;
  const size_t smem = SM::bytes(table_entries);
  auto kern = paged_decode_mma2_kernel<KV, D, QF32, NW, STAGES, CH>;
  if (!opt_in_smem(reinterpret_cast<const void*>(kern), static_cast<int>(smem)))
    return PKV_ERR_CUDA;
  dim3 grid(mp.p.num_kv_heads * mp.q_split, mp.p.max_parts, num_seqs);
  if (launch_pdl(kern, grid, dim3(NW * 32), smem, stream, tk, tv, mp) != cudaSuccess)
    return PKV_ERR_CUDA;
  return PKV_OK;
}

// Tokens per chunk of the transposed kernel: 32 for 8-bit rows, 16 otherwise.
int mma2_chunk(int32_t kv_dtype) { return kv_dtype == PKV_BF16 ? 16 : 32; }

// CTA shape of the transposed kernel: 4 warps, each its own TMA ring.
// 256-byte rows (16-bit, head_dim 128; 8 KiB stages of 16 tokens) run 2 stages
// deep so 3 CTAs share an SM (12 warps): while one CTA is in its start-up
// (context, block table, first TMA round trip) or its epilogue, two others
// keep streaming.  Against 4 x 3 (2 CTAs per SM) the 7B / 70B-shaped layers
// went from 93.5 to 96.7 % and from 87.7 to 91.3 % of HBM.  8-bit rows take
// 32-token chunks (8 KiB stages, the same 3 CTAs per SM): against 16-token
// chunks at 4 CTAs per SM, INT8 121.2 -> 119.2 us per call on the 7B layer and the
// ragged FP8 layer 853 -> 833 us; 2 CTAs per SM lost 15-20 %.  16-bit
// head_dim 64 rows (128 bytes) run 4 x 3 with 16-token chunks.
template <typename KV, int D, bool QF32>
pkv_status launch_mma2(const CUtensorMap& tk, const CUtensorMap& tv, const MmaParams& mp,
                       int num_seqs, cudaStream_t stream) {
  if constexpr (D * KV::kBytes == 256)
    return launch_mma2_shape<KV, D, QF32, 4, 2, 16>(tk, tv, mp, num_seqs, stream);
  else if constexpr (D * KV::kBytes == 512)   // bf16, head_dim 256: 16 KiB stages, 3 CTAs per SM
    return launch_mma2_shape<KV, D, QF32, 2, 2, 16>(tk, tv, mp, num_seqs, stream);
  else if constexpr (KV::kBytes == 1)
    return launch_mma2_shape<KV, D, QF32, 4, 2, 32>(tk, tv, mp, num_seqs, stream);
  else
    return launch_mma2_shape<KV, D, QF32, 4, 3, 16>(tk, tv, mp, num_seqs, stream);
}

}  // namespace

bool mma2_path_supported(int32_t kv_dtype, int head_dim, int group, int block_size,
                         int64_t num_blocks) {
  if (kv_dtype == PKV_BF16) {
    if (head_dim != 64 && head_dim != 128 && head_dim != 256) return false;
  } else if (kv_dtype == PKV_FP8_E4M3 || kv_dtype == PKV_INT8) {
    if (head_dim != 128) return false;
  } else {
    return false;
  }
  if (group < 1 || (group > 8 && group != 16)) return false;   // 16: two CTAs of 8 heads
  if (block_size < 8) return false;
  if (num_blocks * block_size > 0x7fffffffLL) return false;
  return encode_fn() != nullptr;
}

pkv_status launch_decode_mma2(const DecodeLaunch& a, const void* k_cache, const void* v_cache,
                              int head_dim, int64_t num_blocks, bool q_f32, int32_t kv_dtype) {
  const DecodeParams& p = a.p;
  const int bs = 1 << p.bs_log2;
  const int ch = mma2_chunk(kv_dtype);
  MmaParams mp{p, bs < ch ? bs : ch};
  mp.q_split = p.num_q_heads / p.num_kv_heads > 8 ? 2 : 1;
  CUtensorMap tk, tv;
  const int64_t rows = num_blocks * bs;
  const bool byte_codes = kv_dtype != PKV_BF16;
  if (!make_map(&tk, k_cache, head_dim, p.num_kv_heads, rows, mp.box_rows, byte_codes) ||
      !make_map(&tv, v_cache, head_dim, p.num_kv_heads, rows, mp.box_rows, byte_codes))
    return PKV_ERR_CUDA;
  pkv_status st;
  if (kv_dtype == PKV_FP8_E4M3)
    st = q_f32 ? launch_mma2<FP8, 128, true>(tk, tv, mp, a.num_seqs, a.stream)
               : launch_mma2<FP8, 128, false>(tk, tv, mp, a.num_seqs, a.stream);
  else if (kv_dtype == PKV_INT8)
    st = q_f32 ? launch_mma2<INT8, 128, true>(tk, tv, mp, a.num_seqs, a.stream)
               : launch_mma2<INT8, 128, false>(tk, tv, mp, a.num_seqs, a.stream);
  else if (head_dim == 256)
    st = q_f32 ? launch_mma2<BF16, 256, true>(tk, tv, mp, a.num_seqs, a.stream)
               : launch_mma2<BF16, 256, false>(tk, tv, mp, a.num_seqs, a.stream);
  else if (head_dim == 128)
    st = q_f32 ? launch_mma2<BF16, 128, true>(tk, tv, mp, a.num_seqs, a.stream)
               : launch_mma2<BF16, 128, false>(tk, tv, mp, a.num_seqs, a.stream);
  else
    st = q_f32 ? launch_mma2<BF16, 64, true>(tk, tv, mp, a.num_seqs, a.stream)
               : launch_mma2<BF16, 64, false>(tk, tv, mp, a.num_seqs, a.stream);
  if (st != PKV_OK) return st;
  if (p.max_parts > 1) {
    const dim3 rgrid(a.num_seqs * p.num_q_heads);
    const cudaError_t e =
        head_dim == 256   ? launch_pdl(paged_decode_reduce_kernel<256>, rgrid, dim3(32), 0, a.stream, p)
        : head_dim == 128 ? launch_pdl(paged_decode_reduce_kernel<128>, rgrid, dim3(32), 0, a.stream, p)
                          : launch_pdl(paged_decode_reduce_kernel<64>, rgrid, dim3(32), 0, a.stream, p);
    if (e != cudaSuccess) return PKV_ERR_CUDA;
  }
  return PKV_OK;
}

bool mma_path_supported(int32_t kv_dtype, int head_dim, int group, int block_size,
                        int64_t num_blocks) {
  if (kv_dtype == PKV_BF16) {
    if (head_dim != 64 && head_dim != 128) return false;
  } else if (kv_dtype == PKV_FP8_E4M3) {
    if (head_dim != 128) return false;
  } else {
    return false;
  }
  if (group < 1 || group > 16) return false;
  if (block_size < 8) return false;   // a TMA box is at least 8 rows (1 KiB)
  if (num_blocks * block_size > 0x7fffffffLL) return false;
  return encode_fn() != nullptr;
}

pkv_status launch_decode_mma(const DecodeLaunch& a, const void* k_cache, const void* v_cache,
                             int head_dim, int64_t num_blocks, bool q_f32, bool fp8) {
  const DecodeParams& p = a.p;
  const int bs = 1 << p.bs_log2;
  MmaParams mp{p, bs < kMmaChunk ? bs : kMmaChunk};
  CUtensorMap tk, tv;
  const int64_t rows = num_blocks * bs;
  if (!make_map(&tk, k_cache, head_dim, p.num_kv_heads, rows, mp.box_rows, fp8) ||
      !make_map(&tv, v_cache, head_dim, p.num_kv_heads, rows, mp.box_rows, fp8))
    return PKV_ERR_CUDA;
  const bool rows16 = p.num_q_heads / p.num_kv_heads > 8;
  pkv_status st;
  if (fp8) {
    if (q_f32)
      st = rows16 ? launch_fp8<true, true>(tk, tv, mp, a.num_seqs, a.stream)
                  : launch_fp8<true, false>(tk, tv, mp, a.num_seqs, a.stream);
    else
      st = rows16 ? launch_fp8<false, true>(tk, tv, mp, a.num_seqs, a.stream)
                  : launch_fp8<false, false>(tk, tv, mp, a.num_seqs, a.stream);
  } else if (head_dim == 128) {
    if (q_f32)
      st = rows16 ? launch<128, true, true>(tk, tv, mp, a.num_seqs, a.stream)
                  : launch<128, true, false>(tk, tv, mp, a.num_seqs, a.stream);
    else
      st = rows16 ? launch<128, false, true>(tk, tv, mp, a.num_seqs, a.stream)
                  : launch<128, false, false>(tk, tv, mp, a.num_seqs, a.stream);
  } else {
    if (q_f32)
      st = rows16 ? launch<64, true, true>(tk, tv, mp, a.num_seqs, a.stream)
                  : launch<64, true, false>(tk, tv, mp, a.num_seqs, a.stream);
    else
      st = rows16 ? launch<64, false, true>(tk, tv, mp, a.num_seqs, a.stream)
                  : launch<64, false, false>(tk, tv, mp, a.num_seqs, a.stream);
  }
  if (st != PKV_OK) return st;
  if (p.max_parts > 1) {
    const dim3 rgrid(a.num_seqs * p.num_q_heads);
    const cudaError_t e =
        head_dim == 128 ? launch_pdl(paged_decode_reduce_kernel<128>, rgrid, dim3(32), 0, a.stream, p)
                        : launch_pdl(paged_decode_reduce_kernel<64>, rgrid, dim3(32), 0, a.stream, p);
    if (e != cudaSuccess) return PKV_ERR_CUDA;
  }
  return PKV_OK;
}

}  // namespace pkv
