// Launch helper for one (KV type, head_dim, group) instantiation of the decode
// kernels; included by the per-KV-type translation units.
#pragma once

#include "decode_kernel.cuh"

namespace pkv {

// CTA shape of the CUDA-core path: 4 warps, 3-stage rings (2 chunks = 16 KiB
// of K+V in flight per warp, 96 KiB per CTA, two CTAs per SM).
constexpr int kDecodeWarps = 4;
constexpr int kDecodeStages = 3;

template <typename KV, int D, int G>
pkv_status launch_decode(const DecodeLaunch& a) {
  using SM = DecodeSmem<KV, D, G, kDecodeWarps, kDecodeStages>;
  const DecodeParams& p = a.p;
  const int bs = 1 << p.bs_log2;
  const int table_entries = (p.partition_tokens + bs - 1) / bs + 2;
  const size_t smem = SM::bytes(table_entries);
  auto kern = paged_decode_kernel<KV, D, G, kDecodeWarps, kDecodeStages>;
  if (!opt_in_smem(reinterpret_cast<const void*>(kern), static_cast<int>(smem)))
    return PKV_ERR_CUDA;
  dim3 grid(p.num_kv_heads, p.max_parts, a.num_seqs);
  kern<<<grid, kDecodeWarps * 32, smem, a.stream>>>(p);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return PKV_ERR_CUDA;
  if (p.max_parts > 1) {
    e = launch_pdl(paged_decode_reduce_kernel<D>, dim3(a.num_seqs * p.num_q_heads), dim3(32), 0,
                   a.stream, p);
    if (e != cudaSuccess) return PKV_ERR_CUDA;
  }
  return PKV_OK;
}

#define PKV_INSTANTIATE_DECODE(KV, D)                                   \
  template pkv_status launch_decode<KV, D, 1>(const DecodeLaunch&);    \
  template pkv_status launch_decode<KV, D, 2>(const DecodeLaunch&);    \
  template pkv_status launch_decode<KV, D, 4>(const DecodeLaunch&);    \
  template pkv_status launch_decode<KV, D, 8>(const DecodeLaunch&);

}  // namespace pkv
