// PagedAttention decode, CUDA-core path ("nano-vLLM architecture" section 4.2:
// attention that reads K/V through the logical -> physical block mapping;
// "LLM inference tutorial" sections 4.2 get_kv and 4.4 MHA/GQA forward).
//
// Work decomposition.  One CTA per (sequence s, KV head g, partition of P
// tokens).  The CTA owns all G = Hq/Hkv query heads of KV head g, so every
// K/V byte is read from HBM once per KV head (query-group packing).  The grid
// is (Hkv, partitions, sequences) with the KV head fastest: CTAs that start
// together read the same tokens of every head, i.e. whole [Hkv, D] token rows
// of a block, so DRAM pages are read end to end instead of one head's slice
// at a time (worth about 3 % of HBM bandwidth on 128K-token contexts).  Inside
// the CTA each warp is an independent streaming consumer: it takes every
// NW-th chunk of CH tokens of the partition, stages the chunk's K and V rows
// into its own shared-memory ring with 16-byte cp.async copies (STAGES deep,
// so STAGES-1 chunks are in flight per warp), and folds the chunk into a
// running (online) softmax held in registers.  No CTA-wide barrier runs inside
// the token loop.
//
// Lane layout.  A row (one token, one KV head) is RB = D * elem bytes, split
// into LPR = RB/16 segments of 16 bytes; a warp instruction covers TPI =
// 32/LPR rows.  Lane (grp, seg) always handles segment `seg` of rows
// grp, grp+TPI, ... so its slice of q, its accumulator and its smem reads
// stay fixed: the QK dot is a 16-byte partial dot reduced over the LPR lanes
// of the row with xor-shuffles, and PV accumulates 16 bytes' worth of
// dimensions per lane with no shuffles at all.
//
// Softmax in base 2: q is pre-multiplied by scale * log2(e) (and by the FP8
// K scale), so p = exp2(z - m) and the final division by sum(p) gives the
// same result as exp(.) of the unscaled logits.
//
// Split-KV.  With more than one partition the CTA writes (m, l, o) partials
// (o unnormalised, already times the V scale) and a second kernel combines
// them: m* = max m_i, l = sum l_i 2^(m_i - m*), out = sum o_i 2^(m_i - m*) / l.
#pragma once

#include <math_constants.h>

#include "common.cuh"

namespace pkv {

struct DecodeParams {
  const void* q;
  const uint8_t* k_cache;
  const uint8_t* v_cache;
  const int32_t* block_tables;
  const int32_t* context_lens;
  const float* k_scale;
  const float* v_scale;
  float* out;
  float* part_ml;   // [S, Hq, max_parts, 2]  (m in log2 units, l)
  float* part_o;    // [S, Hq, max_parts, D]
  int32_t* status;
  int32_t num_kv_heads;
  int32_t num_q_heads;
  int32_t bs_log2;
  int32_t max_blocks_per_seq;
  int64_t num_blocks;
  int32_t partition_tokens;
  int32_t max_parts;
  int32_t q_is_bf16;
  float qk_scale_log2;   // scale * log2(e)
  // Fused append (transposed kernel only; k_new == nullptr: none): the new
  // token of sequence s, rows k_new/v_new[s, Hkv, D] of type new_src_dtype,
  // goes to slot new_slots[s], which must be the slot of position
  // context_lens[s] - 1; the CTA of that position's partition writes it for
  // its KV head before it reads the block.
  const void* k_new;
  const void* v_new;
  const int64_t* new_slots;
  int32_t new_src_dtype;
  // Tests of the bounded waits (pkv_test_decode_stall): bytes the transposed
  // kernel's CTA (0, 0, 0) adds to warp 0's first barrier phase and never
  // copies, so that wait runs out; 0 in every normal call.
  uint32_t test_stall_bytes;
};

__device__ __forceinline__ void cp_async16(uint32_t smem_addr, const void* gptr, int src_bytes) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;\n" ::"r"(smem_addr), "l"(gptr),
               "r"(src_bytes)
               : "memory");
}
__device__ __forceinline__ void cp_async_commit() {
  asm volatile("cp.async.commit_group;\n" ::: "memory");
}
template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;\n" ::"n"(N) : "memory");
}

// Longest context the launch can cover: the block table's capacity and the
// partitions the grid was sized for.  Longer contexts are clamped and flagged.
__device__ __forceinline__ int context_cap(const DecodeParams& p) {
  const long long by_table = static_cast<long long>(p.max_blocks_per_seq) << p.bs_log2;
  const long long by_grid = static_cast<long long>(p.max_parts) * p.partition_tokens;
  const long long c = by_table < by_grid ? by_table : by_grid;
  return static_cast<int>(c < 0x7fffffffLL ? c : 0x7fffffffLL);
}

template <typename KV, int D>
struct DecodeShape {
  static constexpr int RB = D * KV::kBytes;   // row bytes
  static constexpr int LPR = RB / 16;         // lanes per row
  static constexpr int TPI = 32 / LPR;        // rows per warp instruction
  static constexpr int EPL = KV::kPerVec;     // elements per lane
  static constexpr int CH = 8 * TPI;          // tokens per chunk (8 rows per lane)
  static constexpr int CHUNK_VEC = CH * LPR;  // uint4 per K (or V) chunk = 256
  static_assert(RB >= 64 && RB <= 512 && (RB & (RB - 1)) == 0, "row bytes");
  static_assert(CHUNK_VEC == 256, "chunk is 4 KiB");
};

template <typename KV, int D, int G, int NW, int STAGES>
struct DecodeSmem {
  using S = DecodeShape<KV, D>;
  static constexpr int kStageVec = 2 * S::CHUNK_VEC;                 // K + V
  static constexpr int kWarpVec = STAGES * kStageVec + (S::CH * G + 3) / 4;  // + zbuf
  static constexpr int kWarpBytes = kWarpVec * 16;
  static_assert(STAGES * kStageVec * 16 >= G * (D + 2) * 4, "combine area fits a warp ring");
  static size_t bytes(int table_entries) {
    return static_cast<size_t>(NW) * kWarpBytes + static_cast<size_t>(table_entries) * 4;
  }
};

template <typename KV, int D, int G, int NW, int STAGES>
__global__ void __launch_bounds__(NW * 32)
    paged_decode_kernel(const DecodeParams p) {
  using S = DecodeShape<KV, D>;
  using SM = DecodeSmem<KV, D, G, NW, STAGES>;
  constexpr int LPR = S::LPR, TPI = S::TPI, EPL = S::EPL, CH = S::CH, RB = S::RB;

  extern __shared__ __align__(16) uint4 smem[];
  const int s = blockIdx.z, g = blockIdx.x, part = blockIdx.y;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int grp = lane / LPR, seg = lane % LPR;
  const int P = p.partition_tokens;
  const int bs = 1 << p.bs_log2;

  int ctx = __ldg(p.context_lens + s);
  const int cap = context_cap(p);
  if (ctx < 0 || ctx > cap) {
    if (part == 0 && threadIdx.x == 0) flag_status(p.status, PKV_DEV_BAD_CONTEXT);
    ctx = ctx < 0 ? 0 : cap;
  }
  const int nparts = (ctx + P - 1) / P;
  if (part >= (nparts > 0 ? nparts : 1)) return;
  const int hq0 = g * G;
  if (ctx == 0) {   // nothing to attend: output 0
    for (int i = threadIdx.x; i < G * D; i += NW * 32)
      p.out[(static_cast<int64_t>(s) * p.num_q_heads + hq0) * D + i] = 0.f;
    return;
  }
  const int t_begin = part * P;
  const int t_end = min(t_begin + P, ctx);

  // Block-table entries of this partition -> smem, validated once.
  int32_t* sbt = reinterpret_cast<int32_t*>(smem + NW * SM::kWarpVec);
  const int lb0 = t_begin >> p.bs_log2;
  const int nlb = ((t_end - 1) >> p.bs_log2) - lb0 + 1;
  const int32_t* bt_row = p.block_tables + static_cast<int64_t>(s) * p.max_blocks_per_seq;
  for (int i = threadIdx.x; i < nlb; i += NW * 32) {
    int32_t b = __ldg(bt_row + lb0 + i);
    if (b < 0 || b >= p.num_blocks) {
      flag_status(p.status, PKV_DEV_BAD_BLOCK);
      b = -1;
    }
    sbt[i] = b;
  }
  __syncthreads();

  // This lane's slice of the G query heads, pre-scaled into log2 units.
  float qs[G][EPL];
  {
    float ks = p.qk_scale_log2;
    if (KV::kBytes == 1) ks *= __ldg(p.k_scale + g);
#pragma unroll
    for (int h = 0; h < G; ++h) {
      const int64_t base = (static_cast<int64_t>(s) * p.num_q_heads + hq0 + h) * D + seg * EPL;
#pragma unroll
      for (int e = 0; e < EPL; ++e) {
        float v;
        if (p.q_is_bf16)
          v = __bfloat162float(static_cast<const __nv_bfloat16*>(p.q)[base + e]);
        else
          v = static_cast<const float*>(p.q)[base + e];
        qs[h][e] = v * ks;
      }
    }
  }

  float m[G], l[G], acc[G][EPL];
#pragma unroll
  for (int h = 0; h < G; ++h) {
    m[h] = -CUDART_INF_F;
    l[h] = 0.f;
#pragma unroll
    for (int e = 0; e < EPL; ++e) acc[h][e] = 0.f;
  }

  uint4* ring = smem + warp * SM::kWarpVec;
  float* zbuf = reinterpret_cast<float*>(ring + STAGES * SM::kStageVec);
  const uint32_t ring_addr = static_cast<uint32_t>(__cvta_generic_to_shared(ring));
  const int nchunks = (t_end - t_begin + CH - 1) / CH;
  const int my_n = warp < nchunks ? (nchunks - warp + NW - 1) / NW : 0;
  const int64_t head_off = static_cast<int64_t>(g) * RB + seg * 16;
  const int64_t row_stride = static_cast<int64_t>(p.num_kv_heads) * RB;

  auto issue = [&](int it) {
    if (it < my_n) {
      const int stage = it % STAGES;
      const int t0 = t_begin + (warp + it * NW) * CH;
#pragma unroll
      for (int k = 0; k < 8; ++k) {
        const int row = grp + k * TPI;
        const int t = t0 + row;
        int bytes = 0;
        int64_t off = 0;
        if (t < t_end) {
          const int32_t b = sbt[(t >> p.bs_log2) - lb0];
          if (b >= 0) {
            bytes = 16;
            off = ((static_cast<int64_t>(b) << p.bs_log2) + (t & (bs - 1))) * row_stride + head_off;
          }
        }
        const uint32_t dk = ring_addr + (stage * SM::kStageVec + row * LPR + seg) * 16;
        const uint32_t dv = dk + S::CHUNK_VEC * 16;
        cp_async16(dk, p.k_cache + off, bytes);
        cp_async16(dv, p.v_cache + off, bytes);
      }
    }
    cp_async_commit();
  };

#pragma unroll
  for (int st = 0; st < STAGES - 1; ++st) issue(st);

  for (int it = 0; it < my_n; ++it) {
    issue(it + STAGES - 1);
    cp_async_wait<STAGES - 1>();
    __syncwarp();
    const int stage = it % STAGES;
    const uint4* kb = ring + stage * SM::kStageVec;
    const uint4* vb = kb + S::CHUNK_VEC;
    const int t0 = t_begin + (warp + it * NW) * CH;

    // Pass 1: logits of the chunk's rows, chunk max per head.
    float mc[G];
#pragma unroll
    for (int h = 0; h < G; ++h) mc[h] = -CUDART_INF_F;
#pragma unroll
    for (int k = 0; k < 8; ++k) {
      const int row = grp + k * TPI;
      float x[EPL];
      decode16<KV>(kb[row * LPR + seg], x);
      float z[G];
#pragma unroll
      for (int h = 0; h < G; ++h) {
        float a = 0.f;
#pragma unroll
        for (int e = 0; e < EPL; ++e) a = fmaf(qs[h][e], x[e], a);
        z[h] = a;
      }
#pragma unroll
      for (int off = LPR / 2; off > 0; off >>= 1) {
#pragma unroll
        for (int h = 0; h < G; ++h) z[h] += __shfl_xor_sync(0xffffffffu, z[h], off);
      }
      const bool valid = t0 + row < t_end;
#pragma unroll
      for (int h = 0; h < G; ++h) {
        z[h] = valid ? z[h] : -CUDART_INF_F;
        mc[h] = fmaxf(mc[h], z[h]);
      }
      if (seg == 0) {
#pragma unroll
        for (int h = 0; h < G; ++h) zbuf[row * G + h] = z[h];
      }
    }
#pragma unroll
    for (int off = LPR; off < 32; off <<= 1) {
#pragma unroll
      for (int h = 0; h < G; ++h) mc[h] = fmaxf(mc[h], __shfl_xor_sync(0xffffffffu, mc[h], off));
    }
#pragma unroll
    for (int h = 0; h < G; ++h) {
      const float mn = fmaxf(m[h], mc[h]);
      const float alpha = exp2f(m[h] - mn);
      m[h] = mn;
      l[h] *= alpha;
#pragma unroll
      for (int e = 0; e < EPL; ++e) acc[h][e] *= alpha;
    }
    __syncwarp();

    // Pass 2: probabilities and the PV accumulation.
#pragma unroll
    for (int k = 0; k < 8; ++k) {
      const int row = grp + k * TPI;
      float y[EPL];
      decode16<KV>(vb[row * LPR + seg], y);
#pragma unroll
      for (int h = 0; h < G; ++h) {
        const float pr = exp2f(zbuf[row * G + h] - m[h]);
        l[h] += pr;
#pragma unroll
        for (int e = 0; e < EPL; ++e) acc[h][e] = fmaf(pr, y[e], acc[h][e]);
      }
    }
    __syncwarp();
  }
  cp_async_wait<0>();

  // Warp epilogue: sum the TPI row groups (same m across the warp).
#pragma unroll
  for (int off = LPR; off < 32; off <<= 1) {
#pragma unroll
    for (int h = 0; h < G; ++h) {
      l[h] += __shfl_xor_sync(0xffffffffu, l[h], off);
#pragma unroll
      for (int e = 0; e < EPL; ++e) acc[h][e] += __shfl_xor_sync(0xffffffffu, acc[h][e], off);
    }
  }
  __syncwarp();
  // Per-warp results into the warp's own (now idle) ring: [G][D] acc, then m, l.
  float* wres = reinterpret_cast<float*>(ring);
  if (grp == 0) {
#pragma unroll
    for (int h = 0; h < G; ++h)
#pragma unroll
      for (int e = 0; e < EPL; ++e) wres[h * D + seg * EPL + e] = acc[h][e];
  }
  if (lane == 0) {
#pragma unroll
    for (int h = 0; h < G; ++h) {
      wres[G * D + h] = m[h];
      wres[G * D + G + h] = l[h];
    }
  }
  __syncthreads();

  // CTA combine over warps.
  const float vsc = (KV::kBytes == 1) ? __ldg(p.v_scale + g) : 1.f;
  const bool single = nparts == 1;
  for (int i = threadIdx.x; i < G * D; i += NW * 32) {
    const int h = i / D, d = i % D;
    float M = -CUDART_INF_F;
#pragma unroll
    for (int w = 0; w < NW; ++w) {
      const float* r = reinterpret_cast<const float*>(smem + w * SM::kWarpVec);
      M = fmaxf(M, r[G * D + h]);
    }
    float L = 0.f, O = 0.f;
#pragma unroll
    for (int w = 0; w < NW; ++w) {
      const float* r = reinterpret_cast<const float*>(smem + w * SM::kWarpVec);
      const float c = exp2f(r[G * D + h] - M);   // warps without tokens: exp2(-inf) = 0
      L = fmaf(r[G * D + G + h], c, L);
      O = fmaf(r[h * D + d], c, O);
    }
    const int64_t sh = static_cast<int64_t>(s) * p.num_q_heads + hq0 + h;
    if (single) {
      p.out[sh * D + d] = O / L * vsc;
    } else {
      const int64_t pi = sh * p.max_parts + part;
      p.part_o[pi * D + d] = O * vsc;
      if (d == 0) {
        p.part_ml[pi * 2 + 0] = M;
        p.part_ml[pi * 2 + 1] = L;
      }
    }
  }
}

// Combine split-KV partials: one warp (a CTA of 32 threads) per (sequence,
// query head).  Lane i reads the (m, l) of partitions i, i + 32, ...; the warp
// takes their max and weighted sum by shuffles, so a sequence's partials
// cost one round trip instead of one per partition.  Each lane then merges
// output dims lane + 32 v over the partitions, eight partitions in flight.
template <int D>
__global__ void __launch_bounds__(32) paged_decode_reduce_kernel(const DecodeParams p) {
  grid_dependency_wait();   // launched with launch_pdl: the partials are written
  allow_dependents();
  const int sh = blockIdx.x;
  const int lane = threadIdx.x;
  const int s = sh / p.num_q_heads;
  int ctx = __ldg(p.context_lens + s);
  const int cap = context_cap(p);
  ctx = ctx < 0 ? 0 : (ctx > cap ? cap : ctx);
  const int nparts = (ctx + p.partition_tokens - 1) / p.partition_tokens;
  if (nparts <= 1) return;   // written directly by the main kernel
  const float* ml = p.part_ml + static_cast<int64_t>(sh) * p.max_parts * 2;
  const float* po = p.part_o + static_cast<int64_t>(sh) * p.max_parts * D;
  float M = -CUDART_INF_F;
  for (int i = lane; i < nparts; i += 32) M = fmaxf(M, ml[2 * i]);
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, off));
  float L = 0.f;
  for (int i = lane; i < nparts; i += 32) L = fmaf(ml[2 * i + 1], exp2f(ml[2 * i] - M), L);
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) L += __shfl_xor_sync(0xffffffffu, L, off);
  const float invL = 1.f / L;
  constexpr int V = D / 32;   // output dims per lane
  constexpr int U = 8;        // partitions per step
  float acc[V];
#pragma unroll
  for (int v = 0; v < V; ++v) acc[v] = 0.f;
  for (int i0 = 0; i0 < nparts; i0 += U) {
    float x[U][V], w[U];
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int i = i0 + u;
      const bool in = i < nparts;   // warp-uniform
      w[u] = in ? ml[2 * i] : -CUDART_INF_F;
#pragma unroll
      for (int v = 0; v < V; ++v) x[u][v] = in ? po[static_cast<int64_t>(i) * D + lane + 32 * v] : 0.f;
    }
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const float wu = exp2f(w[u] - M);   // 2^-inf = 0 past the last partition
#pragma unroll
      for (int v = 0; v < V; ++v) acc[v] = fmaf(x[u][v], wu, acc[v]);
    }
  }
#pragma unroll
  for (int v = 0; v < V; ++v) p.out[static_cast<int64_t>(sh) * D + lane + 32 * v] = acc[v] * invL;
}

// Host launcher for one instantiation (defined in decode_launch.cuh).
struct DecodeLaunch {
  DecodeParams p;
  int num_seqs;
  cudaStream_t stream;
};

template <typename KV, int D, int G>
pkv_status launch_decode(const DecodeLaunch& a);

// Tensor-core (TMA + mma) path for 16-bit caches; see decode_mma.cuh.
bool mma_path_supported(int32_t kv_dtype, int head_dim, int group, int block_size,
                        int64_t num_blocks);
pkv_status launch_decode_mma(const DecodeLaunch& a, const void* k_cache, const void* v_cache,
                             int head_dim, int64_t num_blocks, bool q_f32, bool fp8);
// Transposed mma.sync path (heads as the mma N columns); see decode_mma2.cuh.
bool mma2_path_supported(int32_t kv_dtype, int head_dim, int group, int block_size,
                         int64_t num_blocks);
pkv_status launch_decode_mma2(const DecodeLaunch& a, const void* k_cache, const void* v_cache,
                              int head_dim, int64_t num_blocks, bool q_f32, int32_t kv_dtype);
}  // namespace pkv
