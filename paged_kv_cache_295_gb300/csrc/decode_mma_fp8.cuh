// PagedAttention decode, tensor-core path for FP8-E4M3 caches (head_dim 128).
//
// The "ToPG framework" page (section 3.3) stores the KV cache compressed as
// FP8; every E4M3 value is exactly representable in fp16, so the tiles are
// dequantised in registers to fp16 and both products run as fp16
// mma.m16n8k16 with float32 accumulation.  Staging, work split, online
// softmax, tails and the epilogue follow the bf16 tensor-core kernel
// (decode_mma.cuh); what differs is how the 8-bit tiles become mma operands:
//
//  * QK contracts over head_dim, so any fixed permutation of the dimensions
//    applied to both q and K gives the same logits.  Lane (gid, tig) takes the
//    32 contiguous bytes [32*tig, 32*tig + 32) of its token's K row (two
//    16-byte shared loads) and k-step ks uses bytes 4ks..4ks+3 of that slice;
//    q's A fragments are built with the same dimension map.
//  * PV's output dimensions may be permuted too (the epilogue writes each value
//    to its true column): n-tile j, column n holds dimension 16*n + j, so a
//    lane needs bytes [16*gid, 16*gid + 16) of four token rows (four 16-byte
//    loads), paired across tokens with byte permutes.
//  * q (bf16) converts to fp16 exactly in the normal range; a float32 q is
//    split into fp16 hi + lo.  P is rounded to fp16 (2^-11 relative).
//  * The K scale multiplies the logits' base-2 scale; the V scale multiplies
//    the output (value = float(e4m3) * scale[kv_head]).
#pragma once

#include <cuda_fp16.h>

#include "decode_mma.cuh"

namespace pkv {

__device__ __forceinline__ void mma_f16(float* d, const uint32_t* a, uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7},"
      " {%8, %9}, {%0, %1, %2, %3};\n"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// fp16 operands for q: the power of two 2^k that puts the largest |q| `mx` in
// [2^14, 2^15), so any finite q stays finite and a bf16 q exact down to 2^-24
// of that max; `unscale` = 2^-k goes into the logit scale.
__device__ __forceinline__ float q_fp16_scale(float mx, float& unscale) {
  const uint32_t b = __float_as_uint(mx);
  const int ex = b >= 0x00800000u ? static_cast<int>(b >> 23) - 127 : 0;
  const int k = min(max(14 - ex, -126), 126);
  unscale = __uint_as_float(static_cast<uint32_t>(127 - k) << 23);
  return __uint_as_float(static_cast<uint32_t>(127 + k) << 23);
}

__device__ __forceinline__ uint32_t pack_f16(float lo, float hi) {
  __half2 v = __floats2half2_rn(lo, hi);   // .x = lo (low half)
  return *reinterpret_cast<uint32_t*>(&v);
}

// Four E4M3 codes in a 32-bit word -> two f16x2 registers: `lo` holds bytes 0
// and 1 (byte 0 in the low half), `hi` bytes 2 and 3.  One conversion
// instruction per register, no repacking.
__device__ __forceinline__ void e4m3x4_to_f16x2x2(uint32_t w, uint32_t& lo, uint32_t& hi) {
  asm("{\n .reg .b16 a, b;\n mov.b32 {a, b}, %2;\n cvt.rn.f16x2.e4m3x2 %0, a;\n"
      " cvt.rn.f16x2.e4m3x2 %1, b;\n}\n"
      : "=r"(lo), "=r"(hi)
      : "r"(w));
}

// Four signed 8-bit codes -> two f16x2, bytes 0, 1 in lo and 2, 3 in hi (low
// byte in the low half), exactly: with u = code + 128 in [0, 255], the binary16
// whose bits are 0x6400 | u is 1024 + u (exponent 10, mantissa u), so
// subtracting 1152 = 1024 + 128 (bits 0x6480) leaves the code.
__device__ __forceinline__ void s8x4_to_f16x2x2(uint32_t w, uint32_t& lo, uint32_t& hi) {
  const uint32_t u = w ^ 0x80808080u;
  uint32_t a, b;
  asm("prmt.b32 %0, %1, %2, 0x4140;" : "=r"(a) : "r"(u), "r"(0x64646464u));
  asm("prmt.b32 %0, %1, %2, 0x4342;" : "=r"(b) : "r"(u), "r"(0x64646464u));
  asm("sub.rn.f16x2 %0, %1, %2;" : "=r"(lo) : "r"(a), "r"(0x64806480u));
  asm("sub.rn.f16x2 %0, %1, %2;" : "=r"(hi) : "r"(b), "r"(0x64806480u));
}

// The same widening without the final subtraction: each value is code + 1152,
// exactly.  A caller that keeps the offset corrects for it (a constant added
// to every logit of a head cancels in its softmax; for P V it subtracts
// 1152 * sum(P) once at the end).
__device__ __forceinline__ void s8x4_to_f16x2x2_biased(uint32_t w, uint32_t& lo, uint32_t& hi) {
  const uint32_t u = w ^ 0x80808080u;
  asm("prmt.b32 %0, %1, %2, 0x4140;" : "=r"(lo) : "r"(u), "r"(0x64646464u));
  asm("prmt.b32 %0, %1, %2, 0x4342;" : "=r"(hi) : "r"(u), "r"(0x64646464u));
}

// a - b on f16x2 words (round to nearest; exact where the difference is an
// fp16 value, as code + 1152 - 1152 is).
__device__ __forceinline__ uint32_t hsub2_u32(uint32_t a, uint32_t b) {
  uint32_t d;
  asm("sub.rn.f16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
  return d;
}

// Two E4M3 codes (low byte first) -> f16x2 with the low byte in the low half.
__device__ __forceinline__ uint32_t e4m3x2_to_f16x2(uint32_t two) {
  __half2_raw h = __nv_cvt_fp8x2_to_halfraw2(static_cast<__nv_fp8x2_storage_t>(two & 0xFFFFu),
                                             __NV_E4M3);
  return static_cast<uint32_t>(h.x) | (static_cast<uint32_t>(h.y) << 16);
}

template <int NW, int STAGES>
struct MmaFp8Smem {
  static constexpr int kBoxBytes = kMmaChunk * 128;   // [16 rows][128 B] = one K (or V) tile
  static constexpr int kStageBytes = 2 * kBoxBytes;
  static constexpr int kWarpBytes = STAGES * kStageBytes;
  static_assert(kWarpBytes >= 16 * (128 + 2) * 4, "combine area fits a warp ring");
  static size_t bytes(int table_entries) {
    return 1024 + static_cast<size_t>(NW) * kWarpBytes + static_cast<size_t>(table_entries) * 4;
  }
};

template <bool QF32, bool ROWS16, int NW, int STAGES>
__global__ void __launch_bounds__(NW * 32)
    paged_decode_mma_fp8_kernel(const __grid_constant__ CUtensorMap tmap_k,
                                const __grid_constant__ CUtensorMap tmap_v, const MmaParams mp) {
  constexpr int D = 128;
  using SM = MmaFp8Smem<NW, STAGES>;
  constexpr int KSTEPS = D / 16;
  constexpr int NT = D / 8;
  const DecodeParams& p = mp.p;
  const int G = p.num_q_heads / p.num_kv_heads;

  extern __shared__ uint8_t smem_raw[];
  __shared__ __align__(8) uint64_t bars[NW][STAGES];
  uint8_t* smem = smem_raw + ((1024 - (smem_u32(smem_raw) & 1023)) & 1023);

  const int s = blockIdx.z, g = blockIdx.x, part = blockIdx.y;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int gid = lane >> 2, tig = lane & 3;
  const int P = p.partition_tokens;

  int ctx = __ldg(p.context_lens + s);
  const int cap = context_cap(p);
  if (ctx < 0 || ctx > cap) {
    if (part == 0 && threadIdx.x == 0) flag_status(p.status, PKV_DEV_BAD_CONTEXT);
    ctx = ctx < 0 ? 0 : cap;
  }
  const int nparts = (ctx + P - 1) / P;
  if (part >= (nparts > 0 ? nparts : 1)) return;
  const int hq0 = g * G;
  if (ctx == 0) {
    for (int i = threadIdx.x; i < G * D; i += NW * 32)
      p.out[(static_cast<int64_t>(s) * p.num_q_heads + hq0) * D + i] = 0.f;
    return;
  }
  const int t_begin = part * P;
  const int t_end = min(t_begin + P, ctx);

  int32_t* sbt = reinterpret_cast<int32_t*>(smem + NW * SM::kWarpBytes);
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
  if (lane == 0) {
    for (int st = 0; st < STAGES; ++st) mbar_init(smem_u32(&bars[warp][st]), 1);
    asm volatile("fence.mbarrier_init.release.cluster;\n" ::: "memory");
  }
  fence_proxy_async();
  __syncthreads();

  // q as fp16 A fragments with the dimension map of the K slices:
  // logical k = 2*tig + e (+8) of k-step ks  <->  dim 32*tig + 4*ks + e (+2).
  uint32_t qa[KSTEPS][4];
  uint32_t qlo[QF32 ? KSTEPS : 1][4];
  float q_unscale = 1.f;
  {
    const int64_t row0 = static_cast<int64_t>(s) * p.num_q_heads + hq0;
    auto qpair = [&](int ks, int half, int rh, float& x0, float& x1) {
      const int h = gid + 8 * rh;
      const int col = 32 * tig + 4 * ks + 2 * half;
      x0 = x1 = 0.f;
      if (h < G && (ROWS16 || rh == 0)) {
        if (QF32) {
          const float* qf = static_cast<const float*>(p.q) + (row0 + h) * D + col;
          x0 = qf[0];
          x1 = qf[1];
        } else {
          const __nv_bfloat16* qb = static_cast<const __nv_bfloat16*>(p.q) + (row0 + h) * D + col;
          x0 = __bfloat162float(qb[0]);
          x1 = __bfloat162float(qb[1]);
        }
      }
    };
    float mx = 0.f;   // the group's largest |q| (the lanes cover every head and dim)
#pragma unroll
    for (int ks = 0; ks < KSTEPS; ++ks)
#pragma unroll
      for (int half = 0; half < 2; ++half)
#pragma unroll
        for (int rh = 0; rh < 2; ++rh) {
          float x0, x1;
          qpair(ks, half, rh, x0, x1);
          mx = fmaxf(mx, fmaxf(fabsf(x0), fabsf(x1)));
        }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, off));
    const float qmul = q_fp16_scale(mx, q_unscale);
#pragma unroll
    for (int ks = 0; ks < KSTEPS; ++ks) {
#pragma unroll
      for (int half = 0; half < 2; ++half) {
#pragma unroll
        for (int rh = 0; rh < 2; ++rh) {
          float x0, x1;
          qpair(ks, half, rh, x0, x1);
          x0 *= qmul;   // exact: a power of two
          x1 *= qmul;
          const uint32_t hi = pack_f16(x0, x1);
          qa[ks][half * 2 + rh] = hi;
          if (QF32) {
            const __half2 hv = *reinterpret_cast<const __half2*>(&hi);
            qlo[QF32 ? ks : 0][half * 2 + rh] =
                pack_f16(x0 - __low2float(hv), x1 - __high2float(hv));
          }
        }
      }
    }
  }

  float o[NT][4];
#pragma unroll
  for (int j = 0; j < NT; ++j) o[j][0] = o[j][1] = o[j][2] = o[j][3] = 0.f;
  float m0 = -CUDART_INF_F, m1 = -CUDART_INF_F, l0 = 0.f, l1 = 0.f;
  const float sl2 = p.qk_scale_log2 * __ldg(p.k_scale + g) * q_unscale;

  uint8_t* ring = smem + warp * SM::kWarpBytes;
  const uint32_t ring_a = smem_u32(ring);
  const int nchunks = (t_end - t_begin + kMmaChunk - 1) / kMmaChunk;
  const int my_n = warp < nchunks ? (nchunks - warp + NW - 1) / NW : 0;
  const int box_rows = mp.box_rows;
  const int nbox = kMmaChunk / box_rows;
  bool alive = true;

  auto issue = [&](int it) {
    if (it >= my_n || lane != 0) return;
    const int stage = it % STAGES;
    const int t0 = t_begin + (warp + it * NW) * kMmaChunk;
    const uint32_t bar = smem_u32(&bars[warp][stage]);
    uint32_t bytes = 0;
    for (int bx = 0; bx < nbox; ++bx) {
      const int tb = t0 + bx * box_rows;
      if (tb >= ctx) break;
      if (sbt[(tb >> p.bs_log2) - lb0] >= 0) bytes += 2 * box_rows * 128;
    }
    mbar_arrive_expect_tx(bar, bytes);
    const uint32_t sbase = ring_a + stage * SM::kStageBytes;
    for (int bx = 0; bx < nbox; ++bx) {
      const int tb = t0 + bx * box_rows;
      if (tb >= ctx) break;
      const int32_t b = sbt[(tb >> p.bs_log2) - lb0];
      if (b < 0) continue;
      const int z = (b << p.bs_log2) + (tb & ((1 << p.bs_log2) - 1));
      const uint32_t off = bx * box_rows * 128;
      tma_load_3d(sbase + off, &tmap_k, 0, g, z, bar);
      tma_load_3d(sbase + SM::kBoxBytes + off, &tmap_v, 0, g, z, bar);
    }
  };

#pragma unroll
  for (int st = 0; st < STAGES - 1; ++st) issue(st);

  for (int it = 0; it < my_n; ++it) {
    issue(it + STAGES - 1);
    const int stage = it % STAGES;
    const uint32_t parity = (it / STAGES) & 1;
    const bool landed = __all_sync(0xffffffffu, mbar_wait(smem_u32(&bars[warp][stage]), parity));
    if (!landed) {
      if (lane == 0) flag_status(p.status, PKV_DEV_TIMEOUT);
      alive = false;
      for (int k = it + 1; k < min(my_n, it + STAGES); ++k)
        mbar_wait(smem_u32(&bars[warp][k % STAGES]), (k / STAGES) & 1);
      break;
    }
    const int t0 = t_begin + (warp + it * NW) * kMmaChunk;
    const int valid = min(kMmaChunk, ctx - t0);
    uint8_t* kb = ring + stage * SM::kStageBytes;
    uint8_t* vb = kb + SM::kBoxBytes;
    bool hole = valid < kMmaChunk;
    if (!hole) {
      for (int bx = 0; bx < nbox; ++bx)
        if (sbt[((t0 + bx * box_rows) >> p.bs_log2) - lb0] < 0) hole = true;
    }
    if (hole) {   // rows the TMA did not fill become +0 codes
      for (int i = lane; i < kMmaChunk * 8 * 2; i += 32) {
        const int r = (i >> 3) % kMmaChunk;
        const int bx = r / box_rows;
        const bool filled = r < valid && sbt[((t0 + bx * box_rows) >> p.bs_log2) - lb0] >= 0;
        if (!filled) {
          uint8_t* base = (i < kMmaChunk * 8) ? kb : vb;
          *reinterpret_cast<uint4*>(base + r * 128 + ((i & 7) << 4)) = make_uint4(0, 0, 0, 0);
        }
      }
      __syncwarp();
    }

    // ---- S = Q K^T: token gid (n-tile 0) and 8 + gid (n-tile 1) -------------
    float sacc[2][4];
#pragma unroll
    for (int j = 0; j < 2; ++j) {
      sacc[j][0] = sacc[j][1] = sacc[j][2] = sacc[j][3] = 0.f;
      const int r = 8 * j + gid;
      const uint4 w0 = *reinterpret_cast<const uint4*>(kb + swz(r, 2 * tig));
      const uint4 w1 = *reinterpret_cast<const uint4*>(kb + swz(r, 2 * tig + 1));
      const uint32_t wd[8] = {w0.x, w0.y, w0.z, w0.w, w1.x, w1.y, w1.z, w1.w};
#pragma unroll
      for (int ks = 0; ks < KSTEPS; ++ks) {
        const uint32_t b0 = e4m3x2_to_f16x2(wd[ks]);
        const uint32_t b1 = e4m3x2_to_f16x2(wd[ks] >> 16);
        mma_f16(sacc[j], qa[ks], b0, b1);
        if (QF32) mma_f16(sacc[j], qlo[QF32 ? ks : 0], b0, b1);
      }
    }
    // ---- online softmax -----------------------------------------------------------
    float mx0 = -CUDART_INF_F, mx1 = -CUDART_INF_F;
#pragma unroll
    for (int j = 0; j < 2; ++j) {
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        const int t = 8 * j + 2 * tig + e;
        const bool ok = t < valid;
        sacc[j][e] = ok ? sacc[j][e] * sl2 : -CUDART_INF_F;
        sacc[j][2 + e] = ok ? sacc[j][2 + e] * sl2 : -CUDART_INF_F;
        mx0 = fmaxf(mx0, sacc[j][e]);
        mx1 = fmaxf(mx1, sacc[j][2 + e]);
      }
    }
    mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 1));
    mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 2));
    if (ROWS16) {
      mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 1));
      mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 2));
    }
    const float mn0 = fmaxf(m0, mx0);
    const float mn1 = ROWS16 ? fmaxf(m1, mx1) : 0.f;
    const bool grow = mn0 > m0 || (ROWS16 && mn1 > m1);
    if (__any_sync(0xffffffffu, grow)) {
      const float a0 = exp2f(m0 - mn0);
      const float a1 = ROWS16 ? exp2f(m1 - mn1) : 1.f;
      l0 *= a0;
      l1 *= a1;
#pragma unroll
      for (int j = 0; j < NT; ++j) {
        o[j][0] *= a0;
        o[j][1] *= a0;
        if (ROWS16) {
          o[j][2] *= a1;
          o[j][3] *= a1;
        }
      }
      m0 = mn0;
      if (ROWS16) m1 = mn1;
    }
    uint32_t pa[4];
    {
      float pr[2][4];
#pragma unroll
      for (int j = 0; j < 2; ++j) {
        pr[j][0] = exp2f(sacc[j][0] - m0);
        pr[j][1] = exp2f(sacc[j][1] - m0);
        pr[j][2] = ROWS16 ? exp2f(sacc[j][2] - m1) : 0.f;
        pr[j][3] = ROWS16 ? exp2f(sacc[j][3] - m1) : 0.f;
        l0 += pr[j][0] + pr[j][1];
        if (ROWS16) l1 += pr[j][2] + pr[j][3];
      }
      pa[0] = pack_f16(pr[0][0], pr[0][1]);
      pa[1] = pack_f16(pr[0][2], pr[0][3]);
      pa[2] = pack_f16(pr[1][0], pr[1][1]);
      pa[3] = pack_f16(pr[1][2], pr[1][3]);
    }
    // ---- O += P V: n-tile j, column n <-> dimension 16 n + j ----------------------
    {
      const uint4 va = *reinterpret_cast<const uint4*>(vb + swz(2 * tig, gid));
      const uint4 vv = *reinterpret_cast<const uint4*>(vb + swz(2 * tig + 1, gid));
      const uint4 vc = *reinterpret_cast<const uint4*>(vb + swz(2 * tig + 8, gid));
      const uint4 vd = *reinterpret_cast<const uint4*>(vb + swz(2 * tig + 9, gid));
      const uint32_t A[4] = {va.x, va.y, va.z, va.w}, B[4] = {vv.x, vv.y, vv.z, vv.w};
      const uint32_t Cw[4] = {vc.x, vc.y, vc.z, vc.w}, Dw[4] = {vd.x, vd.y, vd.z, vd.w};
#pragma unroll
      for (int w = 0; w < 4; ++w) {
        const uint32_t lo01 = __byte_perm(A[w], B[w], 0x5140);   // tokens 2tig,2tig+1: bytes 0,1
        const uint32_t hi01 = __byte_perm(A[w], B[w], 0x7362);   //                     bytes 2,3
        const uint32_t lo89 = __byte_perm(Cw[w], Dw[w], 0x5140);  // tokens 2tig+8,+9
        const uint32_t hi89 = __byte_perm(Cw[w], Dw[w], 0x7362);
        mma_f16(o[4 * w + 0], pa, e4m3x2_to_f16x2(lo01), e4m3x2_to_f16x2(lo89));
        mma_f16(o[4 * w + 1], pa, e4m3x2_to_f16x2(lo01 >> 16), e4m3x2_to_f16x2(lo89 >> 16));
        mma_f16(o[4 * w + 2], pa, e4m3x2_to_f16x2(hi01), e4m3x2_to_f16x2(hi89));
        mma_f16(o[4 * w + 3], pa, e4m3x2_to_f16x2(hi01 >> 16), e4m3x2_to_f16x2(hi89 >> 16));
      }
    }
    fence_proxy_async();
    __syncwarp();
  }

  l0 += __shfl_xor_sync(0xffffffffu, l0, 1);
  l0 += __shfl_xor_sync(0xffffffffu, l0, 2);
  if (ROWS16) {
    l1 += __shfl_xor_sync(0xffffffffu, l1, 1);
    l1 += __shfl_xor_sync(0xffffffffu, l1, 2);
  }
  if (!alive) {
    m0 = m1 = -CUDART_INF_F;
    l0 = l1 = 0.f;
  }
  __syncwarp();
  float* wres = reinterpret_cast<float*>(ring);   // [16][D] acc, then m[16], l[16]
#pragma unroll
  for (int rh = 0; rh < (ROWS16 ? 2 : 1); ++rh) {
    const int h = gid + 8 * rh;
    if (h < G) {
#pragma unroll
      for (int j = 0; j < NT; ++j) {
        wres[h * D + 16 * (2 * tig) + j] = alive ? o[j][2 * rh] : 0.f;
        wres[h * D + 16 * (2 * tig + 1) + j] = alive ? o[j][2 * rh + 1] : 0.f;
      }
      if (tig == 0) {
        wres[16 * D + h] = rh ? m1 : m0;
        wres[16 * D + 16 + h] = rh ? l1 : l0;
      }
    }
  }
  __syncthreads();

  const float vsc = __ldg(p.v_scale + g);
  const bool single = nparts == 1;
  for (int i = threadIdx.x; i < G * D; i += NW * 32) {
    const int h = i / D, d = i % D;
    float M = -CUDART_INF_F;
#pragma unroll
    for (int w = 0; w < NW; ++w)
      M = fmaxf(M, reinterpret_cast<const float*>(smem + w * SM::kWarpBytes)[16 * D + h]);
    float L = 0.f, O = 0.f;
#pragma unroll
    for (int w = 0; w < NW; ++w) {
      const float* r = reinterpret_cast<const float*>(smem + w * SM::kWarpBytes);
      const float c = exp2f(r[16 * D + h] - M);
      L = fmaf(r[16 * D + 16 + h], c, L);
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

}  // namespace pkv
