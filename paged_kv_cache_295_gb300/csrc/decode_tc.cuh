// PagedAttention decode on the 5th-generation tensor cores (tcgen05 + TMEM),
// 16-bit caches, head_dim 128.
//
// Work split: one CTA (one warp) per sequence x KV head x split-KV partition,
// walking the partition in 64-token tiles that arrive by TMA through the
// block table ("nano-vLLM architecture" section 4.2: attention addressed
// through the logical -> physical block mapping).  Two CTAs share an SM.
//
// Per tile (heads as the MMA's M dimension, "LLM inference tutorial" section
// 4.4 GQA: the G query heads of a KV head share every K/V byte):
//   S[h][t]  = sum_d Q[h][d] K[t][d]        tcgen05.mma M=128 N=64  K=128
//              A = Q rows in smem (K-major), B = the K tile (K-major, TMA layout),
//              accumulator in TMEM (lane h, column t).
//   softmax  : lane h of the warp reads its row of S (64 values), scales by
//              scale*log2(e), masks tokens past the context, and keeps a
//              running max / sum (base 2).  The running max only moves when a
//              tile's max exceeds it by more than 2^8, so O is rarely rescaled
//              (the final division by the sum uses the same max, so the result
//              is unchanged).  P = 2^(s - m) is written to smem as bf16 hi + lo
//              parts (~2^-17 relative).
//   O[h][d] += sum_t P[h][t] V[t][d]        tcgen05.mma M=128 N=128 K=64 (x2: hi, lo)
//              A = P (K-major), B = the V tile as stored (MN-major),
//              accumulator in TMEM (lane h, column d), kept across tiles.
// Only rows h < G are real; rows G..127 of A read other shared memory and
// produce ignored accumulator rows.
//
// Overlap: QK of tile i+1 is issued before the softmax of tile i; the TMA ring
// keeps STAGES tiles in flight; PV(i-1) is waited on only when its P buffer and
// stage are needed again.  Every mbarrier wait is bounded (2 s) and reports
// PKV_DEV_TIMEOUT; TMEM is always released before the CTA exits.
#pragma once

#include <cuda.h>

#include "decode_mma.cuh"

namespace pkv {

constexpr int kTcTile = 64;   // tokens per tile (MMA N of QK, K of PV)
constexpr int kTcD = 128;

struct TcLayout {
  // [Q hi 4K][Q lo 4K][P hi 2K][P lo 2K][stages ...][table]; 1024-aligned blocks
  static constexpr int kQ = 0, kQlo = 4096, kP = 8192, kPlo = 10240, kStages = 12288;
  static constexpr int kHalf = kTcTile * 128;          // [64 rows][128 B] = 8 KB
  static constexpr int kStage = 4 * kHalf;              // K (2 halves) + V (2 halves)
  static size_t bytes(int stages, int table_entries) {
    return 1024 + kStages + static_cast<size_t>(stages) * kStage +
           static_cast<size_t>(table_entries) * 4;
  }
};

__device__ __forceinline__ uint64_t tc_desc(uint32_t saddr, uint32_t lbo, uint32_t sbo) {
  uint64_t d = static_cast<uint64_t>((saddr >> 4) & 0x3FFFu);
  d |= static_cast<uint64_t>((lbo >> 4) & 0x3FFFu) << 16;
  d |= static_cast<uint64_t>((sbo >> 4) & 0x3FFFu) << 32;
  d |= static_cast<uint64_t>(1) << 46;   // descriptor version (sm_100 family)
  d |= static_cast<uint64_t>(2) << 61;   // 128-byte swizzle
  return d;
}

// kind::f16 instruction descriptor: f32 accumulate, A/B bf16 or f16, majors, N, M.
__host__ __device__ constexpr uint32_t tc_idesc(int M, int N, bool a_mn, bool b_mn, bool bf16) {
  return (1u << 4) | ((bf16 ? 1u : 0u) << 7) | ((bf16 ? 1u : 0u) << 10) |
         ((a_mn ? 1u : 0u) << 15) | ((b_mn ? 1u : 0u) << 16) |
         (static_cast<uint32_t>(N >> 3) << 17) | (static_cast<uint32_t>(M >> 4) << 24);
}

__device__ __forceinline__ void tc_mma(uint32_t d, uint64_t a, uint64_t b, uint32_t idesc,
                                       uint32_t accumulate) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
      " tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}\n" ::"r"(d),
      "l"(a), "l"(b), "r"(idesc), "r"(accumulate)
      : "memory");
}

__device__ __forceinline__ void tc_commit(uint32_t bar) {
  asm volatile(
      "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];\n" ::"r"(bar)
      : "memory");
}

__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;\n" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;\n" ::: "memory");
}

// 32 consecutive TMEM columns of this warp's 32 lanes -> 32 registers.
__device__ __forceinline__ void tc_ld32(uint32_t taddr, float* v) {
  uint32_t r[32];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,"
      "%15,%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];\n"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
        "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]),
        "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]),
        "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr));
  asm volatile("tcgen05.wait::ld.sync.aligned;\n" ::: "memory");
#pragma unroll
  for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(r[i]);
}

__device__ __forceinline__ void tc_st32(uint32_t taddr, const float* v) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,"
      "%14,%15,%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};\n" ::"r"(taddr),
      "r"(__float_as_uint(v[0])), "r"(__float_as_uint(v[1])), "r"(__float_as_uint(v[2])),
      "r"(__float_as_uint(v[3])), "r"(__float_as_uint(v[4])), "r"(__float_as_uint(v[5])),
      "r"(__float_as_uint(v[6])), "r"(__float_as_uint(v[7])), "r"(__float_as_uint(v[8])),
      "r"(__float_as_uint(v[9])), "r"(__float_as_uint(v[10])), "r"(__float_as_uint(v[11])),
      "r"(__float_as_uint(v[12])), "r"(__float_as_uint(v[13])), "r"(__float_as_uint(v[14])),
      "r"(__float_as_uint(v[15])), "r"(__float_as_uint(v[16])), "r"(__float_as_uint(v[17])),
      "r"(__float_as_uint(v[18])), "r"(__float_as_uint(v[19])), "r"(__float_as_uint(v[20])),
      "r"(__float_as_uint(v[21])), "r"(__float_as_uint(v[22])), "r"(__float_as_uint(v[23])),
      "r"(__float_as_uint(v[24])), "r"(__float_as_uint(v[25])), "r"(__float_as_uint(v[26])),
      "r"(__float_as_uint(v[27])), "r"(__float_as_uint(v[28])), "r"(__float_as_uint(v[29])),
      "r"(__float_as_uint(v[30])), "r"(__float_as_uint(v[31]))
      : "memory");
  asm volatile("tcgen05.wait::st.sync.aligned;\n" ::: "memory");
}

}  // namespace pkv

namespace pkv {

template <bool QF32, int STAGES>
__global__ void __launch_bounds__(32)
    paged_decode_tc_kernel(const __grid_constant__ CUtensorMap tmap_k,
                           const __grid_constant__ CUtensorMap tmap_v, const MmaParams mp) {
  using LY = TcLayout;
  const DecodeParams& p = mp.p;
  const int G = p.num_q_heads / p.num_kv_heads;

  extern __shared__ uint8_t smem_raw[];
  __shared__ __align__(8) uint64_t full[STAGES];
  __shared__ __align__(8) uint64_t bar_s[2];
  __shared__ __align__(8) uint64_t bar_o;
  __shared__ uint32_t tmem_base_sh;
  uint8_t* sm = smem_raw + ((1024 - (smem_u32(smem_raw) & 1023)) & 1023);
  const uint32_t sma = smem_u32(sm);

  const int s = blockIdx.z, g = blockIdx.y, part = blockIdx.x;
  const int lane = threadIdx.x;
  const int P = p.partition_tokens;

  int ctx = __ldg(p.context_lens + s);
  const int cap = context_cap(p);
  if (ctx < 0 || ctx > cap) {
    if (part == 0 && lane == 0) flag_status(p.status, PKV_DEV_BAD_CONTEXT);
    ctx = ctx < 0 ? 0 : cap;
  }
  const int nparts = (ctx + P - 1) / P;
  if (part >= (nparts > 0 ? nparts : 1)) return;
  const int hq0 = g * G;
  if (ctx == 0) {
    for (int i = lane; i < G * kTcD; i += 32)
      p.out[(static_cast<int64_t>(s) * p.num_q_heads + hq0) * kTcD + i] = 0.f;
    return;
  }
  const int t_begin = part * P;
  const int t_end = min(t_begin + P, ctx);

  // block-table entries of the partition
  int32_t* sbt = reinterpret_cast<int32_t*>(sm + LY::kStages + STAGES * LY::kStage);
  const int lb0 = t_begin >> p.bs_log2;
  const int nlb = ((t_end - 1) >> p.bs_log2) - lb0 + 1;
  const int32_t* bt_row = p.block_tables + static_cast<int64_t>(s) * p.max_blocks_per_seq;
  for (int i = lane; i < nlb; i += 32) {
    int32_t b = __ldg(bt_row + lb0 + i);
    if (b < 0 || b >= p.num_blocks) {
      flag_status(p.status, PKV_DEV_BAD_BLOCK);
      b = -1;
    }
    sbt[i] = b;
  }
  // query rows (A operand of QK): 16 rows x 128 dims, bf16 hi (+ lo for float32 q)
  {
    const int64_t row0 = static_cast<int64_t>(s) * p.num_q_heads + hq0;
    for (int i = lane; i < 16 * 16; i += 32) {
      const int h = i >> 4, u = i & 15, hh = u >> 3, uu = u & 7;
      uint4 hi = make_uint4(0, 0, 0, 0), lo = make_uint4(0, 0, 0, 0);
      if (h < G) {
        if (QF32) {
          const float4* qf = reinterpret_cast<const float4*>(static_cast<const float*>(p.q) +
                                                             (row0 + h) * kTcD + 8 * u);
          const float4 a = qf[0], b = qf[1];
          const float x[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
          uint32_t wh[4], wl[4];
#pragma unroll
          for (int k = 0; k < 4; ++k) {
            wh[k] = pack_bf16(x[2 * k], x[2 * k + 1]);
            const __nv_bfloat162 hv = *reinterpret_cast<const __nv_bfloat162*>(&wh[k]);
            wl[k] = pack_bf16(x[2 * k] - __low2float(hv), x[2 * k + 1] - __high2float(hv));
          }
          hi = make_uint4(wh[0], wh[1], wh[2], wh[3]);
          lo = make_uint4(wl[0], wl[1], wl[2], wl[3]);
        } else {
          hi = *reinterpret_cast<const uint4*>(static_cast<const __nv_bfloat16*>(p.q) +
                                               (row0 + h) * kTcD + 8 * u);
        }
      }
      *reinterpret_cast<uint4*>(sm + LY::kQ + hh * 2048 + swz(h, uu)) = hi;
      if (QF32) *reinterpret_cast<uint4*>(sm + LY::kQlo + hh * 2048 + swz(h, uu)) = lo;
    }
  }
  if (lane == 0) {
    for (int st = 0; st < STAGES; ++st) mbar_init(smem_u32(&full[st]), 1);
    mbar_init(smem_u32(&bar_s[0]), 1);
    mbar_init(smem_u32(&bar_s[1]), 1);
    mbar_init(smem_u32(&bar_o), 1);
    asm volatile("fence.mbarrier_init.release.cluster;\n" ::: "memory");
  }
  __syncwarp();
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], 256;\n" ::"r"(
                   smem_u32(&tmem_base_sh))
               : "memory");
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;\n" ::: "memory");
  fence_proxy_async();
  tc_fence_before();
  __syncwarp();
  tc_fence_after();
  const uint32_t tm = tmem_base_sh;        // S buffers at +0 / +64, O at +128
  const uint32_t tmO = tm + 128;

  const int ntiles = (t_end - t_begin + kTcTile - 1) / kTcTile;
  const int box_rows = mp.box_rows;
  const int nbox = kTcTile / box_rows;
  const uint32_t idesc_qk = tc_idesc(128, kTcTile, false, false, true);
  const uint32_t idesc_pv = tc_idesc(128, kTcD, false, true, true);

  // Rows of tile j that hold cache data (inside the context, valid block id).
  auto filled_rows = [&](int j) -> uint64_t {
    const int t0 = t_begin + j * kTcTile;
    uint64_t mask = 0;
    for (int bx = 0; bx < nbox; ++bx) {
      const int tb = t0 + bx * box_rows;
      if (tb >= ctx) break;
      if (sbt[(tb >> p.bs_log2) - lb0] < 0) continue;
      const int rows = min(box_rows, ctx - tb);
      const uint64_t bits = rows >= 64 ? ~0ull : ((1ull << rows) - 1);
      mask |= bits << (bx * box_rows);
    }
    return mask;
  };
  auto issue_tma = [&](int j) {   // lane 0
    const int stage = j % STAGES;
    const int t0 = t_begin + j * kTcTile;
    const uint32_t bar = smem_u32(&full[stage]);
    uint32_t bytes = 0;
    for (int bx = 0; bx < nbox; ++bx) {
      const int tb = t0 + bx * box_rows;
      if (tb >= ctx) break;
      if (sbt[(tb >> p.bs_log2) - lb0] >= 0) bytes += 4 * box_rows * 128;
    }
    mbar_arrive_expect_tx(bar, bytes);
    const uint32_t sbase = sma + LY::kStages + stage * LY::kStage;
    for (int bx = 0; bx < nbox; ++bx) {
      const int tb = t0 + bx * box_rows;
      if (tb >= ctx) break;
      const int32_t b = sbt[(tb >> p.bs_log2) - lb0];
      if (b < 0) continue;
      const int z = (b << p.bs_log2) + (tb & ((1 << p.bs_log2) - 1));
#pragma unroll
      for (int hh = 0; hh < 2; ++hh) {
        const uint32_t off = hh * LY::kHalf + bx * box_rows * 128;
        tma_load_3d(sbase + off, &tmap_k, hh * 64, g, z, bar);
        tma_load_3d(sbase + 2 * LY::kHalf + off, &tmap_v, hh * 64, g, z, bar);
      }
    }
  };
  auto issue_qk = [&](int j) {    // lane 0, tile j landed
    const uint32_t kb = sma + LY::kStages + (j % STAGES) * LY::kStage;
    const uint32_t dst = tm + (j & 1) * kTcTile;
#pragma unroll
    for (int ks = 0; ks < kTcD / 16; ++ks) {
      const uint32_t koff = (ks >> 2) * LY::kHalf + (ks & 3) * 32;
      const uint32_t qoff = (ks >> 2) * 2048 + (ks & 3) * 32;
      const uint64_t bdesc = tc_desc(kb + koff, 0, 1024);
      tc_mma(dst, tc_desc(sma + LY::kQ + qoff, 0, 1024), bdesc, idesc_qk, ks > 0);
      if (QF32) tc_mma(dst, tc_desc(sma + LY::kQlo + qoff, 0, 1024), bdesc, idesc_qk, 1);
    }
    tc_commit(smem_u32(&bar_s[j & 1]));
  };

  if (lane == 0)
    for (int j = 0; j < min(STAGES, ntiles); ++j) issue_tma(j);
  bool alive = true;
  {
    bool ok = true;
    if (lane == 0) {
      ok = mbar_wait(smem_u32(&full[0]), 0);
      if (ok) issue_qk(0);
    }
    alive = __shfl_sync(0xffffffffu, ok, 0);
  }
  int qk_issued = 1, pv_issued = 0;   // for the bounded drain after a timeout

  float m = -CUDART_INF_F, l = 0.f;
  const bool row_real = lane < G;
  const float sl2 = p.qk_scale_log2;
  for (int i = 0; i < ntiles && alive; ++i) {
    // (a) logits of tile i
    if (!__all_sync(0xffffffffu, mbar_wait(smem_u32(&bar_s[i & 1]), (i >> 1) & 1))) {
      alive = false;
      break;
    }
    tc_fence_after();
    float sv[kTcTile];
    tc_ld32(tm + (i & 1) * kTcTile, sv);
    tc_ld32(tm + (i & 1) * kTcTile + 32, sv + 32);
    tc_fence_before();
    __syncwarp();
    // (b) QK of tile i+1 overlaps this tile's softmax
    if (i + 1 < ntiles) {
      bool ok = true;
      if (lane == 0) {
        tc_fence_after();
        ok = mbar_wait(smem_u32(&full[(i + 1) % STAGES]), ((i + 1) / STAGES) & 1);
        if (ok) issue_qk(i + 1);
      }
      if (!__shfl_sync(0xffffffffu, ok, 0)) {
        alive = false;
        break;
      }
      ++qk_issued;
    }
    // (c) softmax of tile i (row = lane)
    const uint64_t fmask = filled_rows(i);
    float mt = -CUDART_INF_F;
#pragma unroll
    for (int t = 0; t < kTcTile; ++t) {
      sv[t] = ((fmask >> t) & 1) ? sv[t] * sl2 : -CUDART_INF_F;
      mt = fmaxf(mt, sv[t]);
    }
    bool resc = false;
    float alpha = 1.f;
    if (row_real && mt > m + 8.f) {
      if (m != -CUDART_INF_F) {
        alpha = exp2f(m - mt);
        resc = true;
      }
      m = mt;
      l *= alpha;
    }
    const float mref = row_real ? m : 0.f;
    float lsum = 0.f;
#pragma unroll
    for (int t = 0; t < kTcTile; ++t) {
      sv[t] = exp2f(sv[t] - mref);
      lsum += sv[t];
    }
    if (row_real) l += lsum;
    // (d) PV(i-1) done: its P buffer, O and its stage are free again
    if (i > 0) {
      if (!__all_sync(0xffffffffu, mbar_wait(smem_u32(&bar_o), (i - 1) & 1))) {
        alive = false;
        break;
      }
      tc_fence_after();
      if (lane == 0 && i - 1 + STAGES < ntiles) issue_tma(i - 1 + STAGES);
    }
    // (e) rare rescale of the O rows whose max moved
    if (__any_sync(0xffffffffu, resc)) {
#pragma unroll
      for (int c = 0; c < kTcD; c += 32) {
        float ov[32];
        tc_ld32(tmO + c, ov);
#pragma unroll
        for (int k = 0; k < 32; ++k) ov[k] *= alpha;
        tc_st32(tmO + c, ov);
      }
    }
    // (f) P of tile i into smem (rows < 16), zero V rows that hold no cache data
    if (lane < 16) {
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        uint32_t wh[4], wl[4];
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          const float x0 = sv[8 * u + 2 * k], x1 = sv[8 * u + 2 * k + 1];
          wh[k] = pack_bf16(x0, x1);
          const __nv_bfloat162 hv = *reinterpret_cast<const __nv_bfloat162*>(&wh[k]);
          wl[k] = pack_bf16(x0 - __low2float(hv), x1 - __high2float(hv));
        }
        *reinterpret_cast<uint4*>(sm + LY::kP + swz(lane, u)) = make_uint4(wh[0], wh[1], wh[2], wh[3]);
        *reinterpret_cast<uint4*>(sm + LY::kPlo + swz(lane, u)) = make_uint4(wl[0], wl[1], wl[2], wl[3]);
      }
    }
    if (fmask != ~0ull) {
      if (!__all_sync(0xffffffffu, mbar_wait(smem_u32(&full[i % STAGES]), (i / STAGES) & 1))) {
        alive = false;
        break;
      }
      uint8_t* vbase = sm + LY::kStages + (i % STAGES) * LY::kStage + 2 * LY::kHalf;
      for (int k = lane; k < kTcTile * 16; k += 32) {
        const int r = k >> 4, hh = (k >> 3) & 1;
        if (!((fmask >> r) & 1))
          *reinterpret_cast<uint4*>(vbase + hh * LY::kHalf + r * 128 + ((k & 7) << 4)) =
              make_uint4(0, 0, 0, 0);
      }
    }
    fence_proxy_async();
    tc_fence_before();
    __syncwarp();
    // (g) O += P V
    if (lane == 0) {
      tc_fence_after();
      const uint32_t vb = sma + LY::kStages + (i % STAGES) * LY::kStage + 2 * LY::kHalf;
#pragma unroll
      for (int kk = 0; kk < kTcTile / 16; ++kk) {
        const uint64_t bdesc = tc_desc(vb + kk * 2048, LY::kHalf, 1024);
        tc_mma(tmO, tc_desc(sma + LY::kP + kk * 32, 0, 1024), bdesc, idesc_pv, (i > 0 || kk > 0));
        tc_mma(tmO, tc_desc(sma + LY::kPlo + kk * 32, 0, 1024), bdesc, idesc_pv, 1);
      }
      tc_commit(smem_u32(&bar_o));
    }
    ++pv_issued;
    __syncwarp();
  }

  float res[kTcD];
  bool have = false;
  if (alive && pv_issued > 0) {
    have = __all_sync(0xffffffffu, mbar_wait(smem_u32(&bar_o), (pv_issued - 1) & 1));
    if (have) {
      tc_fence_after();
#pragma unroll
      for (int c = 0; c < kTcD; c += 32) tc_ld32(tmO + c, res + c);
    }
  }
  if (!alive || !have) {
    if (lane == 0) flag_status(p.status, PKV_DEV_TIMEOUT);
    // bounded drain of the last issued tensor-core work before TMEM is released
    if (pv_issued > 0) mbar_wait(smem_u32(&bar_o), (pv_issued - 1) & 1);
    if (qk_issued > 0) mbar_wait(smem_u32(&bar_s[(qk_issued - 1) & 1]), ((qk_issued - 1) >> 1) & 1);
  }
  tc_fence_before();
  __syncwarp();
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, 256;\n" ::"r"(tm) : "memory");

  if (!row_real) return;
  const int64_t sh = static_cast<int64_t>(s) * p.num_q_heads + hq0 + lane;
  const bool ok_out = alive && have;
  if (nparts == 1) {
    const float inv = ok_out ? 1.f / l : 0.f;
    for (int d = 0; d < kTcD; ++d) p.out[sh * kTcD + d] = ok_out ? res[d] * inv : 0.f;
  } else {
    const int64_t pi = sh * p.max_parts + part;
    for (int d = 0; d < kTcD; ++d) p.part_o[pi * kTcD + d] = ok_out ? res[d] : 0.f;
    p.part_ml[pi * 2 + 0] = ok_out ? m : -CUDART_INF_F;
    p.part_ml[pi * 2 + 1] = ok_out ? l : 0.f;
  }
}

}  // namespace pkv
