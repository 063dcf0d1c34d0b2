// PagedAttention decode on the 5th-generation tensor cores (tcgen05 + TMEM),
// 16-bit caches, head_dim 128.
//
// Work split: one CTA per sequence x KV head x split-KV partition, walking the
// partition in 64-token tiles that arrive by TMA through the block table
// ("nano-vLLM architecture" section 4.2: attention addressed through the
// logical -> physical block mapping).  Two CTAs share an SM.  Warp roles:
// warps 0-3 softmax and epilogue (one TMEM lane quarter each), warp 4 TMA
// producer (its lanes issue a tile's boxes in parallel), warp 5 MMA issuer.
// The roles talk only through mbarriers, so the issue latencies of TMA and
// tcgen05.mma overlap each other and the softmax.
//
// Per tile, tokens are the MMA rows and the G query heads of the KV head the
// columns ("LLM inference tutorial" section 4.4 GQA: the G heads share every
// K/V byte, read once):
//   S^T[t][h] = sum_d K[t][d] Q[h][d]         tcgen05.mma M=64  N=16 K=128
//               A = the K tile as stored (K-major), B = Q (K-major, 16 rows),
//               accumulator in TMEM: token t in lane 32*(t/16) + t%16.
//   softmax   : the thread of token t scales its G logits by scale*log2(e),
//               masks it if outside the context, and the CTA takes each
//               head's tile max (warp shuffles + one shared exchange).  The
//               running max only moves when a tile max exceeds it by more than
//               2^8, so O is rarely rescaled (the final division by the sum
//               uses the same max, so the result is unchanged).  P = 2^(s - m)
//               goes to smem transposed, as bf16 hi + lo parts (~2^-17).
//   O^T[d][h] += sum_t V[t][d] P[h][t]         tcgen05.mma M=128 N=16 K=64 (x2: hi, lo)
//               A = the V tile as stored (MN-major), B = P^T (K-major),
//               accumulator in TMEM: dimension d in lane d, kept across tiles.
//
// Pipeline per tile j: producer loads stage j%STAGES once PV(j-STAGES) has
// released it; the MMA warp issues QK(j) when the tile has landed and the S
// buffer j%2 has been read, then PV(j-1) when its P^T is written; softmax warps
// read S(j), write P^T(j) into buffer j%2 (after PV(j-2) finished with it).
// Every mbarrier wait is bounded (2 s) and also stops when another role has
// given up (shared abort flag); a give-up reports PKV_DEV_TIMEOUT.  TMEM is
// always released before the CTA exits.
#pragma once

#include <cuda.h>

#include "decode_mma.cuh"

namespace pkv {

constexpr int kTcTile = 64;   // tokens per tile (MMA M of QK, K of PV)
constexpr int kTcD = 128;

struct TcLayout {
  // [Q hi 4K][Q lo 4K][P^T buffer 0: hi 2K, lo 2K][buffer 1][stages ...][table].
  // Q: [16 heads][128 d] as two [16][128 B] halves; P^T: [16 heads][64 tokens].
  static constexpr int kQ = 0, kQlo = 4096, kP = 8192, kPBuf = 4096, kPlo = 2048,
                       kStages = 16384;
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

// The same with the A operand in TMEM (row = lane; column c holds elements 2c
// and 2c+1 of the row, so a 16-element k-step is 8 columns); B from shared memory.
__device__ __forceinline__ void tc_mma_ts(uint32_t d, uint32_t a_tmem, uint64_t b, uint32_t idesc,
                                          uint32_t accumulate) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
      " tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n}\n" ::"r"(d),
      "r"(a_tmem), "l"(b), "r"(idesc), "r"(accumulate)
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

// 16 consecutive TMEM columns of this warp's 32 lanes -> 16 registers.
__device__ __forceinline__ void tc_ld16(uint32_t taddr, float* v) {
  uint32_t r[16];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,"
      "%15}, [%16];\n"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
        "=r"(r[14]), "=r"(r[15])
      : "r"(taddr));
  asm volatile("tcgen05.wait::ld.sync.aligned;\n" ::: "memory");
#pragma unroll
  for (int i = 0; i < 16; ++i) v[i] = __uint_as_float(r[i]);
}

__device__ __forceinline__ void tc_st16(uint32_t taddr, const float* v) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,"
      "%14,%15,%16};\n" ::"r"(taddr),
      "r"(__float_as_uint(v[0])), "r"(__float_as_uint(v[1])), "r"(__float_as_uint(v[2])),
      "r"(__float_as_uint(v[3])), "r"(__float_as_uint(v[4])), "r"(__float_as_uint(v[5])),
      "r"(__float_as_uint(v[6])), "r"(__float_as_uint(v[7])), "r"(__float_as_uint(v[8])),
      "r"(__float_as_uint(v[9])), "r"(__float_as_uint(v[10])), "r"(__float_as_uint(v[11])),
      "r"(__float_as_uint(v[12])), "r"(__float_as_uint(v[13])), "r"(__float_as_uint(v[14])),
      "r"(__float_as_uint(v[15]))
      : "memory");
  asm volatile("tcgen05.wait::st.sync.aligned;\n" ::: "memory");
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

constexpr int kTcThreads = 192;   // warps 0-3 softmax, 4 producer, 5 MMA

// Bounded wait that also gives up once any role of the CTA has given up.
__device__ __forceinline__ bool tc_wait(uint32_t bar, uint32_t parity, volatile int* abort_flag) {
  uint32_t ok = 0;
  const uint64_t t0 = global_ns();
  while (true) {
    asm volatile(
        "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n"
        " selp.u32 %0, 1, 0, p;\n}\n"
        : "=r"(ok)
        : "r"(bar), "r"(parity)
        : "memory");
    if (ok) return true;
    if (*abort_flag) return false;
    if (global_ns() - t0 > kWaitLimitNs) {
      *abort_flag = 1;
      return false;
    }
  }
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];\n" ::"r"(bar) : "memory");
}

// Barrier of the 4 softmax warps (named barrier 1) that also ANDs a flag, so
// every softmax warp takes the same loop exit.
__device__ __forceinline__ bool softmax_bar_all(bool v) {
  uint32_t r;
  asm volatile(
      "{\n .reg .pred p, q;\n setp.ne.u32 q, %1, 0;\n bar.red.and.pred p, 1, 128, q;\n"
      " selp.u32 %0, 1, 0, p;\n}\n"
      : "=r"(r)
      : "r"(static_cast<uint32_t>(v))
      : "memory");
  return r != 0;
}

template <bool QF32, int STAGES>
__global__ void __launch_bounds__(kTcThreads)
    paged_decode_tc_kernel(const __grid_constant__ CUtensorMap tmap_k,
                           const __grid_constant__ CUtensorMap tmap_v, const MmaParams mp) {
  using LY = TcLayout;
  constexpr int GMAX = 16;
  const DecodeParams& p = mp.p;
  const int G = p.num_q_heads / p.num_kv_heads;

  extern __shared__ uint8_t smem_raw[];
  __shared__ __align__(8) uint64_t full[STAGES], empty[STAGES];
  __shared__ __align__(8) uint64_t s_full[2], s_free[2], p_full[2], o_done[2];
  __shared__ uint32_t tmem_base_sh;
  __shared__ float red[2][4][GMAX];
  __shared__ float lred[4][GMAX];
  __shared__ int abort_sh;
  uint8_t* sm = smem_raw + ((1024 - (smem_u32(smem_raw) & 1023)) & 1023);
  const uint32_t sma = smem_u32(sm);
  volatile int* abort_flag = &abort_sh;

  const int s = blockIdx.z, g = blockIdx.x, part = blockIdx.y;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int P = p.partition_tokens;

  int ctx = __ldg(p.context_lens + s);
  const int cap = context_cap(p);
  if (ctx < 0 || ctx > cap) {
    if (part == 0 && tid == 0) flag_status(p.status, PKV_DEV_BAD_CONTEXT);
    ctx = ctx < 0 ? 0 : cap;
  }
  const int nparts = (ctx + P - 1) / P;
  if (part >= (nparts > 0 ? nparts : 1)) return;
  const int hq0 = g * G;
  if (ctx == 0) {
    for (int i = tid; i < G * kTcD; i += kTcThreads)
      p.out[(static_cast<int64_t>(s) * p.num_q_heads + hq0) * kTcD + i] = 0.f;
    return;
  }
  const int t_begin = part * P;
  const int t_end = min(t_begin + P, ctx);

  int32_t* sbt = reinterpret_cast<int32_t*>(sm + LY::kStages + STAGES * LY::kStage);
  const int lb0 = t_begin >> p.bs_log2;
  const int nlb = ((t_end - 1) >> p.bs_log2) - lb0 + 1;
  const int32_t* bt_row = p.block_tables + static_cast<int64_t>(s) * p.max_blocks_per_seq;
  for (int i = tid; i < nlb; i += kTcThreads) {
    int32_t b = __ldg(bt_row + lb0 + i);
    if (b < 0 || b >= p.num_blocks) {
      flag_status(p.status, PKV_DEV_BAD_BLOCK);
      b = -1;
    }
    sbt[i] = b;
  }
  // Q (B operand of QK): 16 rows x 128 dims, bf16 hi (+ lo for float32 q); P^T zeroed
  {
    const int64_t row0 = static_cast<int64_t>(s) * p.num_q_heads + hq0;
    for (int i = tid; i < GMAX * 16; i += kTcThreads) {
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
      // P^T buffers (hi, lo of both): rows >= G stay zero for the whole CTA
      *reinterpret_cast<uint4*>(sm + LY::kP + hh * LY::kPBuf + swz(h, uu)) = make_uint4(0, 0, 0, 0);
      *reinterpret_cast<uint4*>(sm + LY::kP + hh * LY::kPBuf + LY::kPlo + swz(h, uu)) =
          make_uint4(0, 0, 0, 0);
    }
  }
  if (tid == 0) {
    for (int st = 0; st < STAGES; ++st) {
      mbar_init(smem_u32(&full[st]), 1);
      mbar_init(smem_u32(&empty[st]), 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(smem_u32(&s_full[b]), 1);
      mbar_init(smem_u32(&s_free[b]), 4);
      mbar_init(smem_u32(&p_full[b]), 4);
      mbar_init(smem_u32(&o_done[b]), 1);
    }
    abort_sh = 0;
    asm volatile("fence.mbarrier_init.release.cluster;\n" ::: "memory");
  }
  if (warp == 0) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], 64;\n" ::"r"(
                     smem_u32(&tmem_base_sh))
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;\n" ::: "memory");
  }
  fence_proxy_async();
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tm = tmem_base_sh;          // S^T buffers at columns 0 / 16, O^T at 32
  const uint32_t tmO = tm + 32;
  const int ntiles = (t_end - t_begin + kTcTile - 1) / kTcTile;
  const int box_rows = mp.box_rows;
  const int nbox = kTcTile / box_rows;
  int have_out = 0;
  float ov[GMAX];
  float m[GMAX];

  if (warp == 4) {
    // ------------------------------ TMA producer ------------------------------
    for (int j = 0; j < ntiles; ++j) {
      const int st = j % STAGES;
      if (j >= STAGES) {
        bool ok = true;
        if (lane == 0) ok = tc_wait(smem_u32(&empty[st]), ((j / STAGES) - 1) & 1, abort_flag);
        if (!__shfl_sync(0xffffffffu, ok, 0)) break;
      }
      const int t0 = t_begin + j * kTcTile;
      const uint32_t bar = smem_u32(&full[st]);
      if (lane == 0) {
        uint32_t bytes = 0;
        for (int bx = 0; bx < nbox; ++bx) {
          const int tb = t0 + bx * box_rows;
          if (tb < ctx && sbt[(tb >> p.bs_log2) - lb0] >= 0) bytes += 4 * box_rows * 128;
        }
        mbar_arrive_expect_tx(bar, bytes);
      }
      __syncwarp();
      const uint32_t sbase = sma + LY::kStages + st * LY::kStage;
      for (int k = lane; k < 4 * nbox; k += 32) {   // (box, K/V, half) per lane
        const int bx = k >> 2, kv = (k >> 1) & 1, hh = k & 1;
        const int tb = t0 + bx * box_rows;
        if (tb >= ctx) continue;
        const int32_t b = sbt[(tb >> p.bs_log2) - lb0];
        if (b < 0) continue;
        const int z = (b << p.bs_log2) + (tb & ((1 << p.bs_log2) - 1));
        const uint32_t off = kv * 2 * LY::kHalf + hh * LY::kHalf + bx * box_rows * 128;
        tma_load_3d(sbase + off, kv ? &tmap_v : &tmap_k, hh * 64, g, z, bar);
      }
    }
  } else if (warp == 5) {
    // ------------------------------ MMA issuer --------------------------------
    if (lane == 0) {
      const uint32_t idesc_qk = tc_idesc(kTcTile, GMAX, false, false, true);
      const uint32_t idesc_pv = tc_idesc(kTcD, GMAX, true, false, true);
      auto issue_pv = [&](int j) {
        const uint32_t vb = sma + LY::kStages + (j % STAGES) * LY::kStage + 2 * LY::kHalf;
        const uint32_t pb = sma + LY::kP + (j & 1) * LY::kPBuf;
#pragma unroll
        for (int kk = 0; kk < kTcTile / 16; ++kk) {
          const uint64_t adesc = tc_desc(vb + kk * 2048, LY::kHalf, 1024);
          tc_mma(tmO, adesc, tc_desc(pb + kk * 32, 0, 1024), idesc_pv, (j > 0 || kk > 0));
          tc_mma(tmO, adesc, tc_desc(pb + LY::kPlo + kk * 32, 0, 1024), idesc_pv, 1);
        }
        tc_commit(smem_u32(&o_done[j & 1]));
        tc_commit(smem_u32(&empty[j % STAGES]));
      };
      int issued_qk = 0, issued_pv = 0;
      for (int j = 0; j <= ntiles; ++j) {
        if (j < ntiles) {
          if (!tc_wait(smem_u32(&full[j % STAGES]), (j / STAGES) & 1, abort_flag)) break;
          if (j >= 2 && !tc_wait(smem_u32(&s_free[j & 1]), ((j - 2) >> 1) & 1, abort_flag)) break;
          tc_fence_after();
          const uint32_t kb = sma + LY::kStages + (j % STAGES) * LY::kStage;
          const uint32_t dst = tm + (j & 1) * GMAX;
#pragma unroll
          for (int ks = 0; ks < kTcD / 16; ++ks) {
            const uint32_t koff = (ks >> 2) * LY::kHalf + (ks & 3) * 32;
            const uint32_t qoff = (ks >> 2) * 2048 + (ks & 3) * 32;
            const uint64_t adesc = tc_desc(kb + koff, 0, 1024);
            tc_mma(dst, adesc, tc_desc(sma + LY::kQ + qoff, 0, 1024), idesc_qk, ks > 0);
            if (QF32) tc_mma(dst, adesc, tc_desc(sma + LY::kQlo + qoff, 0, 1024), idesc_qk, 1);
          }
          tc_commit(smem_u32(&s_full[j & 1]));
          ++issued_qk;
        }
        if (j >= 1) {
          if (!tc_wait(smem_u32(&p_full[(j - 1) & 1]), ((j - 1) >> 1) & 1, abort_flag)) break;
          tc_fence_after();
          issue_pv(j - 1);
          ++issued_pv;
        }
      }
      if (*abort_flag) {   // let issued tensor-core work finish before TMEM is released
        volatile int no_abort = 0;
        if (issued_pv > 0)
          tc_wait(smem_u32(&o_done[(issued_pv - 1) & 1]), ((issued_pv - 1) >> 1) & 1, &no_abort);
        if (issued_qk > 0)
          tc_wait(smem_u32(&s_full[(issued_qk - 1) & 1]), ((issued_qk - 1) >> 1) & 1, &no_abort);
      }
    }
  } else {
    // ------------------------- softmax warps 0-3 ------------------------------
    const uint32_t lane_q = static_cast<uint32_t>(warp * 32) << 16;
    const bool tok_lane = lane < 16;
    const int tloc = 16 * warp + lane;   // token row of the M=64 accumulator layout
    float lpart[GMAX];
#pragma unroll
    for (int h = 0; h < GMAX; ++h) {
      m[h] = -CUDART_INF_F;
      lpart[h] = 0.f;
    }
    const float sl2 = p.qk_scale_log2;
    bool alive = true;
    for (int j = 0; j < ntiles; ++j) {
      const int tb = t_begin + j * kTcTile + tloc;
      const bool filled = tok_lane && tb < ctx && sbt[(tb >> p.bs_log2) - lb0] >= 0;
      if (!tc_wait(smem_u32(&s_full[j & 1]), (j >> 1) & 1, abort_flag)) alive = false;
      tc_fence_after();
      float sv[GMAX];
      tc_ld16(tm + lane_q + (j & 1) * GMAX, sv);
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_u32(&s_free[j & 1]));
      float mx[GMAX];
#pragma unroll
      for (int h = 0; h < GMAX; ++h) {
        sv[h] = (filled && h < G) ? sv[h] * sl2 : -CUDART_INF_F;
        mx[h] = sv[h];
#pragma unroll
        for (int off = 8; off > 0; off >>= 1)
          mx[h] = fmaxf(mx[h], __shfl_xor_sync(0xffffffffu, mx[h], off));
      }
      if (lane == 0) {
#pragma unroll
        for (int h = 0; h < GMAX; ++h) red[j & 1][warp][h] = mx[h];
      }
      alive = softmax_bar_all(alive);   // also publishes red[][] to all softmax warps
      if (!alive) break;
      bool resc = false;
      float alpha[GMAX];
#pragma unroll
      for (int h = 0; h < GMAX; ++h) {
        const float mt = fmaxf(fmaxf(red[j & 1][0][h], red[j & 1][1][h]),
                               fmaxf(red[j & 1][2][h], red[j & 1][3][h]));
        alpha[h] = 1.f;
        if (h < G && mt > m[h] + 8.f) {
          if (m[h] != -CUDART_INF_F) {
            alpha[h] = exp2f(m[h] - mt);
            resc = true;
          }
          m[h] = mt;
        }
        const float pr = (h < G && filled) ? exp2f(sv[h] - m[h]) : 0.f;
        lpart[h] = lpart[h] * alpha[h] + pr;
        sv[h] = pr;
      }
      // P^T buffer j%2 is free once PV(j-2) is done; a rescale needs PV(j-1) done.
      // A failed wait only clears `alive`; the next vote ends the loop for all.
      if (j >= 2 && !tc_wait(smem_u32(&o_done[j & 1]), ((j - 2) >> 1) & 1, abort_flag))
        alive = false;
      if (resc) {   // same decision in every softmax thread
        if (!tc_wait(smem_u32(&o_done[(j - 1) & 1]), ((j - 1) >> 1) & 1, abort_flag))
          alive = false;
        tc_fence_after();
        float o[GMAX];
        tc_ld16(tmO + lane_q, o);
#pragma unroll
        for (int h = 0; h < GMAX; ++h) o[h] *= alpha[h];
        tc_st16(tmO + lane_q, o);
      }
      uint8_t* pb = sm + LY::kP + (j & 1) * LY::kPBuf;
      if (tok_lane) {
#pragma unroll
        for (int h = 0; h < GMAX; ++h) {
          if (h < G) {
            const __nv_bfloat16 hv = __float2bfloat16_rn(sv[h]);
            const __nv_bfloat16 lv = __float2bfloat16_rn(sv[h] - __bfloat162float(hv));
            const uint32_t off = h * 128 + ((((tloc >> 3) ^ (h & 7))) << 4) + (tloc & 7) * 2;
            *reinterpret_cast<__nv_bfloat16*>(pb + off) = hv;
            *reinterpret_cast<__nv_bfloat16*>(pb + LY::kPlo + off) = lv;
          }
        }
        if (!filled) {   // V rows without cache data must not reach the products
          uint8_t* vrow =
              sm + LY::kStages + (j % STAGES) * LY::kStage + 2 * LY::kHalf + tloc * 128;
#pragma unroll
          for (int u = 0; u < 8; ++u) {
            *reinterpret_cast<uint4*>(vrow + (u << 4)) = make_uint4(0, 0, 0, 0);
            *reinterpret_cast<uint4*>(vrow + LY::kHalf + (u << 4)) = make_uint4(0, 0, 0, 0);
          }
        }
      }
      fence_proxy_async();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_u32(&p_full[j & 1]));
    }
    // epilogue: O^T (lane d) and the sum l per head
    alive = softmax_bar_all(alive);
    const bool last_ok =
        alive && tc_wait(smem_u32(&o_done[(ntiles - 1) & 1]), ((ntiles - 1) >> 1) & 1, abort_flag);
    if (__all_sync(0xffffffffu, last_ok)) {   // warp-uniform: the TMEM load is warp-wide
      tc_fence_after();
      tc_ld16(tmO + lane_q, ov);
      have_out = 1;
    }
#pragma unroll
    for (int h = 0; h < GMAX; ++h) {
      float v = tok_lane ? lpart[h] : 0.f;
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) v += __shfl_xor_sync(0xffffffffu, v, off);
      if (lane == 0) lred[warp][h] = v;
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0)
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, 64;\n" ::"r"(tm) : "memory");
  if (warp >= 4) return;
  const bool ok_out = have_out && !*abort_flag;
  if (tid == 0 && *abort_flag) flag_status(p.status, PKV_DEV_TIMEOUT);
  const int d = tid;   // O^T lane = dimension
  const int64_t sh0 = static_cast<int64_t>(s) * p.num_q_heads + hq0;
  for (int h = 0; h < G; ++h) {
    const float L = lred[0][h] + lred[1][h] + lred[2][h] + lred[3][h];
    const float o = ok_out ? ov[h] : 0.f;
    if (nparts == 1) {
      p.out[(sh0 + h) * kTcD + d] = ok_out ? o / L : 0.f;
    } else {
      const int64_t pi = (sh0 + h) * p.max_parts + part;
      p.part_o[pi * kTcD + d] = o;
      if (d == 0) {
        p.part_ml[pi * 2 + 0] = ok_out ? m[h] : -CUDART_INF_F;
        p.part_ml[pi * 2 + 1] = ok_out ? L : 0.f;
      }
    }
  }
}

}  // namespace pkv
