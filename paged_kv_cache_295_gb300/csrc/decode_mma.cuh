// PagedAttention decode, tensor-core path for 16-bit KV caches.
//
// Same work split as the CUDA-core path (one CTA per sequence x KV head x
// split-KV partition, every warp an independent consumer of 16-token chunks)
// but the two contractions run on the tensor cores and the K/V tiles arrive by
// TMA:
//
//  * Staging.  Each chunk is 16 tokens of one KV head: for K and for V, two
//    TMA boxes of [16 tokens][64 elements] (128 bytes per row, 128B swizzle)
//    fetched straight from the paged cache through a 3-D tensor map over
//    [num_blocks * block_size rows][num_kv_heads][head_dim]; the row coordinate
//    is physical_block * block_size + offset, read from the block table
//    ("nano-vLLM architecture" section 4.2: the kernel addresses K/V through
//    the logical -> physical mapping).  One lane issues the copies of its warp
//    and arms the stage's mbarrier with the byte count; the warp waits on the
//    barrier with a bounded try_wait.
//
//  * QK.  S[h][t] = q_h . K_t as mma.m16n8k16 with A = the query group (the G
//    query heads of this KV head as rows, zero-padded to 16) and B = the K tile
//    (ldmatrix of token rows), so each K byte is read once per KV head and the
//    G heads share it ("LLM inference tutorial" section 4.4 GQA head map
//    h -> h / G).  A float32 q is split into bf16 hi + lo parts and both are
//    applied, so the product keeps float32 accuracy.
//
//  * Softmax.  Logits are scaled by scale * log2(e) in float32 and folded into
//    a running max / sum per query row (online softmax, base 2).
//
//  * PV.  O[h][d] += P[h][t] V[t][d] with the probabilities re-used from the QK
//    accumulator layout as the A operand (16 tokens = one k-step; P is split
//    into bf16 hi + lo parts, two products) and V as the B operand via
//    ldmatrix.trans.  Accumulation is float32.
//
// The epilogue (combining warps, writing the output or split-KV partials) is
// the same as the CUDA-core path's.
#pragma once

#include <cuda.h>

#include "decode_kernel.cuh"

namespace pkv {

constexpr int kMmaChunk = 16;              // tokens per stage
constexpr int kMmaBoxCols = 64;            // 16-bit elements per TMA box row (128 B)
constexpr uint32_t kWaitLimitNs = 2000000000u;   // 2 s bound on any mbarrier wait

struct MmaParams {
  DecodeParams p;
  int32_t box_rows;      // rows per TMA box: min(block_size, 16)
  int32_t q_split = 1;   // transposed kernel: CTAs per KV head (1, or 2 for
                         // G = 16), each taking G / q_split of its query heads
};

__device__ __forceinline__ uint32_t smem_u32(const void* ptr) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(ptr));
}

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;\n" ::"r"(bar), "r"(count) : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;\n" ::"r"(bar), "r"(bytes)
               : "memory");
}

// Raises the barrier's expected transaction bytes without arriving.
__device__ __forceinline__ void mbar_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.expect_tx.relaxed.cta.shared::cta.b64 [%0], %1;\n" ::"r"(bar), "r"(bytes)
               : "memory");
}

__device__ __forceinline__ uint64_t global_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// Bounded wait for the barrier phase `parity`; false after kWaitLimitNs.
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity) {
  uint32_t ok = 0;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n"
      " selp.u32 %0, 1, 0, p;\n}\n"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  if (ok) return true;
  const uint64_t t0 = global_ns();
  while (true) {
    asm volatile(
        "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n"
        " selp.u32 %0, 1, 0, p;\n}\n"
        : "=r"(ok)
        : "r"(bar), "r"(parity)
        : "memory");
    if (ok) return true;
    if (global_ns() - t0 > kWaitLimitNs) return false;
  }
}

__device__ __forceinline__ void tma_load_3d(uint32_t dst, const CUtensorMap* map, int x, int y,
                                            int z, uint32_t bar) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3, %4}], [%5];\n" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(z), "r"(bar)
      : "memory");
}

__device__ __forceinline__ void fence_proxy_async() {
  asm volatile("fence.proxy.async.shared::cta;\n" ::: "memory");
}

__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2,
                                        uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];\n"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}

__device__ __forceinline__ void ldsm_x4_t(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2,
                                          uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0, %1, %2, %3}, [%4];\n"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}

// D = A(16x16 bf16, row) * B(16x8 bf16, col) + D, float32 accumulate.
__device__ __forceinline__ void mma_bf16(float* d, const uint32_t* a, uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7},"
      " {%8, %9}, {%0, %1, %2, %3};\n"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
  __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);   // .x = lo (low half)
  return *reinterpret_cast<uint32_t*>(&v);
}

// Byte offset of 16-byte unit u of row r inside a 128B-swizzled [rows][128 B]
// box whose base is 1024-byte aligned (the TMA SWIZZLE_128B pattern).
__device__ __forceinline__ uint32_t swz(int r, int u) {
  return static_cast<uint32_t>(r * 128 + ((u ^ (r & 7)) << 4));
}

template <int D, int NW, int STAGES>
struct MmaSmem {
  static constexpr int kHalves = D / kMmaBoxCols;                 // TMA boxes per K (or V) row
  static constexpr int kBoxBytes = kMmaChunk * 128;               // one [16][64] box
  static constexpr int kStageBytes = 2 * kHalves * kBoxBytes;     // K + V
  static constexpr int kWarpBytes = STAGES * kStageBytes;
  static_assert(kWarpBytes >= 16 * (D + 2) * 4, "combine area fits a warp ring");
  // layout: [1 KiB alignment slack][NW rings][table entries]
  static size_t bytes(int table_entries) {
    return 1024 + static_cast<size_t>(NW) * kWarpBytes + static_cast<size_t>(table_entries) * 4;
  }
};

template <int D, bool QF32, bool ROWS16, int NW, int STAGES>
__global__ void __launch_bounds__(NW * 32)
    paged_decode_mma_kernel(const __grid_constant__ CUtensorMap tmap_k,
                            const __grid_constant__ CUtensorMap tmap_v, const MmaParams mp) {
  using SM = MmaSmem<D, NW, STAGES>;
  constexpr int H = SM::kHalves;
  constexpr int KSTEPS = D / 16;       // QK k-steps
  constexpr int NT = D / 8;            // PV n-tiles (8 output dims each)
  const DecodeParams& p = mp.p;
  const int G = p.num_q_heads / p.num_kv_heads;

  extern __shared__ uint8_t smem_raw[];
  __shared__ __align__(8) uint64_t bars[NW][STAGES];
  uint8_t* smem = smem_raw + ((1024 - (smem_u32(smem_raw) & 1023)) & 1023);

  const int s = blockIdx.z, g = blockIdx.x, part = blockIdx.y;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int gid = lane >> 2, tig = lane & 3;   // mma group id / thread in group
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

  // Query fragments (A operand, rows = query heads of this group).
  uint32_t qa[KSTEPS][4];
  uint32_t qlo[QF32 ? KSTEPS : 1][4];
  {
    const int64_t row0 = static_cast<int64_t>(s) * p.num_q_heads + hq0;
#pragma unroll
    for (int ks = 0; ks < KSTEPS; ++ks) {
#pragma unroll
      for (int half = 0; half < 2; ++half) {          // columns +0 / +8
#pragma unroll
        for (int rh = 0; rh < 2; ++rh) {              // rows gid / gid + 8
          const int h = gid + 8 * rh;
          const int col = 16 * ks + 8 * half + 2 * tig;
          float x0 = 0.f, x1 = 0.f;
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
          const uint32_t hi = pack_bf16(x0, x1);
          qa[ks][half * 2 + rh] = hi;
          if (QF32) {
            const __nv_bfloat162 hv = *reinterpret_cast<const __nv_bfloat162*>(&hi);
            qlo[QF32 ? ks : 0][half * 2 + rh] =
                pack_bf16(x0 - __low2float(hv), x1 - __high2float(hv));
          }
        }
      }
    }
  }

  float o[NT][4];
#pragma unroll
  for (int j = 0; j < NT; ++j) o[j][0] = o[j][1] = o[j][2] = o[j][3] = 0.f;
  float m0 = -CUDART_INF_F, m1 = -CUDART_INF_F, l0 = 0.f, l1 = 0.f;
  const float sl2 = p.qk_scale_log2;

  uint8_t* ring = smem + warp * SM::kWarpBytes;
  const uint32_t ring_a = smem_u32(ring);
  const int nchunks = (t_end - t_begin + kMmaChunk - 1) / kMmaChunk;
  const int my_n = warp < nchunks ? (nchunks - warp + NW - 1) / NW : 0;
  const int box_rows = mp.box_rows;
  const int nbox = kMmaChunk / box_rows;
  bool alive = true;

  // Issue the TMA boxes of chunk `it` (lane 0); returns nothing, arms the barrier.
  auto issue = [&](int it) {
    if (it >= my_n || lane != 0) return;
    const int stage = it % STAGES;
    const int t0 = t_begin + (warp + it * NW) * kMmaChunk;
    const uint32_t bar = smem_u32(&bars[warp][stage]);
    uint32_t bytes = 0;
    for (int bx = 0; bx < nbox; ++bx) {
      const int tb = t0 + bx * box_rows;
      if (tb >= ctx) break;
      if (sbt[(tb >> p.bs_log2) - lb0] >= 0) bytes += 2 * H * box_rows * 128;
    }
    mbar_arrive_expect_tx(bar, bytes);
    const uint32_t sbase = ring_a + stage * SM::kStageBytes;
    for (int bx = 0; bx < nbox; ++bx) {
      const int tb = t0 + bx * box_rows;
      if (tb >= ctx) break;
      const int32_t b = sbt[(tb >> p.bs_log2) - lb0];
      if (b < 0) continue;
      const int z = (b << p.bs_log2) + (tb & ((1 << p.bs_log2) - 1));
#pragma unroll
      for (int hh = 0; hh < H; ++hh) {
        const uint32_t off = hh * SM::kBoxBytes + bx * box_rows * 128;
        tma_load_3d(sbase + off, &tmap_k, hh * kMmaBoxCols, g, z, bar);
        tma_load_3d(sbase + H * SM::kBoxBytes + off, &tmap_v, hh * kMmaBoxCols, g, z, bar);
      }
    }
  };

#pragma unroll
  for (int st = 0; st < STAGES - 1; ++st) issue(st);

  for (int it = 0; it < my_n; ++it) {
    issue(it + STAGES - 1);
    const int stage = it % STAGES;
    const uint32_t parity = (it / STAGES) & 1;
    // every lane waits; the vote keeps the outcome warp-uniform
    const bool landed = __all_sync(0xffffffffu, mbar_wait(smem_u32(&bars[warp][stage]), parity));
    if (!landed) {
      if (lane == 0) flag_status(p.status, PKV_DEV_TIMEOUT);
      alive = false;
      // wait (bounded) for the copies already issued for later chunks
      for (int k = it + 1; k < min(my_n, it + STAGES); ++k)
        mbar_wait(smem_u32(&bars[warp][k % STAGES]), (k / STAGES) & 1);
      break;
    }
    const int t0 = t_begin + (warp + it * NW) * kMmaChunk;
    const int valid = min(kMmaChunk, ctx - t0);   // rows of this chunk inside the context
    uint8_t* kb = ring + stage * SM::kStageBytes;
    uint8_t* vb = kb + H * SM::kBoxBytes;
    // Rows the TMA did not fill (beyond the context, or a bad block id) are
    // zeroed so the tensor-core products never see stale or NaN bytes.
    bool hole = valid < kMmaChunk;
    if (!hole) {
      for (int bx = 0; bx < nbox; ++bx)
        if (sbt[((t0 + bx * box_rows) >> p.bs_log2) - lb0] < 0) hole = true;
    }
    if (hole) {
      for (int i = lane; i < kMmaChunk * 8 * H * 2; i += 32) {
        const int r = (i >> 3) % kMmaChunk;
        const int rest = i / (8 * kMmaChunk);   // half + kv * H
        const int bx = r / box_rows;
        const bool filled = r < valid && sbt[((t0 + bx * box_rows) >> p.bs_log2) - lb0] >= 0;
        if (!filled) {
          uint8_t* base = (rest < H ? kb : vb) + (rest % H) * SM::kBoxBytes;
          *reinterpret_cast<uint4*>(base + r * 128 + ((i & 7) << 4)) = make_uint4(0, 0, 0, 0);
        }
      }
      __syncwarp();
    }
    const uint32_t kb_a = smem_u32(kb), vb_a = smem_u32(vb);

    // ---- S = Q K^T over 16 tokens: two n-tiles of 8 tokens -------------------
    float sacc[2][4];
#pragma unroll
    for (int j = 0; j < 2; ++j) sacc[j][0] = sacc[j][1] = sacc[j][2] = sacc[j][3] = 0.f;
#pragma unroll
    for (int ks = 0; ks < KSTEPS; ++ks) {
      const int i = lane >> 3, r = (i >> 1) * 8 + (lane & 7);
      const int hh = (16 * ks) / kMmaBoxCols;
      const int u = ((16 * ks) % kMmaBoxCols) / 8 + (i & 1);
      uint32_t b00, b01, b10, b11;
      ldsm_x4(kb_a + hh * SM::kBoxBytes + swz(r, u), b00, b01, b10, b11);
      mma_bf16(sacc[0], qa[ks], b00, b01);
      mma_bf16(sacc[1], qa[ks], b10, b11);
      if (QF32) {
        mma_bf16(sacc[0], qlo[QF32 ? ks : 0], b00, b01);
        mma_bf16(sacc[1], qlo[QF32 ? ks : 0], b10, b11);
      }
    }
    // ---- online softmax (rows gid and gid+8) ------------------------------------
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
    // P as the A operand, split into bf16 hi + lo parts so the PV product
    // keeps ~2^-17 relative precision (a single bf16 P would cost ~2^-9).
    uint32_t pa[4], pl[4];
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
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const float x0 = pr[k >> 1][(k & 1) * 2], x1 = pr[k >> 1][(k & 1) * 2 + 1];
        pa[k] = pack_bf16(x0, x1);
        const __nv_bfloat162 hv = *reinterpret_cast<const __nv_bfloat162*>(&pa[k]);
        pl[k] = pack_bf16(x0 - __low2float(hv), x1 - __high2float(hv));
      }
    }
    // ---- O += P V: 16 tokens x D dims -------------------------------------------
#pragma unroll
    for (int j = 0; j < NT; j += 2) {
      const int i = lane >> 3, r = (i & 1) * 8 + (lane & 7);
      const int dt = j + (i >> 1);                       // dim tile of this matrix
      const int hh = (8 * dt) / kMmaBoxCols;
      const int u = ((8 * dt) % kMmaBoxCols) / 8;
      uint32_t b00, b01, b10, b11;
      ldsm_x4_t(vb_a + hh * SM::kBoxBytes + swz(r, u), b00, b01, b10, b11);
      mma_bf16(o[j], pa, b00, b01);
      mma_bf16(o[j + 1], pa, b10, b11);
      mma_bf16(o[j], pl, b00, b01);
      mma_bf16(o[j + 1], pl, b10, b11);
    }
    // All lanes are done reading this stage before it is refilled; order the
    // generic-proxy accesses before the next async-proxy write.
    fence_proxy_async();
    __syncwarp();
  }

  // ---- warp epilogue: quad sums of l, per-warp rows into the idle ring --------
  l0 += __shfl_xor_sync(0xffffffffu, l0, 1);
  l0 += __shfl_xor_sync(0xffffffffu, l0, 2);
  if (ROWS16) {
    l1 += __shfl_xor_sync(0xffffffffu, l1, 1);
    l1 += __shfl_xor_sync(0xffffffffu, l1, 2);
  }
  if (!alive) {   // a timed-out wait: contribute nothing
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
        wres[h * D + 8 * j + 2 * tig] = alive ? o[j][2 * rh] : 0.f;
        wres[h * D + 8 * j + 2 * tig + 1] = alive ? o[j][2 * rh + 1] : 0.f;
      }
      if (tig == 0) {
        wres[16 * D + h] = rh ? m1 : m0;
        wres[16 * D + 16 + h] = rh ? l1 : l0;
      }
    }
  }
  __syncthreads();

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
      p.out[sh * D + d] = O / L;
    } else {
      const int64_t pi = sh * p.max_parts + part;
      p.part_o[pi * D + d] = O;
      if (d == 0) {
        p.part_ml[pi * 2 + 0] = M;
        p.part_ml[pi * 2 + 1] = L;
      }
    }
  }
}

}  // namespace pkv
