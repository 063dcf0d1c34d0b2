// PagedAttention decode, tensor-core path with the contractions transposed
// (mma.sync m16n8k16; 16-bit, FP8 and INT8 caches; query groups of up to 8 heads).
//
// Same work split and staging as decode_mma.cuh (one CTA per sequence x KV
// head x split-KV partition; each warp streams every NW-th 16-token chunk
// through its own TMA ring), but the operands are laid out so the group's
// query heads ride in the mma's N=8 columns instead of its 16 rows:
//
//   S^T[t][h]  = sum_d K[t][d] q_h[d]     A = K chunk (16 tokens x 16 dims),
//                                         B = q^T (16 dims x 8 heads)
//   O^T[d][h] += sum_t V[t][d] P[h][t]    A = V^T chunk (16 dims x 16 tokens),
//                                         B = P^T (16 tokens x 8 heads)
//
// A 16-token chunk then takes 8 mma for QK and 8 per P part for PV, whatever
// the group size up to 8, half of what the heads-as-rows form needs ("LLM
// inference tutorial" section 4.4: all G heads of a KV head share every K/V
// byte).  The lane that holds S^T for heads 2*tig, 2*tig+1 also holds O^T for
// the same two heads, so the online-softmax rescale is lane-local.  P^T moves
// from the accumulator layout to the B-fragment layout through 512 bytes of
// per-warp shared memory: packed pairs in, one ldmatrix.trans out.
//
// 16-bit caches: fragments come from the swizzled tiles with ldmatrix
// (ldmatrix.trans for V^T); P is split into bf16 hi + lo parts.  8-bit caches
// (FP8 E4M3 or INT8): the codes are converted in registers to fp16 (exact for
// both) using a dimension
// permutation shared by q and K (QK) and an output-dimension permutation (PV)
// so each lane loads contiguous 16-byte slices; P is fp16.
#pragma once

#include <type_traits>

#include "decode_mma_fp8.cuh"

namespace pkv {

// Four 8-bit cache codes -> two f16x2 (bytes 0, 1 -> lo; 2, 3 -> hi), exactly.
// INT8 codes come out as code + 1152 (kBias): in S^T = K q^T the offset adds
// the same 1152 * sum(q) to every logit of a head, which its softmax (and the
// split-KV merge) cancels; in O^T = V^T P^T it adds 1152 * sum(P), which the
// epilogue subtracts, summing P as the fp16 values the MMA used.
constexpr float kI8Bias = 1152.f;
template <typename KV>
__device__ __forceinline__ void byte4_to_f16x2x2(uint32_t w, uint32_t& lo, uint32_t& hi) {
  if constexpr (std::is_same<KV, INT8>::value)
    s8x4_to_f16x2x2_biased(w, lo, hi);
  else
    e4m3x4_to_f16x2x2(w, lo, hi);
}

// Shared memory of one CTA: per warp a ring of STAGES chunks of CH tokens (K
// then V, each kBoxes tiles of [CH rows][128 B]) and a 1 KiB scratch for P^T.
template <typename KV, int D, int NW, int STAGES, int CH>
struct Mma2Smem {
  static constexpr int kBoxes = D * KV::kBytes / 128;             // 128-byte TMA boxes per row
  static constexpr int kBoxBytes = CH * 128;                      // [CH rows][128 B]
  static constexpr int kStageBytes = 2 * kBoxes * kBoxBytes;      // K + V
  static constexpr int kScratch = 32 * 16;                         // P^T rows [32][8 heads]
  static_assert(kScratch <= 1024, "P^T scratch fits its 1 KiB");
  static constexpr int kWarpBytes = STAGES * kStageBytes + 1024;  // + scratch, 1 KiB aligned
  static_assert(STAGES * kStageBytes >= 8 * (D + 3) * 4, "combine area fits a warp ring");
  static size_t bytes(int table_entries) {
    return 1024 + static_cast<size_t>(NW) * kWarpBytes + static_cast<size_t>(table_entries) * 4;
  }
};

// Fused append (16-bit caches): the new token of sequence s, KV head g, is at
// position ctx - 1, inside this CTA's last chunk.  One warp copies its K and V
// rows (16 bytes per lane) into the cache and orders the writes before that
// warp's TMA reads.  Only the slot the block table gives that position is
// accepted, so no other CTA reads the row.
template <int D>
__device__ __forceinline__ void fused_append_row16(const DecodeParams& p, int s, int g, int ctx,
                                                   int lb0, const int32_t* sbt, int lane) {
  const int64_t slot = __ldg(p.new_slots + s);
  if (slot >= 0) {
    const int32_t blk = sbt[((ctx - 1) >> p.bs_log2) - lb0];
    const int64_t want =
        blk < 0 ? -1
                : (static_cast<int64_t>(blk) << p.bs_log2) + ((ctx - 1) & ((1 << p.bs_log2) - 1));
    if (slot != want) {
      if (lane == 0) flag_status(p.status, PKV_DEV_BAD_SLOT);
    } else {
      constexpr int SEGS = D * 2 / 16;   // 16-byte segments per row
#pragma unroll
      for (int i = lane; i < 2 * SEGS; i += 32) {   // one pass for D <= 128, two for 256
        const bool is_v = i >= SEGS;
        const int seg = i % SEGS;
        const int64_t row = static_cast<int64_t>(s) * p.num_kv_heads + g;
        const uint4 val =
            __ldg(reinterpret_cast<const uint4*>(is_v ? p.v_new : p.k_new) + row * SEGS + seg);
        uint8_t* cache = const_cast<uint8_t*>(is_v ? p.v_cache : p.k_cache);
        *reinterpret_cast<uint4*>(cache + (slot * p.num_kv_heads + g) * (SEGS * 16) + seg * 16) = val;
      }
    }
  }
  asm volatile("fence.proxy.async.global;\n" ::: "memory");
  __syncwarp();
}

// 2^x on the SFU (ex2.approx: relative error about 2^-22; 2^-inf = 0).
__device__ __forceinline__ float fast_ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// Largest log2 gap between a head's reference max and a chunk's max before
// the running state is rescaled (p = 2^(s - m) < 2^8 in the P operands).
constexpr float kLazyLog2 = 8.f;

template <typename KV, int D, bool QF32, int NW, int STAGES, int CH>
__global__ void __launch_bounds__(NW * 32)
    paged_decode_mma2_kernel(const __grid_constant__ CUtensorMap tmap_k,
                             const __grid_constant__ CUtensorMap tmap_v, const MmaParams mp) {
  using SM = Mma2Smem<KV, D, NW, STAGES, CH>;
  constexpr bool F8 = KV::kBytes == 1;                      // 8-bit codes (FP8 or INT8)
  constexpr bool I8 = std::is_same<KV, INT8>::value;
  static_assert(!F8 || D == 128, "the 8-bit path is built for head_dim 128");
  // Tokens per chunk: 16 for 16-bit rows; 32 (two 16-token row tiles, RT = 2)
  // for 8-bit rows, so a chunk carries the same 8 KiB and the per-chunk work
  // (barrier wait, copies, softmax reductions, P^T round trip) is paid once
  // per 32 tokens.
  constexpr int RT = CH / 16;
  static_assert(CH == 16 || (F8 && CH == 32), "16-token chunks, or 32 for 8-bit rows");
  constexpr int H = SM::kBoxes;
  constexpr int KSTEPS = D / 16;   // QK k-steps
  constexpr int MT = D / 16;       // PV m-tiles (16 output dims each)
  const DecodeParams& p = mp.p;
  // Groups of 16 heads run as two CTAs per KV head, each with 8 of the heads
  // as the MMA's N columns; they read the same K/V rows one after the other
  // (adjacent in the grid), so the second finds them in L2.
  const int qsl = mp.q_split > 1 ? 1 : 0;   // log2 of the CTAs per KV head (1 or 2)
  const int G = (p.num_q_heads / p.num_kv_heads) >> qsl;   // query heads of this CTA

  extern __shared__ uint8_t smem_raw[];
  __shared__ __align__(8) uint64_t bars[NW][STAGES];
  uint8_t* smem = smem_raw + ((1024 - (smem_u32(smem_raw) & 1023)) & 1023);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int gid = lane >> 2, tig = lane & 3;
  const int P = p.partition_tokens;
  const int s = blockIdx.z, g = static_cast<int>(blockIdx.x) >> qsl, part = blockIdx.y;
  grid_dependency_wait();   // launched with launch_pdl: earlier work on the stream is done
  allow_dependents();

  // The partition's block-table entries are loaded before the context length
  // is known, so the two global round trips overlap (entries past the
  // context come along and are never used; every entry read is inside the
  // table row).  One entry per thread here; a long partition of small blocks
  // loads the rest once the length is known.  q is loaded after the first
  // copies are issued, so its round trip overlaps theirs, and a CTA past its
  // sequence's last partition leaves before either.  Against loading the
  // entries after the length (same box, 0.5 s of steps): 7B layer 185.3 ->
  // 183.5 us, FP8 7B 110.2 -> 107.8, ragged FP8 layer 669.7 -> 664.3.
  const int t_begin = part * P;
  const int lb0 = t_begin >> p.bs_log2;
  const int32_t* bt_row = p.block_tables + static_cast<int64_t>(s) * p.max_blocks_per_seq;
  const int nlb_max =
      min(((t_begin + P - 1) >> p.bs_log2) - lb0 + 1, p.max_blocks_per_seq - lb0);
  const int32_t b_pre =
      static_cast<int>(threadIdx.x) < nlb_max ? __ldg(bt_row + lb0 + threadIdx.x) : -1;
  const int hq0 = static_cast<int>(blockIdx.x) * G;   // (g * CTAs per head + which) * G

  int ctx = __ldg(p.context_lens + s);
  const int cap = context_cap(p);
  if (ctx < 0 || ctx > cap) {
    if (part == 0 && threadIdx.x == 0) flag_status(p.status, PKV_DEV_BAD_CONTEXT);
    ctx = ctx < 0 ? 0 : cap;
  }
  const int nparts = (ctx + P - 1) / P;
  if (part >= (nparts > 0 ? nparts : 1)) return;
  if (ctx == 0) {
    // a fused append needs its token inside the context
    if (p.k_new != nullptr && threadIdx.x == 0 && __ldg(p.new_slots + s) >= 0)
      flag_status(p.status, PKV_DEV_BAD_SLOT);
    for (int i = threadIdx.x; i < G * D; i += NW * 32)
      p.out[(static_cast<int64_t>(s) * p.num_q_heads + hq0) * D + i] = 0.f;
    return;
  }
  const int t_end = min(t_begin + P, ctx);

  int32_t* sbt = reinterpret_cast<int32_t*>(smem + NW * SM::kWarpBytes);
  const int nlb = ((t_end - 1) >> p.bs_log2) - lb0 + 1;
  for (int i = threadIdx.x; i < nlb; i += NW * 32) {
    int32_t b = i == static_cast<int>(threadIdx.x) ? b_pre : __ldg(bt_row + lb0 + i);   // nlb <= nlb_max
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

  float o[MT][4];
#pragma unroll
  for (int mt = 0; mt < MT; ++mt) o[mt][0] = o[mt][1] = o[mt][2] = o[mt][3] = 0.f;
  // softmax state of heads 2*tig and 2*tig+1
  float m0 = -CUDART_INF_F, m1 = -CUDART_INF_F, l0 = 0.f, l1 = 0.f;
  float ps0 = 0.f, ps1 = 0.f;   // INT8: sum of P as rounded to fp16 (the V offset's weight)

  uint8_t* ring = smem + warp * SM::kWarpBytes;
  uint8_t* scratch = ring + STAGES * SM::kStageBytes;      // P^T [32 rows][8 heads]
  const uint32_t ring_a = smem_u32(ring);
  const int nchunks = (t_end - t_begin + CH - 1) / CH;
  const int my_n = warp < nchunks ? (nchunks - warp + NW - 1) / NW : 0;
  const int box_rows = mp.box_rows;
  const int nbox = CH / box_rows;
  bool alive = true;

  // Fused append (16-bit caches): the partition's last chunk holds position
  // ctx - 1, the new token; the warp that owns that chunk copies the token's
  // rows before its first copy, while the other warps start streaming.  With
  // two CTAs per KV head both copy the same bytes, so each reads rows it has
  // written itself.
  const bool fuse_here = !F8 && p.k_new != nullptr && part == nparts - 1 && my_n > 0 &&
                         warp == (nchunks - 1) % NW;

  // One box per lane: K (even lanes) or V (odd), 128-byte column hh, row group
  // bx (at most 2 x 4 boxes: block_size >= 8).  Lane 0 arms the barrier with
  // the bytes of every box that is issued; a block-table hole or the rows past
  // the context issue none.
  auto issue = [&](int it) {
    if (it >= my_n) return;   // warp-uniform
    const int stage = it % STAGES;
    const int t0 = t_begin + (warp + it * NW) * CH;
    const uint32_t bar = smem_u32(&bars[warp][stage]);
    const int kv = lane & 1, hh = (lane >> 1) % H, bx = (lane >> 1) / H;
    const int tb = t0 + bx * box_rows;
    int32_t b = -1;
    if (bx < nbox && tb < ctx) b = sbt[(tb >> p.bs_log2) - lb0];
    const uint32_t n = __popc(__ballot_sync(0xffffffffu, b >= 0));
    if (lane == 0) mbar_arrive_expect_tx(bar, n * box_rows * 128);
    if (b >= 0) {
      const int z = (b << p.bs_log2) + (tb & ((1 << p.bs_log2) - 1));
      tma_load_3d(ring_a + stage * SM::kStageBytes + (kv * H + hh) * SM::kBoxBytes +
                      bx * box_rows * 128,
                  kv ? &tmap_v : &tmap_k, hh * (128 / KV::kBytes), g, z, bar);
    }
  };

  // 8-bit tiles: a lane reads K rows 16rt + gid (+8) at 16-byte units 2tig and
  // 2tig+1, and V rows 16kk + 2tig (+1, +8, +9) at unit gid.  Row r's swizzle
  // term depends on r mod 8 only, which is gid for the K rows and 2tig (+1)
  // for the V rows, so each read is one of these offsets plus a constant.
  const uint32_t k_swz0 = swz(gid, 2 * tig), k_swz1 = swz(gid, 2 * tig + 1);
  const uint32_t v_swz0 = swz(2 * tig, gid), v_swz1 = swz(2 * tig + 1, gid);

  if (!F8 && fuse_here) fused_append_row16<D>(p, s, g, ctx, lb0, sbt, lane);   // warp-uniform
  // Tests of the bounded waits: the first phase of warp 0's stage 0 in CTA
  // (0, 0, 0) expects bytes no copy brings, before any copy is issued, so its
  // wait runs out and the timeout path below runs.
  if (p.test_stall_bytes != 0 && warp == 0 && lane == 0 && my_n > 0 && blockIdx.x == 0 &&
      blockIdx.y == 0 && blockIdx.z == 0)
    mbar_expect_tx(smem_u32(&bars[0][0]), p.test_stall_bytes);
  __syncwarp();
#pragma unroll
  for (int st = 0; st < STAGES - 1; ++st) issue(st);

  // q^T as B fragments: b0 = q[gid][k 2tig..], b1 = q[gid][k 2tig+8..] of each k-step
  // (FP8: logical k 2tig+e (+8) of k-step ks <-> dim 32*tig + 4*ks + e (+2)).
  // log2-domain logit scale.  A negative scale is folded into q (exact sign
  // flip) and a zero one raised to the smallest normal (every logit is then
  // 0 as far as fp32 can tell), so sl2 > 0: the max of the scaled logits is
  // sl2 times the max of the raw ones, and a masked -inf stays -inf.
  // 8-bit caches carry q as fp16: the group's q is scaled by a power of two
  // into fp16's range (q_fp16_scale) and the logit scale takes it back.
  float sl2 = F8 ? p.qk_scale_log2 * __ldg(p.k_scale + g) : p.qk_scale_log2;
  const float qsign = sl2 < 0.f ? -1.f : 1.f;

  uint32_t qb[KSTEPS][2];
  uint32_t qblo[QF32 ? KSTEPS : 1][2];
  float q_unscale = 1.f;
  {
    const int64_t row = static_cast<int64_t>(s) * p.num_q_heads + hq0 + gid;
    const bool real = gid < G;
    auto qpair = [&](int ks, int half, float& x0, float& x1) {
      const int col = F8 ? 32 * tig + 4 * ks + 2 * half : 16 * ks + 8 * half + 2 * tig;
      x0 = x1 = 0.f;
      if (real) {
        if (QF32) {
          const float* qf = static_cast<const float*>(p.q) + row * D + col;
          x0 = qsign * qf[0];
          x1 = qsign * qf[1];
        } else {
          const __nv_bfloat16* qh = static_cast<const __nv_bfloat16*>(p.q) + row * D + col;
          x0 = qsign * __bfloat162float(qh[0]);
          x1 = qsign * __bfloat162float(qh[1]);
        }
      }
    };
    float qmul = 1.f;
    if constexpr (F8) {   // the group's largest |q| (the lanes cover every head and dim)
      float mx = 0.f;
#pragma unroll
      for (int ks = 0; ks < KSTEPS; ++ks)
#pragma unroll
        for (int half = 0; half < 2; ++half) {
          float x0, x1;
          qpair(ks, half, x0, x1);
          mx = fmaxf(mx, fmaxf(fabsf(x0), fabsf(x1)));
        }
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, off));
      qmul = q_fp16_scale(mx, q_unscale);
    }
#pragma unroll
    for (int ks = 0; ks < KSTEPS; ++ks) {
#pragma unroll
      for (int half = 0; half < 2; ++half) {
        float x0, x1;
        qpair(ks, half, x0, x1);
        if (F8) {
          x0 *= qmul;   // exact: a power of two
          x1 *= qmul;
        }
        uint32_t hi, lo;
        if (F8) {
          hi = pack_f16(x0, x1);
          const __half2 hv = *reinterpret_cast<const __half2*>(&hi);
          lo = pack_f16(x0 - __low2float(hv), x1 - __high2float(hv));
        } else {
          hi = pack_bf16(x0, x1);
          const __nv_bfloat162 hv = *reinterpret_cast<const __nv_bfloat162*>(&hi);
          lo = pack_bf16(x0 - __low2float(hv), x1 - __high2float(hv));
        }
        qb[ks][half] = hi;
        if (QF32) qblo[QF32 ? ks : 0][half] = lo;
      }
    }
  }

  sl2 = fmaxf(fabsf(sl2) * q_unscale, 1.17549435e-38f);


  for (int it = 0; it < my_n; ++it) {
    issue(it + STAGES - 1);
    const int stage = it % STAGES;
    const bool landed =
        __all_sync(0xffffffffu, mbar_wait(smem_u32(&bars[warp][stage]), (it / STAGES) & 1));
    if (!landed) {
      if (lane == 0) flag_status(p.status, PKV_DEV_TIMEOUT);
      alive = false;
      for (int k = it + 1; k < min(my_n, it + STAGES); ++k)
        mbar_wait(smem_u32(&bars[warp][k % STAGES]), (k / STAGES) & 1);
      break;
    }
    const int t0 = t_begin + (warp + it * NW) * CH;
    const int valid = min(CH, ctx - t0);
    uint8_t* kb = ring + stage * SM::kStageBytes;
    uint8_t* vb = kb + H * SM::kBoxBytes;
    const bool hole = __any_sync(
        0xffffffffu, valid < CH || (lane < nbox && sbt[((t0 + lane * box_rows) >> p.bs_log2) - lb0] < 0));
    if (hole) {   // rows the TMA did not fill become zero
      for (int i = lane; i < CH * 8 * H * 2; i += 32) {
        const int r = (i >> 3) % CH;
        const int rest = i / (8 * CH);
        const int bx = r / box_rows;
        const bool filled = r < valid && sbt[((t0 + bx * box_rows) >> p.bs_log2) - lb0] >= 0;
        if (!filled) {
          uint8_t* base = (rest < H ? kb : vb) + (rest % H) * SM::kBoxBytes;
          *reinterpret_cast<uint4*>(base + r * 128 + ((i & 7) << 4)) = make_uint4(0, 0, 0, 0);
        }
      }
      fence_proxy_async();   // these generic writes precede the TMA refill of the stage
      __syncwarp();
    }
    const uint32_t kb_a = smem_u32(kb), vb_a = smem_u32(vb);

    // ---- S^T = K q^T: tokens 16rt + gid, 16rt + gid + 8 x heads 2tig, 2tig+1 --------
    float sacc[RT][4];
#pragma unroll
    for (int rt = 0; rt < RT; ++rt) sacc[rt][0] = sacc[rt][1] = sacc[rt][2] = sacc[rt][3] = 0.f;
    if (F8) {
#pragma unroll
      for (int rt = 0; rt < RT; ++rt) {
        uint32_t wa[8], wb[8];   // 32-byte slices [32*tig, +32) of token rows gid, gid+8
        {
          const uint8_t* ka = kb + rt * 2048;   // rows 16rt + gid (+8): swizzle term k_swz*
          const uint4 a0 = *reinterpret_cast<const uint4*>(ka + k_swz0);
          const uint4 a1 = *reinterpret_cast<const uint4*>(ka + k_swz1);
          const uint4 b0 = *reinterpret_cast<const uint4*>(ka + 1024 + k_swz0);
          const uint4 b1 = *reinterpret_cast<const uint4*>(ka + 1024 + k_swz1);
          wa[0] = a0.x; wa[1] = a0.y; wa[2] = a0.z; wa[3] = a0.w;
          wa[4] = a1.x; wa[5] = a1.y; wa[6] = a1.z; wa[7] = a1.w;
          wb[0] = b0.x; wb[1] = b0.y; wb[2] = b0.z; wb[3] = b0.w;
          wb[4] = b1.x; wb[5] = b1.y; wb[6] = b1.z; wb[7] = b1.w;
        }
#pragma unroll
        for (int ks = 0; ks < KSTEPS; ++ks) {
          uint32_t a[4];   // {row gid k, row gid+8 k, row gid k+8, row gid+8 k+8}
          byte4_to_f16x2x2<KV>(wa[ks], a[0], a[2]);
          byte4_to_f16x2x2<KV>(wb[ks], a[1], a[3]);
          mma_f16(sacc[rt], a, qb[ks][0], qb[ks][1]);
          if (QF32) mma_f16(sacc[rt], a, qblo[QF32 ? ks : 0][0], qblo[QF32 ? ks : 0][1]);
        }
      }
    } else {
#pragma unroll
      for (int ks = 0; ks < KSTEPS; ++ks) {
        const int i = lane >> 3, r = (i & 1) * 8 + (lane & 7);
        const int hh = (16 * ks) / 64;
        const int u = ((16 * ks) % 64) / 8 + (i >> 1);
        uint32_t a[4];
        ldsm_x4(kb_a + hh * SM::kBoxBytes + swz(r, u), a[0], a[1], a[2], a[3]);
        mma_bf16(sacc[0], a, qb[ks][0], qb[ks][1]);
        if (QF32) mma_bf16(sacc[0], a, qblo[QF32 ? ks : 0][0], qblo[QF32 ? ks : 0][1]);
      }
    }
    // ---- online softmax (columns = heads 2tig, 2tig+1; rows = tokens) ------------
    // Columns of heads past the group are 0 (their q^T columns are 0): they stay
    // finite and are never written out, so only tokens past the context (a
    // partial chunk) are masked.
    if (valid < CH) {   // warp-uniform
#pragma unroll
      for (int rt = 0; rt < RT; ++rt) {
        if (16 * rt + gid >= valid) sacc[rt][0] = sacc[rt][1] = -CUDART_INF_F;
        if (16 * rt + gid + 8 >= valid) sacc[rt][2] = sacc[rt][3] = -CUDART_INF_F;
      }
    }
    float mx0 = fmaxf(sacc[0][0], sacc[0][2]), mx1 = fmaxf(sacc[0][1], sacc[0][3]);
#pragma unroll
    for (int rt = 1; rt < RT; ++rt) {
      mx0 = fmaxf(mx0, fmaxf(sacc[rt][0], sacc[rt][2]));
      mx1 = fmaxf(mx1, fmaxf(sacc[rt][1], sacc[rt][3]));
    }
#pragma unroll
    for (int off = 4; off < 32; off <<= 1) {
      mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, off));
      mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, off));
    }
    mx0 *= sl2;   // sl2 > 0: the max of the scaled logits
    mx1 *= sl2;
    // Lazy rescale: a head's reference max moves only when the chunk's max is
    // more than 2^kLazyLog2 above it, so p = 2^(s - m) stays below 256 and the
    // O rescale runs about once per partition instead of on most chunks (with
    // 8 heads one of them sets a new max in most chunks).  l and O share m, so
    // the normalised result is unchanged.  m = -inf first: every head moves.
    const bool up0 = mx0 > m0 + kLazyLog2, up1 = mx1 > m1 + kLazyLog2;
    if (__any_sync(0xffffffffu, up0 || up1)) {
      const float mn0 = up0 ? mx0 : m0, mn1 = up1 ? mx1 : m1;
      const float a0 = fast_ex2(m0 - mn0);   // 2^-inf = 0; 2^0 = 1
      const float a1 = fast_ex2(m1 - mn1);
      l0 *= a0;
      l1 *= a1;
      if (I8) {
        ps0 *= a0;
        ps1 *= a1;
      }
#pragma unroll
      for (int mt = 0; mt < MT; ++mt) {
        o[mt][0] *= a0;
        o[mt][1] *= a1;
        o[mt][2] *= a0;
        o[mt][3] *= a1;
      }
      m0 = mn0;
      m1 = mn1;
    }
    // P^T to B fragments via scratch laid out [token][8 heads] (16-byte rows):
    // each lane stores (token, heads 2tig, 2tig+1) as one packed pair, and one
    // ldmatrix.trans hands every lane its (tokens 2tig, 2tig+1; head gid) pairs.
    // 16-bit caches: bf16 hi rows 0..15, lo rows 16..31; 8-bit: fp16 rows 0..31.
#pragma unroll
    for (int rt = 0; rt < RT; ++rt) {
      const float p00 = fast_ex2(fmaf(sacc[rt][0], sl2, -m0));   // token 16rt+gid, head 2tig
      const float p01 = fast_ex2(fmaf(sacc[rt][1], sl2, -m1));   // head 2tig+1
      const float p10 = fast_ex2(fmaf(sacc[rt][2], sl2, -m0));   // token 16rt+gid+8
      const float p11 = fast_ex2(fmaf(sacc[rt][3], sl2, -m1));
      l0 += p00 + p10;
      l1 += p01 + p11;
      uint8_t* row0 = scratch + (16 * rt + gid) * 16 + 4 * tig;
      uint8_t* row1 = row0 + 8 * 16;
      if (F8) {
        const uint32_t h0 = pack_f16(p00, p01), h1 = pack_f16(p10, p11);
        *reinterpret_cast<uint32_t*>(row0) = h0;
        *reinterpret_cast<uint32_t*>(row1) = h1;
        if (I8) {   // P as the MMA sees it (rounded to fp16)
          const float2 f0 = __half22float2(*reinterpret_cast<const __half2*>(&h0));
          const float2 f1 = __half22float2(*reinterpret_cast<const __half2*>(&h1));
          ps0 += f0.x + f1.x;
          ps1 += f0.y + f1.y;
        }
      } else {
        const uint32_t h0 = pack_bf16(p00, p01), h1 = pack_bf16(p10, p11);
        *reinterpret_cast<uint32_t*>(row0) = h0;
        *reinterpret_cast<uint32_t*>(row1) = h1;
        *reinterpret_cast<uint32_t*>(row0 + 16 * 16) =
            pack_bf16(p00 - bf16_lo(h0), p01 - bf16_hi(h0));
        *reinterpret_cast<uint32_t*>(row1 + 16 * 16) =
            pack_bf16(p10 - bf16_lo(h1), p11 - bf16_hi(h1));
      }
    }
    __syncwarp();
    // matrix j = rows 8j..8j+7: 8-bit caches pb0/pb1 of k-steps 0 and 1; 16-bit
    // caches hi (k 0..7, 8..15) then lo
    uint32_t pb0[RT], pb1[RT];
    uint32_t pl0 = 0, pl1 = 0;
    {
      uint32_t r0, r1, r2, r3;
      ldsm_x4_t(smem_u32(scratch) + lane * 16, r0, r1, r2, r3);
      pb0[0] = r0;
      pb1[0] = r1;
      if constexpr (RT == 2) {
        pb0[RT - 1] = r2;
        pb1[RT - 1] = r3;
      } else {
        pl0 = r2;
        pl1 = r3;
      }
    }

    // ---- O^T += V^T P^T -----------------------------------------------------------
    if (F8) {
#pragma unroll
      for (int kk = 0; kk < RT; ++kk) {
        // lane owns output dims 16*gid + 2*mt + (0 | 1); tokens 16kk + 2tig, +1, +8, +9
        const uint8_t* va_row = vb + kk * 2048;   // rows 16kk + 2tig, +1, +8, +9
        const uint4 va = *reinterpret_cast<const uint4*>(va_row + v_swz0);
        const uint4 vv = *reinterpret_cast<const uint4*>(va_row + v_swz1);
        const uint4 vc = *reinterpret_cast<const uint4*>(va_row + 1024 + v_swz0);
        const uint4 vd = *reinterpret_cast<const uint4*>(va_row + 1024 + v_swz1);
        const uint32_t A[4] = {va.x, va.y, va.z, va.w}, B[4] = {vv.x, vv.y, vv.z, vv.w};
        const uint32_t Cw[4] = {vc.x, vc.y, vc.z, vc.w}, Dw[4] = {vd.x, vd.y, vd.z, vd.w};
#pragma unroll
        for (int w = 0; w < 4; ++w) {
          const uint32_t lo01 = __byte_perm(A[w], B[w], 0x5140);   // bytes 4w, 4w+1 of r0 / r0+1
          const uint32_t hi01 = __byte_perm(A[w], B[w], 0x7362);   // bytes 4w+2, 4w+3
          const uint32_t lo89 = __byte_perm(Cw[w], Dw[w], 0x5140);
          const uint32_t hi89 = __byte_perm(Cw[w], Dw[w], 0x7362);
          uint32_t aA[4], aB[4];   // m-tiles 2w and 2w+1
          byte4_to_f16x2x2<KV>(lo01, aA[0], aA[1]);
          byte4_to_f16x2x2<KV>(lo89, aA[2], aA[3]);
          byte4_to_f16x2x2<KV>(hi01, aB[0], aB[1]);
          byte4_to_f16x2x2<KV>(hi89, aB[2], aB[3]);
          mma_f16(o[2 * w], aA, pb0[kk], pb1[kk]);
          mma_f16(o[2 * w + 1], aB, pb0[kk], pb1[kk]);
        }
      }
    } else {
#pragma unroll
      for (int mt = 0; mt < MT; ++mt) {
        const int i = lane >> 3, r = (i >> 1) * 8 + (lane & 7);
        const int hh = (16 * mt) / 64;
        const int u = ((16 * mt) % 64) / 8 + (i & 1);
        uint32_t a[4];
        ldsm_x4_t(vb_a + hh * SM::kBoxBytes + swz(r, u), a[0], a[1], a[2], a[3]);
        mma_bf16(o[mt], a, pb0[0], pb1[0]);
        mma_bf16(o[mt], a, pl0, pl1);
      }
    }
    __syncwarp();   // every lane is done with this stage before it is refilled
  }

  // ---- warp epilogue: l summed over the 8 token-row lanes; rows into the idle ring ----
#pragma unroll
  for (int off = 4; off < 32; off <<= 1) {
    l0 += __shfl_xor_sync(0xffffffffu, l0, off);
    l1 += __shfl_xor_sync(0xffffffffu, l1, off);
    if (I8) {
      ps0 += __shfl_xor_sync(0xffffffffu, ps0, off);
      ps1 += __shfl_xor_sync(0xffffffffu, ps1, off);
    }
  }
  if (!alive) {
    m0 = m1 = -CUDART_INF_F;
    l0 = l1 = 0.f;
  }
  __syncwarp();
  float* wres = reinterpret_cast<float*>(ring);   // [8][D] acc, then m[8], l[8], psum[8]
#pragma unroll
  for (int e = 0; e < 2; ++e) {
    const int h = 2 * tig + e;
    if (h < G) {
#pragma unroll
      for (int mt = 0; mt < MT; ++mt) {
        const int d_lo = F8 ? 16 * gid + 2 * mt : 16 * mt + gid;
        const int d_hi = F8 ? 16 * gid + 2 * mt + 1 : 16 * mt + gid + 8;
        wres[h * D + d_lo] = alive ? o[mt][e] : 0.f;
        wres[h * D + d_hi] = alive ? o[mt][2 + e] : 0.f;
      }
      if (gid == 0) {
        wres[8 * D + h] = e ? m1 : m0;
        wres[8 * D + 8 + h] = e ? l1 : l0;
        wres[8 * D + 16 + h] = alive ? (e ? ps1 : ps0) : 0.f;
      }
    }
  }
  __syncthreads();

  const float vsc = F8 ? __ldg(p.v_scale + g) : 1.f;
  const bool single = nparts == 1;
  for (int i = threadIdx.x; i < G * D; i += NW * 32) {
    const int h = i / D, d = i % D;
    float M = -CUDART_INF_F;
#pragma unroll
    for (int w = 0; w < NW; ++w)
      M = fmaxf(M, reinterpret_cast<const float*>(smem + w * SM::kWarpBytes)[8 * D + h]);
    float L = 0.f, O = 0.f, PS = 0.f;
#pragma unroll
    for (int w = 0; w < NW; ++w) {
      const float* r = reinterpret_cast<const float*>(smem + w * SM::kWarpBytes);
      const float c = exp2f(r[8 * D + h] - M);
      L = fmaf(r[8 * D + 8 + h], c, L);
      O = fmaf(r[h * D + d], c, O);
      if (I8) PS = fmaf(r[8 * D + 16 + h], c, PS);
    }
    if (I8) O = fmaf(-kI8Bias, PS, O);   // the V codes' offset
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
