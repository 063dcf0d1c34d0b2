// Paged (chunked) prefill attention on the 5th-generation tensor cores
// (tcgen05 + TMEM), bf16 q and caches, head_dim 128.
//
// Prefill is the compute-bound phase ("LLM inference tutorial" section 1.2);
// a chunk of a prompt's tokens ("LLM inference tutorial" section 6.2 chunked
// prefill) attends, causally, over every cached key of its sequence, which the
// kernel reads through the block table ("nano-vLLM architecture" section 4.2).
//
// Work split: one CTA per (pair of query tiles, KV head, sequence).  A query
// tile is 128 accumulator rows: TQ = 128 / G consecutive query tokens times the
// G query heads that share the KV head ("LLM inference tutorial" section 4.4
// GQA), row r = token (r / G), head (r % G), so every K/V byte a CTA loads
// serves all G heads of both tiles.  The CTA walks its keys in 64-token tiles:
//
//   S_t  = Q_t K^T    tcgen05.mma M=128 N=64  K=128   A = Q_t (TMEM, written once)
//                                                     B = K tile (smem, K-major)
//   P_t  = 2^(S_t*scale*log2e - m)  in tile t's softmax warpgroup, one TMEM
//                                   lane = one row
//   O_t += P_t V      tcgen05.mma M=128 N=128 K=64    A = P_t (smem, K-major,
//                                                          bf16 hi + lo parts;
//                                                          8-bit caches: fp16)
//                                                     B = V tile (smem, MN-major)
//
// for t = A (the earlier tokens) and B.  TMEM: per tile, Q in 64 columns (row =
// lane, column c = dims 2c and 2c+1), S in 64 and O in 128 (512 columns in
// all).  Q read from TMEM takes its 32 KB per key tile and tile off the
// tensor cores' shared-memory reads, which are close to the port's limit, and
// frees the shared memory for 5 K/V stages; S is single-buffered, so QK of key
// tile j+1 waits until the softmax has loaded S(j).  Warp roles: warps 0-3
// softmax of tile A, warps 4-7 softmax of tile B (warp w owns TMEM lanes
// 32(w%4)..+31, i.e. rows), warps 8 and 11 TMA producers of K and V (lanes
// look up one key tile's blocks in one round trip and issue its boxes, one
// 64-column half each), warp 9 issues the QK MMAs
// and warp 10 the PV MMAs: a single thread issues one tcgen05.mma about every
// 125 cycles, so two issuing threads double the MMA rate and let QK run ahead
// of PV.  The two softmax warpgroups work on the same key tile at once, so each SM sub-
// partition has two softmax warps to interleave.  Tile A needs no key past
// its last token: its MMAs and softmax stop there.  The running max moves only
// when a tile's row max exceeds it by more than 2^8, so O is rarely rescaled.
// Every wait is bounded (2 s) and gives up when another role has given up;
// TMEM is released before the CTA exits.
#pragma once

#include <type_traits>

#include "decode_mma_fp8.cuh"
#include "tcgen05.cuh"

namespace pkv {

constexpr int kPfRows = 128;   // accumulator rows per query tile (M)
constexpr int kPfKeys = 64;    // keys per tile (N of QK, K of PV)
constexpr int kPfD = 128;
constexpr int kPfThreads = 384;   // 2 softmax warpgroups, K producer, QK issuer, PV issuer,
                                  // V producer
constexpr int kPfStages = 5;       // 16-bit caches
constexpr int kPfStagesFp8 = 3;    // 8-bit caches: the raw tiles take two stages' room
constexpr int kPfRawBufs = 4;      // FP8 raw tiles in flight per tensor
constexpr int kPfRankSeqs = 128;   // sequences ranked by context length for the work order

struct PrefillParams {
  const __nv_bfloat16* q;        // [T, Hq, D]
  const int32_t* query_start;    // [S + 1]
  const int32_t* block_tables;   // [S, max_blocks_per_seq]
  const int32_t* context_lens;   // [S]
  float* out;                    // [T, Hq, D]
  int32_t* status;
  int64_t num_blocks;
  int32_t num_q_heads;
  int32_t num_kv_heads;
  int32_t max_blocks_per_seq;
  int32_t bs_log2;
  int32_t box_rows;              // min(block_size, 64)
  int32_t tile_tokens;           // TQ = 128 / G tokens per query tile (two per CTA)
  int32_t causal;
  int32_t max_context_len;       // host bound: larger context_lens are flagged
  int32_t num_tokens;            // T: rows of q and out
  float qk_scale_log2;
  const float* k_scale;          // FP8 caches: [num_kv_heads] dequant scales
  const float* v_scale;
};

// 2^x with the MUFU instruction (relative error about 2^-22; 2^-inf = +0,
// results below 2^-126 flush to 0, which only drops terms that small).
// max(a, b, c) in one instruction (sm_100 and later)
__device__ __forceinline__ float pf_max3(float a, float b, float c) {
  float y;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(y) : "f"(a), "f"(b), "f"(c));
  return y;
}

__device__ __forceinline__ float pf_ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// 64 consecutive TMEM columns of this warp's 32 lanes -> 64 registers, with one
// wait for both loads.
__device__ __forceinline__ void pf_ld64(uint32_t taddr, float* v) {
  uint32_t r[64];
#define PKV_R8(i) "=r"(r[i]), "=r"(r[i + 1]), "=r"(r[i + 2]), "=r"(r[i + 3]), "=r"(r[i + 4]), \
                  "=r"(r[i + 5]), "=r"(r[i + 6]), "=r"(r[i + 7])
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,"
      "%15,%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];\n"
      : PKV_R8(0), PKV_R8(8), PKV_R8(16), PKV_R8(24)
      : "r"(taddr));
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,"
      "%15,%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];\n"
      : PKV_R8(32), PKV_R8(40), PKV_R8(48), PKV_R8(56)
      : "r"(taddr + 32));
#undef PKV_R8
  asm volatile("tcgen05.wait::ld.sync.aligned;\n" ::: "memory");
#pragma unroll
  for (int i = 0; i < 64; ++i) v[i] = __uint_as_float(r[i]);
}

struct PfLayout {
  // [P_A][P_B]: 16-bit caches bf16 hi 16 KB + lo 16 KB per tile, 8-bit caches
  // fp16 16 KB; [8-bit only: raw tiles, K x4 then V x4, 8 KB each]
  // [stages: K 16 KB, V 16 KB]
  static constexpr int kPPart = kPfRows * 128;         // [128 rows][64 keys x 2 B]
  __host__ __device__ static constexpr int pbuf(bool fp8) { return fp8 ? kPPart : 2 * kPPart; }
  static constexpr int kP = 0;                         // P_A, then P_B
  static constexpr int kKVHalf = kPfKeys * 128;        // [64 keys][128 B]
  static constexpr int kStage = 4 * kKVHalf;           // K (2 halves) + V (2 halves)
  __host__ __device__ static constexpr int raw(bool fp8) { return kP + 2 * pbuf(fp8); }
  static constexpr int kRawTile = kPfKeys * 128;       // [64 keys][128 codes]
  static constexpr int kRawBytes = 2 * kPfRawBufs * kRawTile;   // (K, V) x buffers
  __host__ __device__ static constexpr int ring(bool fp8) { return raw(fp8) + (fp8 ? kRawBytes : 0); }
  static constexpr size_t bytes(int stages, bool fp8) {
    return 1024 + static_cast<size_t>(ring(fp8)) + static_cast<size_t>(stages) * kStage;
  }
};

// KIND: 0 bf16 cache; 1 FP8-E4M3 codes; 2 INT8 codes.  Both 8-bit kinds take
// the widening path (FP8 below means "8-bit codes").
template <int STAGES, int KIND>
__global__ void __launch_bounds__(kPfThreads, 1)
    paged_prefill_tc_kernel(const __grid_constant__ CUtensorMap tmap_k,
                            const __grid_constant__ CUtensorMap tmap_v, const PrefillParams p) {
  using LY = PfLayout;
  // FP8 caches: the tiles are widened to fp16 in shared memory, so both
  // contractions run as f16 MMAs (q and P in fp16 too); bf16 caches run bf16.
  constexpr bool FP8 = KIND != 0;
  constexpr bool I8 = KIND == 2;
  constexpr int kRing = LY::ring(FP8);
  const int G = p.num_q_heads / p.num_kv_heads;
  const int TQ = p.tile_tokens;

  extern __shared__ uint8_t smem_raw[];
  __shared__ __align__(8) uint64_t full[STAGES], full_v[STAGES], empty[STAGES];
  __shared__ __align__(8) uint64_t s_full[2], s_free[2], q_ready[2], p_full[2], o_done[2], drain[2];
  __shared__ __align__(8) uint64_t raw_full[2][kPfRawBufs];   // FP8: [K | V][buffer] landed
  __shared__ uint64_t key_mask[STAGES];   // per stage: keys with cache data
  __shared__ uint32_t tmem_base_sh;
  __shared__ int abort_sh;
  __shared__ int seq_sh;
  uint8_t* sm = smem_raw + ((1024 - (smem_u32(smem_raw) & 1023)) & 1023);
  const uint32_t sma = smem_u32(sm);
  volatile int* abort_flag = &abort_sh;

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  // Work order.  CTAs start roughly in the order of their linear block index,
  // so that index is mapped to (sequence, pair, KV head) longest context
  // first: a long prompt's CTAs then start in the first waves instead of
  // trailing the grid.  KV heads run fastest (their CTAs are alike), then the
  // pairs of a sequence (latest, i.e. heaviest, first), then the sequences by
  // context length, descending, ties by index.  Each CTA ranks the sequences
  // itself (one pass over the context lengths per thread), so this is done
  // for up to kPfRankSeqs sequences; more keep their order.
  const uint64_t lin = blockIdx.x + static_cast<uint64_t>(gridDim.x) *
                                        (blockIdx.y + static_cast<uint64_t>(gridDim.y) * blockIdx.z);
  const int g = static_cast<int>(lin % gridDim.y);
  const uint64_t unit = lin / gridDim.y;
  const int pair = static_cast<int>(gridDim.x - 1 - unit % gridDim.x);
  const int rank = static_cast<int>(unit / gridDim.x);   // < gridDim.z
  int s = rank;
  if (gridDim.z <= kPfRankSeqs) {
    if (tid == 0) seq_sh = rank;   // kept if no sequence claims the rank
    __syncthreads();
    if (tid < static_cast<int>(gridDim.z)) {
      const int c = __ldg(p.context_lens + tid);
      int r = 0;
      for (int i = 0; i < static_cast<int>(gridDim.z); ++i) {
        const int ci = __ldg(p.context_lens + i);
        r += (ci > c || (ci == c && i < tid)) ? 1 : 0;
      }
      if (r == rank) seq_sh = tid;   // ranks are distinct: one writer
    }
    __syncthreads();
    s = seq_sh;
  }

  const int q0 = __ldg(p.query_start + s);
  const int q1 = __ldg(p.query_start + s + 1);
  if (q0 < 0 || q1 < q0 || q1 > p.num_tokens) {   // rows outside q / out: touch nothing
    if (pair == 0 && g == 0 && tid == 0) flag_status(p.status, PKV_DEV_BAD_CONTEXT);
    return;
  }
  const int n = q1 - q0;
  if (pair == 0 && tid == 0 && n > 2 * static_cast<int>(gridDim.x) * TQ)
    flag_status(p.status, PKV_DEV_BAD_CONTEXT);   // more queries than max_query_len
  const int tok0 = pair * 2 * TQ;                 // tile A: tok0 .., tile B: tok0 + TQ ..
  if (n <= 0 || tok0 >= n) return;
  const bool has_b = tok0 + TQ < n;
  int ctx = __ldg(p.context_lens + s);
  const int cap = min(p.max_context_len, p.max_blocks_per_seq << p.bs_log2);
  if (ctx < n || ctx > cap) {   // queries must be the last n of a context the table covers
    if (pair == 0 && tid == 0) flag_status(p.status, PKV_DEV_BAD_CONTEXT);
    const int ntok = min(2 * TQ, n - tok0);
    for (int i = tid; i < ntok * G * kPfD; i += kPfThreads) {
      const int t = i / (G * kPfD), r = i % (G * kPfD);
      p.out[(static_cast<int64_t>(q0 + tok0 + t) * p.num_q_heads + g * G) * kPfD + r] = 0.f;
    }
    return;
  }
  // key tiles each query tile needs (causal: up to its last token's position)
  const int end_a = min(tok0 + TQ, n), end_b = min(tok0 + 2 * TQ, n);
  const int nt_a = ((p.causal ? ctx - n + end_a : ctx) + kPfKeys - 1) / kPfKeys;
  const int nt_b = has_b ? ((p.causal ? ctx - n + end_b : ctx) + kPfKeys - 1) / kPfKeys : 0;
  const int ntiles = max(nt_a, nt_b);
  const int32_t* bt_row = p.block_tables + static_cast<int64_t>(s) * p.max_blocks_per_seq;

  if (tid == 0) {
    for (int st = 0; st < STAGES; ++st) {
      mbar_init(smem_u32(&full[st]), 1);     // K copies and the key mask
      mbar_init(smem_u32(&full_v[st]), 1);   // V copies
      mbar_init(smem_u32(&empty[st]), 1);
    }
    for (int t = 0; t < 2; ++t) {
      mbar_init(smem_u32(&s_full[t]), 1);
      mbar_init(smem_u32(&s_free[t]), 4);
      mbar_init(smem_u32(&q_ready[t]), 4);
      mbar_init(smem_u32(&p_full[t]), 4);
      mbar_init(smem_u32(&o_done[t]), 1);
    }
    mbar_init(smem_u32(&drain[0]), 1);
    mbar_init(smem_u32(&drain[1]), 1);
    for (int i = 0; i < 2 * kPfRawBufs; ++i)
      mbar_init(smem_u32(&raw_full[i / kPfRawBufs][i % kPfRawBufs]), 1);
    abort_sh = 0;
    asm volatile("fence.mbarrier_init.release.cluster;\n" ::: "memory");
  }
  if (warp == 0) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], 512;\n" ::"r"(
                     smem_u32(&tmem_base_sh))
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;\n" ::: "memory");
  }
  fence_proxy_async();
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  // TMEM: tile t's Q at columns 256t + [0, 64), S at 256t + 64, O at 256t + 128
  const uint32_t tm = tmem_base_sh;

  if (warp == 8 || warp == 11) {
    // --------------------- TMA producers: warp 8 K, warp 11 V -------------------
    // Per key tile, lane 2i + h looks up box i's block (one round trip, issued
    // before the wait for the stage) and copies its 64-column half h, so one
    // instruction issues the tile's boxes of this producer's tensor.  Warp 8's
    // lane 0 publishes the tile's key mask next to the stage; each producer
    // arms its own barrier (full_k / full_v) with its bytes.
    const bool is_v = warp == 11;
    const int box_rows = p.box_rows;
    const int nbox = kPfKeys / box_rows;
    bool flagged = false;
    if constexpr (!FP8) {
    const int bx = lane >> 1, hh = lane & 1;
    for (int j = 0; j < ntiles; ++j) {
      const int st = j % STAGES;
      const int k0 = j * kPfKeys;
      const int kb = k0 + bx * box_rows;
      int32_t blk = -1;
      if (bx < nbox && kb < ctx) {
        const int32_t b = __ldg(bt_row + (kb >> p.bs_log2));
        blk = (b >= 0 && b < p.num_blocks) ? b : -2;
      }
      const uint32_t valid = __ballot_sync(0xffffffffu, blk >= 0 && hh == 0);   // bit 2i: box i
      if (!is_v && __ballot_sync(0xffffffffu, blk == -2) && !flagged) {
        if (lane == 0) flag_status(p.status, PKV_DEV_BAD_BLOCK);
        flagged = true;
      }
      if (j >= STAGES) {
        bool ok = true;
        if (lane == 0) ok = tc_wait(smem_u32(&empty[st]), ((j / STAGES) - 1) & 1, abort_flag);
        if (!__shfl_sync(0xffffffffu, ok, 0)) break;
      }
      const uint32_t bar = smem_u32(is_v ? &full_v[st] : &full[st]);
      if (lane == 0) {
        if (!is_v) {
          uint64_t m = 0;
          for (int i = 0; i < nbox; ++i) {
            if (!((valid >> (2 * i)) & 1u)) continue;
            const int rows = min(box_rows, ctx - (k0 + i * box_rows));
            const uint64_t run = rows >= 64 ? ~0ull : ((1ull << rows) - 1ull);
            m |= run << (i * box_rows);
          }
          key_mask[st] = m;
        }
        mbar_arrive_expect_tx(bar, static_cast<uint32_t>(__popc(valid)) * 2u * box_rows * 128u);
      }
      __syncwarp();
      if (blk >= 0) {
        const uint32_t dst = sma + kRing + st * LY::kStage + (is_v ? 2 * LY::kKVHalf : 0) +
                             hh * LY::kKVHalf + bx * box_rows * 128;
        const int z = (blk << p.bs_log2) + (kb & ((1 << p.bs_log2) - 1));
        tma_load_3d(dst, is_v ? &tmap_v : &tmap_k, hh * 64, g, z, bar);
      }
    }
    } else {
      // FP8 caches.  TMA brings a key tile's codes, [64 keys][128 B] in one
      // 128-byte box per row block, into one of kPfRawBufs raw buffers (lane i
      // looks up box i's block); the warp widens them to fp16 (exact for E4M3)
      // into the stage, in the swizzled K-major halves the MMAs read, and
      // arrives on the stage's barrier.  Tile j + kPfRawBufs's copy goes into
      // the raw buffer tile j has just left, so kPfRawBufs copies are in flight.
      const uint32_t raw_a = sma + LY::raw(true) + (is_v ? kPfRawBufs * LY::kRawTile : 0);
      const uint8_t* raw_p = sm + LY::raw(true) + (is_v ? kPfRawBufs * LY::kRawTile : 0);
      // Lane i's block of box i of tile jj: -1 past the context, -2 out of range.
      // Looked up one tile ahead of its copy, so the table load's latency
      // overlaps the widening of the tile in between.
      auto lookup = [&](int jj) -> int32_t {
        const int kb = jj * kPfKeys + lane * box_rows;
        if (jj >= ntiles || lane >= nbox || kb >= ctx) return -1;
        const int32_t b = __ldg(bt_row + (kb >> p.bs_log2));
        return (b >= 0 && b < p.num_blocks) ? b : -2;
      };
      auto issue_raw = [&](int jj, int32_t blk) -> uint32_t {   // bit i: box i has data
        const int kb = jj * kPfKeys + lane * box_rows;
        const uint32_t valid = __ballot_sync(0xffffffffu, blk >= 0);
        if (!is_v && __ballot_sync(0xffffffffu, blk == -2) && !flagged) {
          if (lane == 0) flag_status(p.status, PKV_DEV_BAD_BLOCK);
          flagged = true;
        }
        const uint32_t rbar = smem_u32(&raw_full[is_v ? 1 : 0][jj % kPfRawBufs]);
        if (lane == 0) mbar_arrive_expect_tx(rbar, static_cast<uint32_t>(__popc(valid)) * box_rows * 128u);
        __syncwarp();
        if (blk >= 0) {
          const int z = (blk << p.bs_log2) + (kb & ((1 << p.bs_log2) - 1));
          tma_load_3d(raw_a + (jj % kPfRawBufs) * LY::kRawTile + lane * box_rows * 128,
                      is_v ? &tmap_v : &tmap_k, 0, g, z, rbar);
        }
        return valid;
      };
      // valids[i]: the boxes of tile j + i that have data (a window that moves
      // with j, so it stays in registers)
      uint32_t valids[kPfRawBufs];
#pragma unroll
      for (int b = 0; b < kPfRawBufs; ++b) valids[b] = b < ntiles ? issue_raw(b, lookup(b)) : 0u;
      // Four codes -> two f16x2.  E4M3: exact.  INT8: code + 1152 (one XOR and
      // two PRMT): in K it adds the same 1152 * sum(q) to every logit of a row,
      // which its softmax cancels.  V takes the offset off again (two HSUB2 per
      // four codes): kept, it would make O about 1152 times the sum of P, and
      // over tens of thousands of keys the float32 accumulation of those large
      // products in the tensor cores drifts by more than the 8-bit bound (0.02
      // on 32K keys with one key 13 nats above the rest, against 1e-2), and the
      // P the MMA sees (rounded to fp16) need not sum to l either.
      auto widen4 = [&](uint32_t w, uint32_t& lo, uint32_t& hi) {
        if constexpr (I8)
          s8x4_to_f16x2x2_biased(w, lo, hi);
        else
          e4m3x4_to_f16x2x2(w, lo, hi);
      };
      uint32_t unit_off[8];   // where 16-byte unit u sits in a row r = lane (mod 8): swz(r, u) - 128 r
#pragma unroll
      for (int u = 0; u < 8; ++u) unit_off[u] = static_cast<uint32_t>((u ^ (lane & 7)) << 4);
      for (int j = 0; j < ntiles; ++j) {
        const int st = j % STAGES;
        const int k0 = j * kPfKeys;
        const int32_t next_blk = lookup(j + kPfRawBufs);   // used after this tile's widening
        if (j >= STAGES) {
          bool ok = true;
          if (lane == 0) ok = tc_wait(smem_u32(&empty[st]), ((j / STAGES) - 1) & 1, abort_flag);
          if (!__shfl_sync(0xffffffffu, ok, 0)) break;
        }
        // every lane waits, so the copied codes are visible to all of them
        const int rb = j % kPfRawBufs;
        if (!__all_sync(0xffffffffu, tc_wait(smem_u32(&raw_full[is_v ? 1 : 0][rb]),
                                             (j / kPfRawBufs) & 1, abort_flag)))
          break;
        const uint8_t* raw = raw_p + rb * LY::kRawTile;
        uint8_t* dst = sm + kRing + st * LY::kStage + (is_v ? 2 * LY::kKVHalf : 0);
        // raw row r, 16-byte chunk u = dims 16u .. 16u+15 -> fp16 half u / 4,
        // 16-byte chunks 2 (u % 4) and 2 (u % 4) + 1 of row r.  Lane = row and
        // one chunk per step: the swizzle then spreads each step's 32 loads and
        // 32 stores evenly over the banks (lanes on different chunks of the same
        // rows, or the two halves 8 KiB apart, would collide 4 ways).
        // Row r = 32k + lane: its swizzle term depends on lane mod 8 only, so
        // every address is a per-lane offset (unit_off) plus a constant.
        const uint8_t* raw_l = raw + lane * 128;
        uint8_t* dst_l = dst + lane * 128;
        // All of a lane's codes are loaded before the first store: the
        // compiler cannot tell the raw buffer from the stage, so a load after
        // a store would wait for it, and one load's latency per 16 codes made
        // the widening of a tile take about 2,000 cycles.
        auto widen_tile = [&](auto exact) {
          constexpr int kSteps = (kPfKeys / 32) * 8;
          uint4 cs[kSteps];
#pragma unroll
          for (int it = 0; it < kSteps; ++it)
            cs[it] = *reinterpret_cast<const uint4*>(raw_l + (it >> 3) * 32 * 128 + unit_off[it & 7]);
#pragma unroll
          for (int it = 0; it < kSteps; ++it) {
            const int rk = (it >> 3) * 32 * 128, u = it & 7;
            const uint4 c = cs[it];
            uint32_t h[8];
            widen4(c.x, h[0], h[1]);
            widen4(c.y, h[2], h[3]);
            widen4(c.z, h[4], h[5]);
            widen4(c.w, h[6], h[7]);
            if constexpr (decltype(exact)::value) {   // code + 1152 - 1152: the code, exactly
#pragma unroll
              for (int e = 0; e < 8; ++e) h[e] = hsub2_u32(h[e], 0x64806480u);
            }
            uint8_t* half = dst_l + (u >> 2) * LY::kKVHalf + rk;
            const int uu = 2 * (u & 3);
            *reinterpret_cast<uint4*>(half + unit_off[uu]) = make_uint4(h[0], h[1], h[2], h[3]);
            *reinterpret_cast<uint4*>(half + unit_off[uu + 1]) = make_uint4(h[4], h[5], h[6], h[7]);
          }
        };
        // INT8 V codes are widened exactly (K keeps the offset, see widen4)
        if (I8 && is_v)
          widen_tile(std::true_type{});
        else
          widen_tile(std::false_type{});
        fence_proxy_async();   // the stage's generic writes before the MMAs' reads; the
        __syncwarp();          // raw buffer's reads before the next copy into it
        if (lane == 0) {
          if (!is_v) {
            uint64_t m = 0;
            for (int i = 0; i < nbox; ++i) {
              if (!((valids[0] >> i) & 1u)) continue;
              const int rows = min(box_rows, ctx - (k0 + i * box_rows));
              const uint64_t run = rows >= 64 ? ~0ull : ((1ull << rows) - 1ull);
              m |= run << (i * box_rows);
            }
            key_mask[st] = m;
          }
          mbar_arrive(smem_u32(is_v ? &full_v[st] : &full[st]));
        }
#pragma unroll
        for (int b = 0; b + 1 < kPfRawBufs; ++b) valids[b] = valids[b + 1];
        valids[kPfRawBufs - 1] = j + kPfRawBufs < ntiles ? issue_raw(j + kPfRawBufs, next_blk) : 0u;
      }
    }
  } else if (warp == 9) {
    // ---------------------------- QK issuer ------------------------------------
    // Key tiles in order, tile A then B: once the stage has landed and the S
    // buffer is free (the softmax has loaded the previous S; Q is in TMEM
    // before the first).  Its commits cover only its own MMAs (s_full).
    if (lane == 0) {
      const uint32_t idesc_qk = tc_idesc(kPfRows, kPfKeys, false, false, !FP8);
      for (int j = 0; j < ntiles; ++j) {
        if (!tc_wait(smem_u32(&full[j % STAGES]), (j / STAGES) & 1, abort_flag)) break;
        const uint32_t kb = sma + kRing + (j % STAGES) * LY::kStage;
        bool ok = true;
        for (int t = 0; t < 2; ++t) {
          if (j >= (t == 0 ? nt_a : nt_b)) continue;
          const bool ready = j == 0 ? tc_wait(smem_u32(&q_ready[t]), 0, abort_flag)
                                    : tc_wait(smem_u32(&s_free[t]), (j - 1) & 1, abort_flag);
          if (!ready) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t dst = tm + 256 * t + kPfKeys;
          // the K descriptor is built once; a k-step only moves its start
          // address (bits 0-13, in 16-byte units) and Q's TMEM column (8 per
          // 16 dims)
          const uint64_t kd = tc_desc(kb, 0, 1024);
#pragma unroll
          for (int ks = 0; ks < kPfD / 16; ++ks) {
            const uint32_t off_k = (ks >> 2) * LY::kKVHalf + (ks & 3) * 32;
            tc_mma_ts(dst, tm + 256 * t + 8 * ks, kd + (off_k >> 4), idesc_qk, ks > 0);
          }
          tc_commit(smem_u32(&s_full[t]));
        }
        if (!ok) break;
      }
      tc_commit(smem_u32(&drain[0]));   // its MMAs finish before TMEM is released
      volatile int no_abort = 0;
      tc_wait(smem_u32(&drain[0]), 0, &no_abort);
    }
  } else if (warp == 10) {
    // ---------------------------- PV issuer ------------------------------------
    // Tile A then B of each key tile, once its P is written; after the last PV
    // that reads a stage, the stage is released (its QK finished before its P
    // could be written).
    if (lane == 0) {
      const uint32_t idesc_pv = tc_idesc(kPfRows, kPfD, false, true, !FP8);
      for (int j = 0; j < ntiles; ++j) {
        const uint32_t vb = sma + kRing + (j % STAGES) * LY::kStage + 2 * LY::kKVHalf;
        if (!tc_wait(smem_u32(&full_v[j % STAGES]), (j / STAGES) & 1, abort_flag)) break;
        bool ok = true;
        for (int t = 0; t < 2; ++t) {
          if (j >= (t == 0 ? nt_a : nt_b)) continue;
          if (!tc_wait(smem_u32(&p_full[t]), j & 1, abort_flag)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t dO = tm + 256 * t + 2 * kPfKeys;
          const uint64_t pd = tc_desc(sma + LY::kP + t * LY::pbuf(FP8), 0, 1024);
          const uint64_t vd = tc_desc(vb, LY::kKVHalf, 1024);
#pragma unroll
          for (int kk = 0; kk < kPfKeys / 16; ++kk) {
            const uint64_t bdesc = vd + ((kk * 2048) >> 4);
            tc_mma(dO, pd + ((kk * 32) >> 4), bdesc, idesc_pv, (j > 0 || kk > 0));
            if constexpr (!FP8) tc_mma(dO, pd + ((LY::kPPart + kk * 32) >> 4), bdesc, idesc_pv, 1);
          }
          tc_commit(smem_u32(&o_done[t]));
        }
        if (!ok) break;
        tc_commit(smem_u32(&empty[j % STAGES]));
      }
      tc_commit(smem_u32(&drain[1]));
      volatile int no_abort = 0;
      tc_wait(smem_u32(&drain[1]), 0, &no_abort);
    }
  } else {
    // -------------------- softmax warpgroups (A: 0-3, B: 4-7) -----------------
    const int t = warp >> 2;                            // query tile of this warpgroup
    const int r = tid & 127;                            // accumulator row = TMEM lane
    const int my_nt = t == 0 ? nt_a : nt_b;
    const uint32_t lane_q = static_cast<uint32_t>((warp & 3) * 32) << 16;
    const uint32_t tQ = tm + 256 * t, tS = tQ + kPfKeys, tO = tQ + 2 * kPfKeys;
    const int tl = r / G;
    const bool row_ok = r < TQ * G && tok0 + t * TQ + tl < n;
    // FP8 caches: the row goes to fp16 scaled by 2^qsh, which puts its largest
    // |q| in [2^14, 2^15): inside fp16's range whatever q's magnitude, and
    // exact for every element within 2^-24 of that max (a bf16 has 8
    // significant bits).  The logit scale takes 2^-qsh back.
    float q_unscale = 1.f;
    {   // this row of Q_t (token tok0 + t*TQ + r/G, head g*G + r%G; 0 past the
        // chunk) into TMEM, bf16 pairs per column (fp16 for FP8 caches): the A
        // operand of every QK
      float w[64];
      const uint4* src = reinterpret_cast<const uint4*>(
          p.q + (static_cast<int64_t>(q0 + tok0 + t * TQ + tl) * p.num_q_heads + g * G + r % G) *
                    kPfD);
      float qmul = 1.f;
      if constexpr (FP8) {
        uint32_t mbits = 0;   // the largest |bf16| of the row, as its bit pattern
#pragma unroll 4
        for (int i = 0; i < 16; ++i) {
          const uint4 v = row_ok ? src[i] : make_uint4(0, 0, 0, 0);
          const uint32_t x[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
          for (int e = 0; e < 4; ++e)
            mbits = max(mbits, max(x[e] & 0x7FFFu, (x[e] >> 16) & 0x7FFFu));
        }
        // exponent of the max (bf16 keeps fp32's); none for a zero row
        const int ex = mbits >= 0x0080u ? static_cast<int>(mbits >> 7) - 127 : 0;
        const int qsh = min(max(14 - ex, -126), 126);
        qmul = __uint_as_float(static_cast<uint32_t>(127 + qsh) << 23);
        q_unscale = __uint_as_float(static_cast<uint32_t>(127 - qsh) << 23);
      }
#pragma unroll
      for (int i = 0; i < 16; ++i) {
        const uint4 v = row_ok ? src[i] : make_uint4(0, 0, 0, 0);
        const uint32_t x[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
        for (int e = 0; e < 4; ++e)   // FP8 caches: the scaled bf16 pair as an fp16 pair
          w[4 * i + e] = __uint_as_float(
              FP8 ? pack_f16(qmul * __uint_as_float(x[e] << 16),
                             qmul * __uint_as_float(x[e] & 0xFFFF0000u))
                  : x[e]);
      }
      tc_st32(tQ + lane_q, w);
      tc_st32(tQ + lane_q + 32, w + 32);
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_u32(&q_ready[t]));
    }
    const int qpos = ctx - n + tok0 + t * TQ + tl;      // this row's position
    const int last = p.causal ? qpos : ctx - 1;         // last key it sees
    const float sl2 = FP8 ? p.qk_scale_log2 * __ldg(p.k_scale + g) * q_unscale : p.qk_scale_log2;
    const bool pos_scale = sl2 > 0.f;
    uint8_t* pb = sm + LY::kP + t * LY::pbuf(FP8);
    float m = -CUDART_INF_F, l = 0.f;                   // m in scaled (log2) units
    bool alive = true;
    for (int j = 0; j < my_nt && alive; ++j) {
      const int k0 = j * kPfKeys;
      // S(j) ready implies the stage's copies landed; waiting on the stage's
      // barrier as well makes the producer's key mask for it visible here.
      if (!tc_wait(smem_u32(&s_full[t]), j & 1, abort_flag) ||
          !tc_wait(smem_u32(&full[j % STAGES]), (j / STAGES) & 1, abort_flag))
        alive = false;
      if (!__all_sync(0xffffffffu, alive)) break;
      const uint64_t vmask = key_mask[j % STAGES];
      // keys of this tile the row sees: those with cache data, up to `last`
      const int lim = last - k0 + 1;
      uint64_t rmask = lim >= kPfKeys ? ~0ull : (lim <= 0 ? 0ull : ((1ull << lim) - 1ull));
      rmask = row_ok ? (rmask & vmask) : 0ull;
      const bool dense = pos_scale && __all_sync(0xffffffffu, rmask == ~0ull);
      tc_fence_after();
      float sv[kPfKeys];
      pf_ld64(tS + lane_q, sv);
      tc_fence_before();
      __syncwarp();
      if ((lane & 31) == 0) mbar_arrive(smem_u32(&s_free[t]));
      float mt;
      if (dense) {   // warp-uniform: nothing masked; max of the raw logits, then scale
        static_assert(kPfKeys % 4 == 0, "two three-input max chains");
        float ma = sv[0], mb = sv[1];
#pragma unroll
        for (int c = 2; c + 3 < kPfKeys; c += 4) {
          ma = pf_max3(ma, sv[c], sv[c + 1]);
          mb = pf_max3(mb, sv[c + 2], sv[c + 3]);
        }
        mt = fmaxf(pf_max3(ma, sv[kPfKeys - 2], sv[kPfKeys - 1]), mb) * sl2;
      } else {
        const uint32_t mlo = static_cast<uint32_t>(rmask), mhi = static_cast<uint32_t>(rmask >> 32);
        float mx4[4] = {-CUDART_INF_F, -CUDART_INF_F, -CUDART_INF_F, -CUDART_INF_F};
#pragma unroll
        for (int c = 0; c < kPfKeys; ++c) {
          const bool ok = ((c < 32 ? mlo : mhi) >> (c & 31)) & 1u;
          sv[c] = ok ? sv[c] * sl2 : -CUDART_INF_F;
          mx4[c & 3] = fmaxf(mx4[c & 3], sv[c]);
        }
        mt = fmaxf(fmaxf(mx4[0], mx4[1]), fmaxf(mx4[2], mx4[3]));
      }
      float alpha = 1.f;
      bool resc = false;
      if (mt > m + 8.f) {
        if (m != -CUDART_INF_F) {
          alpha = pf_ex2(m - mt);
          resc = true;
        }
        m = mt;
      }
      const float mu = m == -CUDART_INF_F ? 0.f : m;   // rows with nothing seen yet: p = 0
      // Key pairs go through the packed fp32 pipe (fma / add .f32x2: each lane
      // rounds as the scalar op would); ls[i] holds the partial sums of keys
      // 4k + 2i and 4k + 2i + 1.
      const float2 nmu = make_float2(-mu, -mu);
      float2 ls[2] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f)};
      if (dense) {
        const float2 s2 = make_float2(sl2, sl2);
#pragma unroll
        for (int c = 0; c < kPfKeys; c += 2) {
          const float2 x = __ffma2_rn(make_float2(sv[c], sv[c + 1]), s2, nmu);
          sv[c] = pf_ex2(x.x);
          sv[c + 1] = pf_ex2(x.y);
          ls[(c >> 1) & 1] = __fadd2_rn(ls[(c >> 1) & 1], make_float2(sv[c], sv[c + 1]));
        }
      } else {
#pragma unroll
        for (int c = 0; c < kPfKeys; c += 2) {
          const float2 x = __fadd2_rn(make_float2(sv[c], sv[c + 1]), nmu);
          sv[c] = pf_ex2(x.x);   // 2^-inf = 0 for masked keys
          sv[c + 1] = pf_ex2(x.y);
          ls[(c >> 1) & 1] = __fadd2_rn(ls[(c >> 1) & 1], make_float2(sv[c], sv[c + 1]));
        }
      }
      l = l * alpha + ((ls[0].x + ls[0].y) + (ls[1].x + ls[1].y));
      // PV(j-1) must be finished before P is overwritten and before O is scaled
      if (j >= 1 && !tc_wait(smem_u32(&o_done[t]), (j - 1) & 1, abort_flag)) alive = false;
      if (!__all_sync(0xffffffffu, alive)) break;
      // P for the MMA.  16-bit caches: bf16 hi part, then what it left (about
      // 2^-17 relative together; bf16 alone would cost up to 2.7e-3 on N(0,1)
      // inputs against the 2e-3 bound).  8-bit caches: fp16 alone, as in the
      // decode kernels (2^-11 relative, within their 1e-2 bound by far).
#pragma unroll
      for (int u = 0; u < 8; ++u) {   // 8 keys per 16-byte chunk
        uint32_t wh[4], wl[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const float2 ab = make_float2(sv[8 * u + 2 * e], sv[8 * u + 2 * e + 1]);
          if constexpr (FP8) {
            wh[e] = pack_f16(ab.x, ab.y);
          } else {
            wh[e] = pack_bf16(ab.x, ab.y);
            const float2 hi =
                make_float2(__uint_as_float(wh[e] << 16), __uint_as_float(wh[e] & 0xFFFF0000u));
            const float2 lo = __ffma2_rn(hi, make_float2(-1.f, -1.f), ab);   // ab - hi, exact
            wl[e] = pack_bf16(lo.x, lo.y);
          }
        }
        *reinterpret_cast<uint4*>(pb + swz(r, u)) = make_uint4(wh[0], wh[1], wh[2], wh[3]);
        if constexpr (!FP8)
          *reinterpret_cast<uint4*>(pb + LY::kPPart + swz(r, u)) =
              make_uint4(wl[0], wl[1], wl[2], wl[3]);
      }
      if (__any_sync(0xffffffffu, resc)) {   // after P is out of the registers
        tc_fence_after();
#pragma unroll
        for (int c = 0; c < kPfD; c += 32) {
          float o[32];
          tc_ld32(tO + lane_q + c, o);
#pragma unroll
          for (int e = 0; e < 32; ++e) o[e] *= alpha;
          tc_st32(tO + lane_q + c, o);
        }
      }
      // V rows without cache data -> 0, once per key tile: by tile A's group
      // while it still needs this tile, else by tile B's; after the V copies
      // landed (a partly valid box also brings rows past the context)
      const bool zeroer = (t == 0) == (j < nt_a);
      if (zeroer && vmask != ~0ull &&
          !tc_wait(smem_u32(&full_v[j % STAGES]), (j / STAGES) & 1, abort_flag))
        alive = false;
      if (zeroer && alive && r < kPfKeys && !((vmask >> r) & 1ull)) {
        uint8_t* vrow = sm + kRing + (j % STAGES) * LY::kStage + 2 * LY::kKVHalf + r * 128;
#pragma unroll
        for (int u = 0; u < 8; ++u) {
          *reinterpret_cast<uint4*>(vrow + (u << 4)) = make_uint4(0, 0, 0, 0);
          *reinterpret_cast<uint4*>(vrow + LY::kKVHalf + (u << 4)) = make_uint4(0, 0, 0, 0);
        }
      }
      fence_proxy_async();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_u32(&p_full[t]));
    }
    // epilogue: this warp's O rows / l
    const bool ok = alive && my_nt > 0 &&
                    tc_wait(smem_u32(&o_done[t]), (my_nt - 1) & 1, abort_flag);
    if (__all_sync(0xffffffffu, ok)) {   // warp-uniform: the TMEM load is warp-wide
      tc_fence_after();
      // 1 / l, times the V scale for 8-bit caches
      const float vsc = FP8 ? __ldg(p.v_scale + g) : 1.f;
      const float inv = l > 0.f ? vsc / l : 0.f;
      float* orow = p.out + (static_cast<int64_t>(q0 + tok0 + t * TQ + tl) * p.num_q_heads +
                             g * G + r % G) * kPfD;
#pragma unroll
      for (int c = 0; c < kPfD; c += 32) {
        float o[32];
        tc_ld32(tO + lane_q + c, o);
        if (row_ok) {
#pragma unroll
          for (int e = 0; e < 32; e += 4)
            *reinterpret_cast<float4*>(orow + c + e) =
                make_float4(o[e] * inv, o[e + 1] * inv, o[e + 2] * inv, o[e + 3] * inv);
        }
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0)
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, 512;\n" ::"r"(tm) : "memory");
  if (tid == 0 && *abort_flag) flag_status(p.status, PKV_DEV_TIMEOUT);
}

}  // namespace pkv
