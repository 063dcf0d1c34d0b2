/*
 * pagedkv.h - C ABI of libpagedkv: a paged KV cache and PagedAttention decode
 * for one NVIDIA GB300 (sm_103a).
 *
 * Sources of the operations (web pages on LLM inference):
 *   [TUT]  "LLM inference tutorial" (xurj.top Tutorial/Detail/167)
 *          section 1.2 prefill and decode phases, 3.1 symmetric
 *          quantisation, 4.1 KVCache, 4.2 PagedAttention (class
 *          PagedKVCache, copy-on-write for beam search), 4.3 Prefix Caching
 *          (class PrefixCacheManager), 4.4 MHA/GQA/MQA, 6.2 chunked prefill.
 *   [NANO] "nano-vLLM architecture" (intelliparadigm 2014318), section 4.2
 *          PagedAttention (logical -> physical block mapping, attention that
 *          reads through the mapping), 4.3 memory-pool formula, 5 CUDA graph
 *          capture and replay with batch-size buckets and padding.
 *   [TGI]  "TGI architecture" (intelliparadigm 2004249), section 3.2 paged
 *          blocks of 128-256 tokens shared between requests; 5.1 CUDA graphs
 *          recorded for common batch sizes at warm-up.
 *   [TOPG] "ToPG framework" (intelliparadigm 2232463), section 2.3: KV pages
 *          managed LRU so contexts can exceed device memory; section 3.3: the
 *          KV cache stored compressed as FP8.
 *
 * Conventions for every call:
 *   - Host functions never abort; they return a pkv_status.
 *   - Device functions are asynchronous on the caller's stream: they validate
 *     their arguments on the host, launch, and return.  They never allocate,
 *     never synchronise, and report launch failures as PKV_ERR_CUDA.  Errors
 *     found on the device (a block id or slot out of range, a context longer
 *     than the block table) skip the offending access and OR a bit into the
 *     optional caller-owned device word `device_status` (PKV_DEV_* below).
 *   - All device buffers are owned by the caller and passed as device
 *     pointers; host buffers are owned by the caller and passed as host
 *     pointers.
 *   - A pool handle is not thread-safe: the caller serialises calls on it.
 *   - decode_graph_create is the one device-side call that allocates (graph
 *     objects, a private stream, a page-locked staging area) and synchronises;
 *     it is a set-up call.  decode_graph_step_host synchronises by design: it
 *     returns with the step's output in host memory.
 */
#ifndef PAGEDKV_H
#define PAGEDKV_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Same type as cudaStream_t; NULL means the legacy default stream. */
typedef struct CUstream_st* pkv_stream_t;

typedef enum {
  PKV_OK = 0,
  PKV_ERR_INVALID_ARG = 1,    /* null pointer, bad size, unknown sequence ... */
  PKV_ERR_NO_FREE_BLOCK = 2,  /* free list cannot cover the request [TUT 4.2] */
  PKV_ERR_BAD_BLOCK = 3,      /* block id outside [0, num_blocks) */
  PKV_ERR_REFCOUNT = 4,       /* ref or free of a block whose count is 0 */
  PKV_ERR_UNSUPPORTED = 5,    /* head_dim / block_size / dtype / group not built */
  PKV_ERR_CUDA = 6,           /* a CUDA runtime call or launch failed */
  PKV_ERR_HOST_MEMORY = 7,    /* host allocation failed */
  PKV_ERR_SCRATCH_LIMIT = 8   /* paged_attention_decode_noalloc: the request needs more
                                 than PKV_NOALLOC_SCRATCH_BYTES of split-KV scratch */
} pkv_status;

/* Bits a kernel ORs into *device_status (when that pointer is non-null). */
#define PKV_DEV_BAD_BLOCK 0x1     /* a block-table entry outside [0, num_blocks) */
#define PKV_DEV_BAD_SLOT 0x2      /* a slot >= num_blocks * block_size */
#define PKV_DEV_BAD_CONTEXT 0x4   /* context_lens[s] < 0 or > max_blocks_per_seq * block_size */
#define PKV_DEV_TIMEOUT 0x8       /* an asynchronous copy did not land within 2 s; the CTA
                                     stopped early and its output is not valid */

/* Element types.  INT8 is the tutorial's section 3.1 symmetric 8-bit code
 * (value = code * scale); FP8_E4M3 the OCP E4M3 code (value = e4m3 * scale). */
typedef enum { PKV_F32 = 0, PKV_BF16 = 1, PKV_FP8_E4M3 = 2, PKV_INT8 = 3 } pkv_dtype;

/* Human-readable name of a status (static string). */
const char* pkv_status_string(int32_t status);

/* ------------------------------------------------------------------------ */
/* Host block pool [TUT 4.2, 4.3; NANO 4.3].                                 */
/* ------------------------------------------------------------------------ */

typedef struct {
  int32_t num_layers;      /* layers sharing one block id (one view per layer) */
  int32_t num_kv_heads;
  int32_t head_dim;
  int32_t block_size;      /* tokens per block, > 0 */
  int32_t kv_dtype;        /* pkv_dtype of the cache elements */
  int64_t num_blocks;      /* physical blocks; 0 => free_bytes / block_bytes */
  int64_t free_bytes;      /* memory for the pool when num_blocks == 0 */
  /* Optional permutation of 0..num_blocks-1: the initial free-list order
   * (NULL => 0, 1, 2, ...).  Copied at init; not retained. */
  const int32_t* initial_free_order;
} pkv_pool_config;

typedef struct {
  int64_t total_blocks;
  int64_t used_blocks;     /* total - free */
  int64_t free_blocks;
  double utilization;      /* used / total * 100 [TUT 4.2 memory_usage] */
  int64_t block_bytes;     /* pkv_block_bytes() of the pool's config */
  int64_t total_bytes;     /* total_blocks * block_bytes */
  int64_t used_bytes;      /* used_blocks * block_bytes */
} pkv_pool_stats;

typedef struct pkv_pool pkv_pool;

/* Bytes of one physical block over all layers, K and V:
 * 2 * num_layers * block_size * num_kv_heads * head_dim * dtype_size
 * [NANO 4.3].  Returns -1 if cfg is NULL or a field is not positive. */
int64_t pkv_block_bytes(const pkv_pool_config* cfg);

/* Create a pool (host metadata only; the caller allocates the device cache,
 * one [num_blocks, block_size, num_kv_heads, head_dim] view per layer and per
 * K/V, as the pool tensor of [TUT 4.2]).  With num_blocks == 0 the pool gets
 * free_bytes / block_bytes blocks [NANO 4.3].  *out receives the handle.
 * INVALID_ARG for bad fields or a non-permutation free order. */
pkv_status kv_pool_init(const pkv_pool_config* cfg, pkv_pool** out);
void kv_pool_destroy(pkv_pool* pool);

/* Take the block at the FRONT of the free list (FIFO, [TUT 4.2] pop(0)) and
 * set its reference count to 1.  NO_FREE_BLOCK when the list is empty. */
pkv_status block_alloc(pkv_pool* pool, int32_t* block_id);
/* Share a block: count += 1 [TUT 4.3].  BAD_BLOCK / REFCOUNT (count 0). */
pkv_status block_ref(pkv_pool* pool, int32_t block_id);
/* Drop one reference; at 0 the block goes to the TAIL of the free list
 * [TUT 4.2 free_sequence].  BAD_BLOCK / REFCOUNT (already free). */
pkv_status block_free(pkv_pool* pool, int32_t block_id);
/* Current reference count of a block (0 = free). */
pkv_status block_refcount(const pkv_pool* pool, int32_t block_id, int32_t* count);
pkv_status kv_pool_stats(const pkv_pool* pool, pkv_pool_stats* out);
/* Copy the free list, front first, into out[0 .. cap); *n = its length.
 * INVALID_ARG if cap < *n (nothing beyond cap is written). */
pkv_status kv_pool_free_list(const pkv_pool* pool, int32_t* out, int64_t cap, int64_t* n);

/* Sequences.  seq_create takes one block at once and starts at length 0, as
 * allocate_sequence in [TUT 4.2]; INVALID_ARG if seq_id exists. */
pkv_status seq_create(pkv_pool* pool, int64_t seq_id);
/* New sequence dst sharing src's first ntok tokens, 1 <= ntok <= src's
 * length: the ceil(ntok / block_size) blocks holding them get one more
 * reference each [TUT 4.3].  A partly filled last block is shared too; the
 * first write into it by either sequence is copied on write (below).
 * ntok = src's length forks a whole beam [TUT 4.2, copy-on-write for beam
 * search]. */
pkv_status seq_fork_prefix(pkv_pool* pool, int64_t dst, int64_t src, int32_t ntok);
/* Append ONE token to each of n distinct sequences.  For the token at
 * position p: logical block p / block_size, offset p % block_size; a new block
 * is taken from the free list when that logical block is not in the table;
 * slot_mapping_out[i] = table[p / block_size] * block_size + p % block_size
 * [TUT 4.2 append_token].  Copy-on-write: when that block is in the table but
 * shared (reference count > 1), the sequence takes a new block from the
 * free-list front in its place, drops its reference on the shared one and a
 * (shared, new) pair is queued for pool_take_copies; the slot is in the new
 * block.  All-or-nothing: NO_FREE_BLOCK / INVALID_ARG leave the pool
 * unchanged.  slot_mapping_out is a host array of n int64. */
pkv_status seq_append_slots(pkv_pool* pool, const int64_t* seq_ids, int32_t n,
                            int64_t* slot_mapping_out);
/* Append n tokens to one sequence (a prompt).  Same rule and all-or-nothing
 * behaviour; slots_out (host, n int64) may be NULL. */
pkv_status seq_append_tokens(pkv_pool* pool, int64_t seq_id, int32_t n, int64_t* slots_out);
pkv_status seq_length(const pkv_pool* pool, int64_t seq_id, int32_t* len);
/* Copy a sequence's block table into out[0 .. cap); *nblocks = its length;
 * INVALID_ARG if cap < *nblocks. */
pkv_status seq_block_table(const pkv_pool* pool, int64_t seq_id, int32_t* out, int32_t cap,
                           int32_t* nblocks);
/* Batch view for a decode step: tables_out is a host [n, max_blocks] int32
 * row-major array (rows padded with -1), context_lens_out a host [n] int32
 * array of current lengths.  INVALID_ARG if a table is longer than
 * max_blocks. */
pkv_status seq_batch_tables(const pkv_pool* pool, const int64_t* seq_ids, int32_t n,
                            int32_t max_blocks, int32_t* tables_out, int32_t* context_lens_out);
/* Drop one reference on each block of the table, in table order (blocks that
 * reach 0 go to the free-list tail), and forget the sequence. */
pkv_status seq_free(pkv_pool* pool, int64_t seq_id);

/* Copy-on-write queue [TUT 4.2].  Writes the pending (source, destination)
 * block pairs, oldest first, to pairs[0 .. 2 * *n) and clears the queue;
 * *n = the number of pairs.  INVALID_ARG (queue kept) if cap < *n.  Drain it
 * after every call that appends and run copy_blocks on the pairs before the
 * device writes the appended tokens: within one such batch every destination
 * is a fresh block that is nobody's source. */
pkv_status pool_take_copies(pkv_pool* pool, int32_t* pairs, int32_t cap, int32_t* n);

/* Swap to host memory [TOPG 2.3: pages managed LRU, contexts beyond device
 * memory].  The pool's clock ticks on every seq_create, fork, append and
 * swap-in; a sequence's last tick orders it for eviction.
 *   kv_pool_host_init: a host swap area of num_host_blocks block slots (FIFO
 *     free list 0 .. n-1); once per pool.
 *   pool_lru_order: resident sequence ids, least recently used first, into
 *     seq_ids[0 .. cap); *n = their number (INVALID_ARG if cap < *n).
 *   seq_swap_out: every block of the sequence with reference count 1 moves to
 *     a host slot (front of the host free list; the device block goes to the
 *     free-list tail), in table order; shared blocks stay.  pairs[0 .. 2 *n)
 *     = (device block, host slot).  Copy them device -> host (swap_blocks)
 *     before the freed device blocks are written again.  All-or-nothing:
 *     NO_FREE_BLOCK if the host area is short; INVALID_ARG (nothing changed,
 *     *n = pairs needed) if cap < *n.
 *   seq_swap_in: every host block of a swapped-out sequence gets a device
 *     block from the free-list front; pairs = (host slot, device block); copy
 *     them host -> device before the sequence is read.  Same error rules.
 *   seq_is_swapped: 1 while the sequence is swapped out.
 * A swapped-out sequence refuses appends, forks, prefix inserts and batch
 * tables (INVALID_ARG); seq_free returns its host slots to the host free-list
 * tail. */
pkv_status kv_pool_host_init(pkv_pool* pool, int64_t num_host_blocks);
pkv_status pool_lru_order(const pkv_pool* pool, int64_t* seq_ids, int64_t cap, int64_t* n);
pkv_status seq_swap_out(pkv_pool* pool, int64_t seq_id, int32_t* pairs, int32_t cap, int32_t* n);
pkv_status seq_swap_in(pkv_pool* pool, int64_t seq_id, int32_t* pairs, int32_t cap, int32_t* n);
pkv_status seq_is_swapped(const pkv_pool* pool, int64_t seq_id, int32_t* swapped);

/* Prefix cache [TUT 4.3 PrefixCacheManager].  Entries are keyed by the token
 * ids themselves (host int32 arrays; a hash only speeds the search and a hit
 * is confirmed token by token).
 *   prefix_cache_insert: remember the blocks holding seq_id's first n tokens
 *     (ceil(n / block_size) of them; each gains a reference held by the
 *     cache) under tokens[0 .. n), with count 1 (cache_prefix).  INVALID_ARG
 *     if n < 1, n > the sequence's length or the prefix is already cached.
 *   prefix_cache_lookup: the longest cached prefix of tokens[0 .. n), trying
 *     lengths from n down (get_cached_prefix); *matched = its length (0 if
 *     none), *nblocks = its block count and, when blocks is not NULL, the
 *     blocks (INVALID_ARG if cap < *nblocks, count unchanged).  A hit adds one
 *     to the entry's count.
 *   seq_create_from_prefix: a new sequence seq_id starting with the longest
 *     cached prefix of tokens[0 .. n) (its blocks gain a reference, the
 *     entry's count one more; *matched its length), or a plain seq_create
 *     when nothing matches (*matched = 0).  A partly filled last block is
 *     copied on the first write into it.
 *   prefix_cache_release: one fewer on the entry cached for exactly
 *     tokens[0 .. n) (release_prefix); at zero the entry is dropped and its
 *     blocks lose the cache's reference.  INVALID_ARG if not cached.
 *   prefix_cache_count: that entry's count, 0 if not cached. */
pkv_status prefix_cache_insert(pkv_pool* pool, const int32_t* tokens, int32_t n, int64_t seq_id);
pkv_status prefix_cache_lookup(pkv_pool* pool, const int32_t* tokens, int32_t n,
                               int32_t* matched, int32_t* blocks, int32_t cap,
                               int32_t* nblocks);
pkv_status seq_create_from_prefix(pkv_pool* pool, int64_t seq_id, const int32_t* tokens,
                                  int32_t n, int32_t* matched);
pkv_status prefix_cache_release(pkv_pool* pool, const int32_t* tokens, int32_t n);
pkv_status prefix_cache_count(const pkv_pool* pool, const int32_t* tokens, int32_t n,
                              int32_t* count);

/* ------------------------------------------------------------------------ */
/* Device: cache append [TUT 4.2 append_token, write half; TOPG 3.3].        */
/* ------------------------------------------------------------------------ */

/* Write the K and V rows of num_tokens new tokens into one layer's cache.
 *   k_new, v_new  : device [num_tokens, num_kv_heads, head_dim], src_dtype.
 *   slot_mapping  : device [num_tokens] int64; token i goes to physical block
 *                   slot / block_size, offset slot % block_size.  A negative
 *                   slot skips the token; slot >= num_blocks * block_size is
 *                   skipped and flagged PKV_DEV_BAD_SLOT.
 *   k_cache, v_cache : device [num_blocks, block_size, num_kv_heads, head_dim],
 *                   cache_dtype.
 *   src_dtype == cache_dtype (f32 or bf16): the row bytes are copied.
 *   cache_dtype == FP8_E4M3 with src f32 or bf16: each element becomes
 *     E4M3(round-to-nearest-even, saturate to +-448)(float(x) / k_scale[h])
 *     with an IEEE float32 division [TUT 3.1 symmetric rule, qmax = 448];
 *     k_scale / v_scale are device [num_kv_heads] float32.
 *   cache_dtype == INT8 with src f32 or bf16: each element becomes
 *     clamp(round_half_even(float(x) / k_scale[h]), -128, 127), the quotient
 *     an IEEE float32 division, a NaN quotient 0 [TUT 3.1 symmetric_quantize,
 *     bits = 8].
 * Requirements: all buffers 16-byte aligned; head_dim * elem_size a multiple of
 * 16 bytes.  UNSUPPORTED for other dtype pairs. */
pkv_status reshape_and_cache(const void* k_new, const void* v_new, const int64_t* slot_mapping,
                             void* k_cache, void* v_cache, int32_t num_tokens,
                             int32_t num_kv_heads, int32_t head_dim, int32_t block_size,
                             int64_t num_blocks, int32_t src_dtype, int32_t cache_dtype,
                             const float* k_scale, const float* v_scale,
                             int32_t* device_status, pkv_stream_t stream);

/* ------------------------------------------------------------------------ */
/* Device: PagedAttention decode [NANO 4.2; TUT 4.2 get_kv + 4.4 forward].   */
/* ------------------------------------------------------------------------ */

/* Tokens per split-KV partition that paged_attention_decode uses for this
 * problem when its partition_tokens argument is 0 (a power of two in [256,
 * 4096] that depends on the current device's SM count, the group size
 * num_q_heads / num_kv_heads and the context length) on f32 and bf16 caches; FP8 and INT8 caches, whose rows are half the bytes, take
 * twice this, at most 4096.  A non-zero partition_tokens (a multiple of 64) is
 * returned as is.  Returns 0 on bad arguments (negative sizes, num_q_heads not
 * a multiple of num_kv_heads, partition_tokens not a multiple of 64). */
int32_t paged_attention_partition_tokens(int32_t num_seqs, int32_t num_q_heads,
                                         int32_t num_kv_heads, int32_t max_context_len,
                                         int32_t partition_tokens);

/* Device scratch that paged_attention_decode needs for its split-KV partials
 * (0 when every sequence fits one partition): num_seqs * num_q_heads *
 * ceil(max_context_len / P) * (head_dim + 2) * 4 bytes, P as above for a
 * 16-bit cache - enough for 8-bit caches too, whose automatic partitions are
 * longer. */
size_t paged_attention_workspace_bytes(int32_t num_seqs, int32_t num_q_heads,
                                       int32_t num_kv_heads, int32_t head_dim,
                                       int32_t max_context_len, int32_t partition_tokens);

/* One query token per sequence attends over its whole paged context.
 *   q            : device [num_seqs, num_q_heads, head_dim], q_dtype (f32|bf16).
 *   k_cache, v_cache : device [num_blocks, block_size, num_kv_heads, head_dim],
 *                  kv_dtype (f32|bf16|fp8_e4m3|int8); one layer's views.
 *   block_tables : device [num_seqs, max_blocks_per_seq] int32, row-major;
 *                  entry j of row s is the physical block of logical block j.
 *                  Entries at or beyond ceil(context_lens[s]/block_size) are
 *                  never used; the kernel may load some of them (always inside
 *                  the row) before it knows the context length, so the whole
 *                  row must be readable device memory, whatever it holds.
 *   context_lens : device [num_seqs] int32, tokens to attend (including the
 *                  token appended this step).  0 gives an output of 0.
 *   max_context_len : host upper bound of context_lens (sizes the grid).
 *   scale        : logit scale (1/sqrt(head_dim) in [TUT 4.4]).
 *   k_scale, v_scale : device [num_kv_heads] float32 dequant scales, FP8 and
 *                  INT8 only (value = float(code) * scale[kv_head]); else
 *                  ignored.
 *   out          : device [num_seqs, num_q_heads, head_dim] float32.
 *   workspace    : device scratch of workspace_bytes >=
 *                  paged_attention_workspace_bytes(...) (may be NULL when that
 *                  is 0); contents need not be initialised.
 *   partition_tokens : split-KV partition length in tokens (a multiple of 64,
 *                  or 0 = automatic).
 * Computes, for every sequence s and query head h with G = num_q_heads /
 * num_kv_heads and KV head g = h / G [TUT 4.4 repeat_interleave]:
 *   out[s,h,:] = sum_t softmax_t(scale * q[s,h,:] . K[s,t,g,:]) * V[s,t,g,:]
 * over t < context_lens[s], K/V gathered through the block table [TUT 4.2
 * get_kv], with float32 accumulation and a running (online) softmax.
 * Supported: head_dim in {64, 128, 256} with head_dim * kv_elem_size in
 * [64, 512] bytes; G in {1, 2, 4, 8}, and G up to 16 for bf16 and FP8 caches
 * with head_dim 128 (bf16 also 64) and block_size >= 8; block_size a power of
 * two in [1, 4096]; 16-byte aligned buffers.  UNSUPPORTED / INVALID_ARG
 * otherwise. */
pkv_status paged_attention_decode(const void* q, const void* k_cache, const void* v_cache,
                                  const int32_t* block_tables, const int32_t* context_lens,
                                  int32_t num_seqs, int32_t num_q_heads, int32_t num_kv_heads,
                                  int32_t head_dim, int32_t block_size, int64_t num_blocks,
                                  int32_t max_blocks_per_seq, int32_t max_context_len,
                                  float scale, int32_t q_dtype, int32_t kv_dtype,
                                  const float* k_scale, const float* v_scale, float* out,
                                  void* workspace, size_t workspace_bytes,
                                  int32_t partition_tokens, int32_t* device_status,
                                  pkv_stream_t stream);

/* Decode kernel choice, for tests and profiles.  paged_attention_decode and
 * paged_attention_decode_append pick one kernel by shape: the transposed
 * mma.sync kernel for G <= 8 or G = 16 (two CTAs of 8 heads per KV head;
 * bf16 head_dim 64 / 128 / 256, 8-bit head_dim 128, block_size >= 8), else the
 * heads-as-rows mma.sync kernel (bf16 head_dim 64 / 128, FP8 head_dim 128,
 * G <= 16, block_size >= 8), else the CUDA-core kernel.  pkv_test_force_decode_kernel(k) makes every later call in the
 * process skip to kernel k where k supports the shape (falling back down the
 * same order where it does not); PKV_DECODE_KERNEL_AUTO restores the choice
 * by shape.  It exists so that tests can run every kernel on the same inputs.
 * The setting is process-wide: calls racing with a change may take either
 * kernel.  An unknown value returns INVALID_ARG and changes nothing.  Not a
 * paged-attention operation of the source pages. */
typedef enum {
  PKV_DECODE_KERNEL_AUTO = 0,
  PKV_DECODE_KERNEL_HEADS_AS_ROWS = 1,
  PKV_DECODE_KERNEL_CUDA_CORE = 2
} pkv_decode_kernel;
pkv_status pkv_test_force_decode_kernel(int32_t kernel);

/* Test of the bounded device waits, not a paged-attention operation of the
 * source pages.  pkv_test_decode_stall(bytes) with bytes > 0 makes every
 * later launch of the transposed decode kernel (chosen for G <= 8 and 16)
 * arm one barrier phase - warp 0, first stage, CTA (sequence 0, KV head 0,
 * partition 0) - for `bytes` more than its copies bring, before issuing them.
 * The copies land, the phase never completes, and after the 2 s bound the
 * warp flags PKV_DEV_TIMEOUT in device_status, waits (bounded) for its other
 * copies in flight and leaves its share out of the output; the call itself
 * returns PKV_OK and the context stays usable.  bytes = 0 restores normal
 * launches.  bytes must be a multiple of 16 and at most 65536, else
 * INVALID_ARG.  Process-wide, like pkv_test_force_decode_kernel. */
pkv_status pkv_test_decode_stall(uint32_t bytes);

/* One decode step with the append fused in: the same as
 *   reshape_and_cache(k_new, v_new, slot_mapping, k_cache, v_cache, num_seqs, ...)
 *   paged_attention_decode(q, k_cache, v_cache, ...)
 * on the same stream [TUT 4.2 append_token, then 4.4 forward], for one new
 * token per sequence: k_new / v_new are device [num_seqs, num_kv_heads,
 * head_dim] of src_dtype (f32|bf16; equal to kv_dtype for f32 / bf16
 * caches), slot_mapping device [num_seqs] int64.  slot_mapping[s] must be the
 * slot of position context_lens[s] - 1 (the appended token is the last one
 * attended), or negative for no append.
 * Where the transposed tensor-core kernel runs on a bf16 cache (head_dim 64
 * or 128, G <= 8, block_size >= 8), that kernel copies each sequence's new
 * row for its KV head into the cache before it reads the block, in the same
 * launch.  A slot that is not the block table's slot for position
 * context_lens[s] - 1 (or a context of 0 with a slot) is then not written and
 * flags PKV_DEV_BAD_SLOT, and the attention reads the cache as it was.
 * Elsewhere (8-bit caches, whose quantisation stays in the append kernel, and
 * the other decode kernels) the call runs the two kernels in order.
 * Arguments and errors otherwise as the two calls'. */
pkv_status paged_attention_decode_append(
    const void* q, const void* k_new, const void* v_new, const int64_t* slot_mapping,
    int32_t src_dtype, void* k_cache, void* v_cache, const int32_t* block_tables,
    const int32_t* context_lens, int32_t num_seqs, int32_t num_q_heads, int32_t num_kv_heads,
    int32_t head_dim, int32_t block_size, int64_t num_blocks, int32_t max_blocks_per_seq,
    int32_t max_context_len, float scale, int32_t q_dtype, int32_t kv_dtype, const float* k_scale,
    const float* v_scale, float* out, void* workspace, size_t workspace_bytes,
    int32_t partition_tokens, int32_t* device_status, pkv_stream_t stream);

/* Copy-on-write block copies [TUT 4.2]: for each (src, dst) pair of
 * pairs[0 .. 2n) (device int32), every plane's block dst becomes a copy of its
 * block src.  A plane is one (layer, K or V) slice of the pool tensor
 * [num_layers, 2, num_blocks, block_size, num_kv_heads, head_dim]:
 * plane i's block b starts at base + i * plane_stride_bytes + b * block_bytes,
 * so the whole pool has num_planes = 2 * num_layers, plane_stride_bytes =
 * num_blocks * block_bytes and block_bytes = block_size * num_kv_heads *
 * head_dim * element size.  Destinations must be distinct and no destination
 * may be another pair's source (true of one pool_take_copies batch); pairs
 * that share a source are best placed side by side, so its re-reads hit L2.  Pairs
 * with an id outside [0, num_blocks) are skipped and flagged
 * PKV_DEV_BAD_BLOCK.  base 16-byte aligned; block_bytes and
 * plane_stride_bytes multiples of 16. */
pkv_status copy_blocks(void* base, int32_t num_planes, int64_t plane_stride_bytes,
                       int64_t block_bytes, int64_t num_blocks, const int32_t* pairs, int32_t n,
                       int32_t* device_status, pkv_stream_t stream);

/* Swap copies [TOPG 2.3]: for each pair of pairs[0 .. 2n) (device int32),
 * with to_host = 1 (device block, host slot): host slot <- every plane's
 * block; with to_host = 0 (host slot, device block): every plane's block <-
 * host slot.  Planes as in copy_blocks.  host is page-locked host memory
 * (cudaHostAlloc / pinned) of num_host_blocks slots, slot h holding
 * [num_planes][block_bytes] at host + h * num_planes * block_bytes; the
 * kernel reads and writes it directly over the host link.  Ids outside
 * [0, num_blocks) or [0, num_host_blocks) are skipped and flagged
 * PKV_DEV_BAD_BLOCK.  INVALID_ARG if host is not page-locked memory the
 * device can address. */
pkv_status swap_blocks(void* base, int32_t num_planes, int64_t plane_stride_bytes,
                       int64_t block_bytes, int64_t num_blocks, void* host,
                       int64_t num_host_blocks, const int32_t* pairs, int32_t n, int32_t to_host,
                       int32_t* device_status, pkv_stream_t stream);

/* Paged prefill attention: a chunk of query tokens per sequence attends,
 * causally, over the sequence's whole paged context ("LLM inference tutorial"
 * section 1.2 prefill phase; section 6.2 chunked prefill; section 4.4 MHA/GQA
 * forward).  The chunk's K/V rows must already be in the cache
 * (reshape_and_cache), so the chunk is the LAST n_s tokens of the context.
 *   q            : device [num_tokens, num_q_heads, 128] bf16; the chunks of all
 *                  sequences back to back.
 *   query_start  : device [num_seqs + 1] int32, non-decreasing, query_start[0]
 *                  = 0 and query_start[num_seqs] <= num_tokens; sequence s owns
 *                  rows query_start[s] .. query_start[s+1]-1 (n_s of them, 0
 *                  allowed) of q and out.
 *   k_cache, v_cache : device [num_blocks, block_size, num_kv_heads, 128],
 *                  kv_dtype bf16, fp8_e4m3 or int8.
 *   k_scale, v_scale : device [num_kv_heads] float32 dequant scales for an FP8
 *                  or INT8 cache (value = code * scale[kv_head], as in
 *                  decode); else ignored.
 *   block_tables : device [num_seqs, max_blocks_per_seq] int32 (as in decode).
 *   context_lens : device [num_seqs] int32, the context INCLUDING the chunk;
 *                  n_s <= context_lens[s] <= max_context_len.
 *   max_query_len : host upper bound of n_s (sizes the grid).
 *   causal       : 1 - query token i of sequence s (position
 *                  context_lens[s] - n_s + i) sees keys 0 .. its position;
 *                  0 - it sees all context_lens[s] keys.
 *   out          : device [num_tokens, num_q_heads, 128] float32; rows outside
 *                  every chunk are not written.
 * Computes out[query_start[s]+i, h, :] = softmax(scale * q . K_g^T) V_g over
 * the visible keys, g = h / G, with float32 accumulation.  Runs on tcgen05
 * tensor cores (Q K^T and P V with P carried as bf16 hi + lo parts).  FP8 and
 * INT8 tiles are widened to fp16 in shared memory (exact), so the
 * contractions run in fp16 (each q row scaled by a power of two into fp16's
 * range, P as one fp16 value, as in decode), the K scale folded into the
 * logit scale and the V scale into the output.
 * Supported: head_dim 128, bf16 q, bf16, FP8-E4M3 or INT8 caches (8-bit
 * caches need both scales), G = num_q_heads / num_kv_heads
 * <= 16, block_size a power of two in [8, 4096], 16-byte aligned q, caches and
 * out.  Device-side problems (a bad query_start or context, a bad block) are
 * flagged in device_status; bad rows are skipped or zeroed. */
pkv_status paged_attention_prefill(const void* q, const int32_t* query_start,
                                   const void* k_cache, const void* v_cache,
                                   const int32_t* block_tables, const int32_t* context_lens,
                                   int32_t num_seqs, int32_t num_tokens, int32_t max_query_len,
                                   int32_t num_q_heads, int32_t num_kv_heads, int32_t head_dim,
                                   int32_t block_size, int64_t num_blocks,
                                   int32_t max_blocks_per_seq, int32_t max_context_len,
                                   float scale, int32_t causal, int32_t q_dtype,
                                   int32_t kv_dtype, const float* k_scale,
                                   const float* v_scale, float* out, int32_t* device_status,
                                   pkv_stream_t stream);

/* ------------------------------------------------------------------------ */
/* CUDA-graph decode step with batch-size buckets and padding.               */
/* ------------------------------------------------------------------------ */
/* A whole decode step - for every layer, reshape_and_cache of the new token
 * then paged_attention_decode - is captured once per batch-size bucket into a
 * CUDA graph over fixed device buffers, and replayed; a batch of B sequences
 * runs the smallest bucket >= B, its rows B .. bucket-1 padded as context 0
 * (output 0) and slot -1 (no append) [NANO 5.1 record and replay, 5.2
 * buckets: pick the nearest larger bucket, pad to it; TGI 5.1 graphs
 * recorded for common batch sizes].  The buffer layout below is this
 * library's own.
 * Buffers (device, caller-owned, sized for the largest bucket Bmax):
 *   q            : [num_layers][Bmax][num_q_heads][head_dim], q_dtype.
 *   k_new, v_new : [num_layers][Bmax][num_kv_heads][head_dim], src_dtype.
 *   slot_mapping : [Bmax] int64; block_tables [Bmax][max_blocks_per_seq]
 *                  int32; context_lens [Bmax] int32 (shared by all layers).
 *   out          : [num_layers][Bmax][num_q_heads][head_dim] float32.
 *   workspace    : >= paged_attention_workspace_bytes(Bmax, num_q_heads,
 *                  num_kv_heads, head_dim, max_blocks_per_seq * block_size, 0).
 *   k_caches, v_caches : HOST arrays of num_layers device pointers, each a
 *                  [num_blocks, block_size, num_kv_heads, head_dim] view.
 *   k_scales, v_scales : HOST arrays of num_layers device [num_kv_heads]
 *                  float32 pointers (8-bit caches; else NULL).
 * The graphs keep every pointer; the caller writes a step's inputs into the
 * buffers before decode_graph_launch and reads out after it.  Partitions are
 * sized for a context of max_blocks_per_seq * block_size. */
typedef struct {
  int32_t num_layers, num_q_heads, num_kv_heads, head_dim, block_size;
  int64_t num_blocks;
  int32_t max_blocks_per_seq;
  int32_t q_dtype, kv_dtype, src_dtype;
  float scale;
  void* const* k_caches;
  void* const* v_caches;
  const float* const* k_scales;
  const float* const* v_scales;
  void* q;
  void* k_new;
  void* v_new;
  int64_t* slot_mapping;
  int32_t* block_tables;
  int32_t* context_lens;
  float* out;
  void* workspace;
  size_t workspace_bytes;
  int32_t* device_status;
  const int32_t* buckets;   /* host, ascending batch sizes; the last is Bmax */
  int32_t num_buckets;
} pkv_decode_graph_config;

typedef struct pkv_decode_graph pkv_decode_graph;

/* Captures one graph per bucket on a private stream of the current device.
 * Before capturing, it runs each bucket's step once with every row padded
 * (nothing is appended, so no cache changes) to load the kernels; this
 * overwrites slot_mapping and context_lens.  Returns INVALID_ARG /
 * UNSUPPORTED for arguments paged_attention_decode would refuse, CUDA if a
 * capture fails. */
pkv_status decode_graph_create(const pkv_decode_graph_config* cfg, pkv_decode_graph** out);
/* Replays the step for a batch of 1 .. Bmax sequences on stream: pads rows
 * batch .. bucket-1 (context 0, slot -1), then launches the bucket's graph.
 * *bucket_out (nullable) receives the bucket used. */
pkv_status decode_graph_launch(pkv_decode_graph* g, int32_t batch, int32_t* bucket_out,
                               pkv_stream_t stream);
void decode_graph_destroy(pkv_decode_graph* g);
/* One decode step from host memory: the whole step a caller makes per token.
 * Builds the batch's block tables and lengths from the pool into a
 * page-locked staging area the graph owns, copies them and the step's inputs
 * to the graph's buffers (one cudaMemcpyAsync or cudaMemcpy2DAsync per
 * buffer), replays the bucket's graph, copies the output back and waits for
 * the stream.
 *   seq_ids   : host [batch] int64, resident sequences whose tables fit
 *               max_blocks_per_seq.
 *   q_host    : host [num_layers][batch][num_q_heads][head_dim], q_dtype.
 *   k_new_host, v_new_host : host [num_layers][batch][num_kv_heads][head_dim],
 *               src_dtype.
 *   slots_host: host [batch] int64, the slots of the step's tokens
 *               (seq_append_slots; the pool's lengths already include them).
 *   out_host  : host [num_layers][batch][num_q_heads][head_dim] float32.
 * Page-locked host buffers make the copies asynchronous; pageable ones work
 * but are staged by the CUDA driver.  Returns INVALID_ARG for a bad batch, an
 * unknown or swapped-out sequence or a table longer than max_blocks_per_seq,
 * CUDA if a copy or the launch fails. */
pkv_status decode_graph_step_host(pkv_decode_graph* g, const pkv_pool* pool,
                                  const int64_t* seq_ids, int32_t batch, const void* q_host,
                                  const void* k_new_host, const void* v_new_host,
                                  const int64_t* slots_host, float* out_host,
                                  pkv_stream_t stream);

/* Size of the device scratch compiled into the library for
 * paged_attention_decode_noalloc (held on every GPU that loads the library,
 * until the process exits). */
#define PKV_NOALLOC_SCRATCH_BYTES (16u * 1024u * 1024u)

/* paged_attention_decode for callers that cannot allocate device memory.
 * The source pages have no counterpart of this call; it exists for code that
 * may not call cudaMalloc or any allocating routine - a plug-in inside a host
 * program that owns every device allocation, a runtime that plans all of its
 * memory once at start-up and forbids allocation on the per-token path, or a
 * caller that cannot afford the device-wide synchronisation an allocation can
 * cause.  Arguments and results are those of paged_attention_decode without
 * the workspace: the split-KV partials go to a fixed device array inside the
 * library, PKV_NOALLOC_SCRATCH_BYTES long.  The call allocates nothing.
 *   - A request whose partials need more than PKV_NOALLOC_SCRATCH_BYTES
 *     (paged_attention_workspace_bytes(...) of the same arguments) returns
 *     PKV_ERR_SCRATCH_LIMIT without launching anything.
 *   - All calls on a device share that array.  Calls whose kernels may overlap
 *     on the GPU (different streams with no ordering between them) race on it
 *     and can corrupt each other's outputs; calls on one stream are safe.
 *   - The array keeps the previous call's contents; nothing in it needs to
 *     start at zero, since a call writes every partial before reading it.
 *   - The first call on each device looks up the array's device address (with
 *     that device current) and caches it, keyed by the unique id of the
 *     device's current context; make that first call before any stream
 *     capture begins.  A call that finds a different context (the previous
 *     one was destroyed, e.g. by cudaDeviceReset) looks the address up again,
 *     so after such a reset, too, call once before capturing. */
pkv_status paged_attention_decode_noalloc(
    const void* q, const void* k_cache, const void* v_cache, const int32_t* block_tables,
    const int32_t* context_lens, int32_t num_seqs, int32_t num_q_heads, int32_t num_kv_heads,
    int32_t head_dim, int32_t block_size, int64_t num_blocks, int32_t max_blocks_per_seq,
    int32_t max_context_len, float scale, int32_t q_dtype, int32_t kv_dtype, const float* k_scale,
    const float* v_scale, float* out, int32_t partition_tokens, int32_t* device_status,
    pkv_stream_t stream);

/* ------------------------------------------------------------------------ */
/* Device: bandwidth reference kernels (the roofline denominators).          */
/* ------------------------------------------------------------------------ */

/* dst[0 .. bytes) = src[0 .. bytes) with 16-byte vector loads/stores; bytes a
 * multiple of 16, both pointers 16-byte aligned. */
pkv_status pkv_copy_kernel(const void* src, void* dst, size_t bytes, pkv_stream_t stream);
/* Reads src[0 .. bytes) with 16-byte loads and writes one float per CTA of a
 * checksum into sink (device, >= pkv_read_kernel_sink_floats() floats). */
pkv_status pkv_read_kernel(const void* src, size_t bytes, float* sink, pkv_stream_t stream);
int32_t pkv_read_kernel_sink_floats(void);

#ifdef __cplusplus
}
#endif

#endif /* PAGEDKV_H */
