"""Seeded synthetic inputs shared by the tests, the bench and the oracle checks.

This module holds input recipes only - shapes, seeds, context-length laws,
initial free-list permutations and random values - and none of the method's
arithmetic: no slot computation, no block tables, no attention, no FP8
encoding.  Both the CUDA library and the oracle consume what it produces.

The five workloads are decode steps shaped like the pages' LLaMA-7B / 70B
examples ("LLM inference tutorial" sections 4.1-4.4: 7B = 32 layers x 32 heads
x 128, 70B = 64 query heads / 8 KV heads x 128; "TGI architecture" section
3.2: blocks of 128-256 tokens; "nano-vLLM architecture" section 4.3 pool
formula).  No dataset is involved; these stand in for the pages' ShareGPT-style
benchmark traffic.
"""
from __future__ import annotations

import math
from dataclasses import dataclass

import numpy as np

F32, BF16, FP8, INT8 = "f32", "bf16", "fp8_e4m3", "int8"
ELEM_BYTES = {F32: 4, BF16: 2, FP8: 1, INT8: 1}


@dataclass(frozen=True)
class DecodeWorkload:
    name: str
    num_seqs: int
    num_q_heads: int
    num_kv_heads: int
    head_dim: int
    block_size: int
    kv_dtype: str
    q_dtype: str
    seed: int
    num_layers: int = 1
    ctx_law: str = "uniform"          # "fixed" | "uniform" | "lognormal"
    ctx_fixed: tuple = ()
    ctx_lo: int = 1
    ctx_hi: int = 1
    lognormal_median: float = 1024.0
    lognormal_sigma: float = 1.0
    pool_slack: float = 1.5
    fixed_num_blocks: int = 0         # overrides the slack sizing when > 0
    k_head_scale: tuple = ()          # (lo, hi): K of head g scaled by linspace
    prefix_tokens: int = 0            # shared prompt prefix (whole blocks)
    prefix_seqs: int = 0              # sequences 0 .. prefix_seqs-1 share it
    graph: bool = False               # time the step as a replayed CUDA graph

    @property
    def group(self) -> int:
        return self.num_q_heads // self.num_kv_heads

    @property
    def scale(self) -> float:
        """Logit scale 1/sqrt(head_dim) as float32 (section 4.4 forward)."""
        return float(np.float32(1.0 / math.sqrt(self.head_dim)))


TINY = DecodeWorkload("tiny_fp32_mha", 2, 4, 4, 64, 16, F32, F32, seed=0,
                      ctx_law="fixed", ctx_fixed=(37, 70), fixed_num_blocks=16)
LLAMA7B_LAYER = DecodeWorkload("llama7b_layer_bf16", 32, 32, 32, 128, 16, BF16, BF16,
                               seed=1, ctx_lo=512, ctx_hi=4096)
LLAMA70B_GQA = DecodeWorkload("llama70b_gqa8_bf16", 64, 64, 8, 128, 128, BF16, BF16,
                              seed=2, ctx_lo=1024, ctx_hi=8192)
LONG_CTX = DecodeWorkload("long_ctx_splitkv_bf16", 8, 32, 8, 128, 256, BF16, BF16,
                          seed=3, ctx_lo=32768, ctx_hi=131072, k_head_scale=(1.0, 4.5))
RAGGED_FP8 = DecodeWorkload("ragged_32layer_fp8", 256, 32, 32, 128, 16, FP8, BF16,
                            seed=4, num_layers=32, ctx_law="lognormal", ctx_lo=1,
                            ctx_hi=16384, pool_slack=1.25, prefix_tokens=2048,
                            prefix_seqs=128)
ALL = (TINY, LLAMA7B_LAYER, LLAMA70B_GQA, LONG_CTX, RAGGED_FP8)
# One layer of the ragged FP8 step (same per-layer shape; a few GB on the device),
# for profiling runs.
RAGGED_FP8_LAYER = DecodeWorkload("ragged_fp8_1layer", 256, 32, 32, 128, 16, FP8, BF16,
                                  seed=4, num_layers=1, ctx_law="lognormal", ctx_lo=1,
                                  ctx_hi=16384, pool_slack=1.25, prefix_tokens=2048,
                                  prefix_seqs=128)
# The 7B layer with an INT8 cache (section 3.1 symmetric codes, per-head scale).
LLAMA7B_LAYER_INT8 = DecodeWorkload("llama7b_layer_int8", 32, 32, 32, 128, 16, INT8, BF16,
                                    seed=1, ctx_lo=512, ctx_hi=4096)
# The same layer with an FP8-E4M3 cache: the in-register dequantisation measured
# on plain (unshared) contexts.
LLAMA7B_LAYER_FP8 = DecodeWorkload("llama7b_layer_fp8", 32, 32, 32, 128, 16, FP8, BF16,
                                   seed=1, ctx_lo=512, ctx_hi=4096)
# Small-batch decode of all 32 layers of the 7B shape with short contexts, where
# launch cost matters: timed as a CUDA-graph replay (and eagerly, for contrast).
LLAMA7B_B8_GRAPH = DecodeWorkload("llama7b_32layer_b8_graph", 8, 32, 32, 128, 16, BF16, BF16,
                                  seed=9, num_layers=32, ctx_lo=256, ctx_hi=1024, graph=True)
# The 70B-shaped layer with 16 query heads per KV head (128 over 8, as in 405B-class
# models): the transposed kernel runs it as two CTAs of 8 heads per KV head.
GQA16_LAYER = DecodeWorkload("gqa16_128q_8kv_bf16", 64, 128, 8, 128, 128, BF16, BF16,
                             seed=2, ctx_lo=1024, ctx_hi=8192)
# The 7B layer's contexts with head_dim 256 and 2 query heads per KV head (16 over 8).
D256_LAYER = DecodeWorkload("d256_gqa2_bf16", 32, 16, 8, 256, 16, BF16, BF16,
                            seed=1, ctx_lo=512, ctx_hi=4096)
EXTRA = (RAGGED_FP8_LAYER, LLAMA7B_LAYER_INT8, LLAMA7B_LAYER_FP8, LLAMA7B_B8_GRAPH, GQA16_LAYER,
         D256_LAYER)


@dataclass(frozen=True)
class PrefillWorkload:
    """One chunked-prefill step ("LLM inference tutorial" section 6.2: prompts
    cut into chunks of ``chunk_size`` = 512 tokens, at most ``max_batch_tokens``
    = 8192 tokens per batch).  Every sequence brings one chunk of
    ``chunk_tokens`` new tokens; its earlier chunks (``chunk_tokens`` x
    U{0 .. max_prefix_chunks}) are already in the cache."""
    name: str
    num_seqs: int
    chunk_tokens: int
    max_prefix_chunks: int
    num_q_heads: int
    num_kv_heads: int
    head_dim: int
    block_size: int
    seed: int
    kv_dtype: str = BF16
    q_dtype: str = BF16
    num_layers: int = 1
    pool_slack: float = 1.5
    chunk_fixed: tuple = ()           # per-sequence chunk lengths (small cases)
    prefix_fixed: tuple = ()          # per-sequence cached prefix lengths

    @property
    def group(self) -> int:
        return self.num_q_heads // self.num_kv_heads

    @property
    def scale(self) -> float:
        return float(np.float32(1.0 / math.sqrt(self.head_dim)))


# 7B-shaped layer (32 heads x 128): 16 sequences x 512-token chunks = 8192 tokens.
PREFILL_7B = PrefillWorkload("chunked_prefill_7b_bf16", 16, 512, 7, 32, 32, 128, 16, seed=5)
# 70B-shaped GQA layer (64 query / 8 KV heads), blocks of 128 tokens, prompts to 8192.
PREFILL_70B = PrefillWorkload("chunked_prefill_70b_gqa8_bf16", 16, 512, 15, 64, 8, 128, 128,
                              seed=6)
# Small ragged case the oracle finishes in seconds.
PREFILL_TINY = PrefillWorkload("tiny_prefill_bf16", 3, 0, 0, 8, 2, 128, 16, seed=7,
                               chunk_fixed=(5, 130, 64), prefix_fixed=(0, 37, 300))
# The 7B-shaped step with an FP8-E4M3 cache (tiles widened to fp16 in the kernel).
PREFILL_7B_FP8 = PrefillWorkload("chunked_prefill_7b_fp8", 16, 512, 7, 32, 32, 128, 16, seed=5,
                                 kv_dtype=FP8)
# The same step with an INT8 cache (section 3.1 symmetric codes, per-head scales).
PREFILL_7B_INT8 = PrefillWorkload("chunked_prefill_7b_int8", 16, 512, 7, 32, 32, 128, 16, seed=5,
                                  kv_dtype=INT8)
PREFILL = (PREFILL_TINY, PREFILL_7B, PREFILL_70B, PREFILL_7B_FP8, PREFILL_7B_INT8)


def prefill_lens(w: PrefillWorkload):
    """(chunk lengths, context lengths after the chunk) per sequence."""
    if w.chunk_fixed:
        n = np.asarray(w.chunk_fixed, dtype=np.int64)
        pre = np.asarray(w.prefix_fixed, dtype=np.int64)
    else:
        n = np.full(w.num_seqs, w.chunk_tokens, dtype=np.int64)
        pre = w.chunk_tokens * rng(w.seed, 1).integers(0, w.max_prefix_chunks + 1,
                                                       size=w.num_seqs).astype(np.int64)
    return n, pre + n


def prefill_num_blocks(w: PrefillWorkload, ctx: np.ndarray) -> int:
    return int(math.ceil(w.pool_slack * int(np.maximum(1, -(-ctx // w.block_size)).sum())))


def rng(seed: int, stream: int = 0) -> np.random.Generator:
    """PCG64 generator for (workload seed, sub-stream)."""
    return np.random.default_rng([seed, stream])


def context_lens(w: DecodeWorkload) -> np.ndarray:
    """Context length of each sequence AFTER this step's appended token."""
    r = rng(w.seed, 1)
    if w.ctx_law == "fixed":
        return np.asarray(w.ctx_fixed, dtype=np.int64)
    if w.ctx_law == "uniform":
        return r.integers(w.ctx_lo, w.ctx_hi + 1, size=w.num_seqs).astype(np.int64)
    if w.ctx_law == "lognormal":
        x = np.exp(r.normal(math.log(w.lognormal_median), w.lognormal_sigma, w.num_seqs))
        lens = np.clip(np.rint(x), w.ctx_lo, w.ctx_hi).astype(np.int64)
        if w.prefix_tokens:
            # sharers: prefix + own suffix (at least 1 token), total <= ctx_hi
            suf = np.clip(lens[: w.prefix_seqs], 1, w.ctx_hi - w.prefix_tokens)
            lens[: w.prefix_seqs] = w.prefix_tokens + suf
        return lens
    raise ValueError(w.ctx_law)


def blocks_needed(w: DecodeWorkload, lens: np.ndarray) -> int:
    """Physical blocks the workload occupies (prefix blocks counted once).

    Each sequence holds ceil(len / block_size) blocks (at least one), and a
    sharer's prefix blocks are the owner's.
    """
    bs = w.block_size
    per = np.maximum(1, -(-lens // bs))
    n = int(per.sum())
    if w.prefix_tokens:
        n -= (w.prefix_tokens // bs) * w.prefix_seqs
        n += w.prefix_tokens // bs          # the owner's copy
    return n


def num_blocks(w: DecodeWorkload, lens: np.ndarray) -> int:
    if w.fixed_num_blocks:
        return w.fixed_num_blocks
    return int(math.ceil(w.pool_slack * blocks_needed(w, lens)))


def free_order(w: DecodeWorkload, nblocks: int) -> np.ndarray:
    """Seeded initial free-list permutation (blocks handed out shuffled)."""
    return rng(w.seed, 2).permutation(nblocks).astype(np.int32)


def normal_f32(seed: int, stream: int, shape) -> np.ndarray:
    return rng(seed, stream).standard_normal(shape, dtype=np.float32)


def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Store float32 values as bfloat16 (round to nearest even), as uint16 bits.

    This is how synthetic inputs are stored, not a step of the method.
    """
    b = np.asarray(x, dtype=np.float32).view(np.uint32).astype(np.uint64)
    nan = np.isnan(np.asarray(x, dtype=np.float32))
    r = (b + 0x7FFF + ((b >> 16) & 1)) >> 16
    r = r.astype(np.uint16)
    r[nan] = 0x7FC0
    return r


def store(x_f32: np.ndarray, dtype: str) -> np.ndarray:
    """Synthetic float32 values in the storage type of q / k_new / v_new."""
    if dtype == F32:
        return np.asarray(x_f32, dtype=np.float32)
    if dtype == BF16:
        return f32_to_bf16_bits(x_f32)
    raise ValueError(dtype)


def k_head_scales(w: DecodeWorkload) -> np.ndarray:
    """Per-KV-head multiplier of K (long-context logits spanning about +-20)."""
    if not w.k_head_scale:
        return np.ones(w.num_kv_heads, dtype=np.float32)
    lo, hi = w.k_head_scale
    return np.linspace(lo, hi, w.num_kv_heads).astype(np.float32)


def fp8_scale_from_absmax(absmax: np.ndarray) -> np.ndarray:
    """Static per-head FP8 scale absmax / 448 (symmetric rule, qmax = 448)."""
    a = np.asarray(absmax, dtype=np.float32)
    return np.where(a > 0, a / np.float32(448.0), np.float32(1.0)).astype(np.float32)


def int8_scale_from_absmax(absmax: np.ndarray) -> np.ndarray:
    """Static per-head INT8 scale absmax / 127 (section 3.1 symmetric rule,
    qmax = 2^7 - 1)."""
    a = np.asarray(absmax, dtype=np.float32)
    return np.where(a > 0, a / np.float32(127.0), np.float32(1.0)).astype(np.float32)


@dataclass(frozen=True)
class ForkWorkload:
    """Beam search over a pool ("LLM inference tutorial" section 4.2: blocks
    shared copy-on-write between beams): ``num_prompts`` prompts of U[ctx_lo,
    ctx_hi] tokens, each forked into ``beams`` beams, then one decode token per
    beam; every shared, partly filled last block is copied on write."""
    name: str
    num_prompts: int
    beams: int
    num_layers: int
    num_kv_heads: int
    head_dim: int
    block_size: int
    seed: int
    ctx_lo: int
    ctx_hi: int
    kv_dtype: str = BF16
    pool_slack: float = 1.5


# 32 layers of the 7B shape, 64 prompts x 4 beams: 192 block copies x 64 planes.
BEAM_FORK_7B = ForkWorkload("beam_fork_cow_7b_bf16", 64, 4, 32, 32, 128, 16, seed=8,
                            ctx_lo=64, ctx_hi=512)
FORK = (BEAM_FORK_7B,)


def fork_prompt_lens(w: ForkWorkload) -> np.ndarray:
    """Prompt lengths, none a multiple of the block size (the fork shares a
    partly filled block, as a beam fork mid-block does)."""
    lens = rng(w.seed, 1).integers(w.ctx_lo, w.ctx_hi + 1, size=w.num_prompts)
    lens = np.where(lens % w.block_size == 0, lens + 1, lens)
    return lens.astype(np.int64)


@dataclass(frozen=True)
class SwapWorkload:
    """Swapping whole sequences to host memory and back ("ToPG framework"
    section 2.3: pages beyond device memory): ``num_seqs`` sequences of
    U[ctx_lo, ctx_hi] tokens over ``num_layers`` layers; one step swaps every
    sequence out, then back in."""
    name: str
    num_seqs: int
    num_layers: int
    num_kv_heads: int
    head_dim: int
    block_size: int
    seed: int
    ctx_lo: int
    ctx_hi: int
    kv_dtype: str = BF16


# 8 layers of the 7B shape, 16 sequences of 256-1024 tokens (~1.2 GB each way).
SWAP_7B = SwapWorkload("swap_7b_8layer_bf16", 16, 8, 32, 128, 16, seed=10, ctx_lo=256,
                       ctx_hi=1024)
SWAP = (SWAP_7B,)


def swap_lens(w: SwapWorkload) -> np.ndarray:
    return rng(w.seed, 1).integers(w.ctx_lo, w.ctx_hi + 1, size=w.num_seqs).astype(np.int64)

