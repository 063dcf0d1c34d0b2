"""Device KV pool + decode-step driver over the C ABI.

"nano-vLLM architecture" section 4.3: the KV pool is allocated once at start-up
and each layer gets a view of it, with the block as the unit of management.
The storage here is one tensor ``[num_layers, 2, num_blocks, block_size,
num_kv_heads, head_dim]`` (the pool tensor of "LLM inference tutorial" section
4.2); ``k_cache(l)`` / ``v_cache(l)`` are its contiguous per-layer views, and
the same block id / slot addresses every layer.

Only marshalling lives here: slots and tables come from the C++ pool, and the
cache writes and attention run in the CUDA kernels.
"""
from __future__ import annotations

import numpy as np

from . import (BF16, F32, FP8_E4M3, INT8, Pool, copy_blocks, paged_attention_decode, paged_attention_decode_append,
               paged_attention_prefill, reshape_and_cache, swap_blocks, workspace_bytes)


def _torch():
    import torch
    return torch


def torch_kv_dtype(code):
    torch = _torch()
    return {F32: torch.float32, BF16: torch.bfloat16, FP8_E4M3: torch.uint8,
            INT8: torch.int8}[code]


class PagedKVCache:
    """One allocation for all layers' K/V blocks plus the host block pool."""

    def __init__(self, num_layers, num_kv_heads, head_dim, block_size, num_blocks, kv_dtype,
                 device="cuda", initial_free_order=None, poison=True):
        torch = _torch()
        self.num_layers, self.num_kv_heads = num_layers, num_kv_heads
        self.head_dim, self.block_size, self.kv_dtype = head_dim, block_size, kv_dtype
        self.pool = Pool(num_layers, num_kv_heads, head_dim, block_size, kv_dtype,
                         num_blocks=num_blocks, initial_free_order=initial_free_order)
        self.num_blocks = num_blocks
        self.storage = torch.empty((num_layers, 2, num_blocks, block_size, num_kv_heads,
                                    head_dim), dtype=torch_kv_dtype(kv_dtype), device=device)
        if poison:   # unused slots hold NaN so a stray read shows in the output
            if kv_dtype == FP8_E4M3:
                self.storage.fill_(0x7F)
            elif kv_dtype == INT8:       # no NaN code: the largest one distorts a stray read
                self.storage.fill_(127)
            else:
                self.storage.fill_(float("nan"))
        # logit scale 1/sqrt(head_dim) as float32 ("LLM inference tutorial" 4.4)
        self.scale = float(np.float32(1.0 / np.sqrt(head_dim)))
        self.k_scale = None
        self.v_scale = None
        if kv_dtype in (FP8_E4M3, INT8):
            self.k_scale = torch.ones((num_layers, num_kv_heads), dtype=torch.float32,
                                      device=device)
            self.v_scale = torch.ones_like(self.k_scale)

    def k_cache(self, layer):
        return self.storage[layer, 0]

    def v_cache(self, layer):
        return self.storage[layer, 1]

    def append(self, layer, k_new, v_new, slot_mapping, device_status=None, stream=None):
        ks = None if self.k_scale is None else self.k_scale[layer]
        vs = None if self.v_scale is None else self.v_scale[layer]
        reshape_and_cache(k_new, v_new, slot_mapping, self.k_cache(layer), self.v_cache(layer),
                          ks, vs, device_status=device_status, stream=stream)

    def run_copies(self, device_status=None, stream=None):
        """Drain the pool's copy-on-write queue and copy those blocks (every
        layer, K and V) on the device; returns the pairs (host ``[k, 2]``)."""
        torch = _torch()
        pairs = self.pool.take_copies()
        if pairs.shape[0]:
            # pairs of one source side by side: its re-reads then hit L2
            grouped = pairs[np.argsort(pairs[:, 0], kind="stable")]
            d = torch.from_numpy(np.ascontiguousarray(grouped)).to(self.storage.device)
            copy_blocks(self.storage, d, device_status=device_status, stream=stream)
        return pairs

    def host_area(self, num_host_blocks):
        """Page-locked host swap area ``[H, L, 2, bs, Hkv, D]`` and the pool's
        host slot list (once)."""
        torch = _torch()
        self.pool.host_init(num_host_blocks)
        self.host = torch.empty((num_host_blocks,) + tuple(self.storage.shape[:2]) +
                                tuple(self.storage.shape[3:]), dtype=self.storage.dtype,
                                pin_memory=True)
        return self.host

    def swap_out(self, sid, device_status=None, stream=None):
        """Move the sequence's private blocks to host slots (device -> host copies)."""
        torch = _torch()
        pairs = self.pool.swap_out(sid)
        if pairs.shape[0]:
            swap_blocks(self.storage, self.host, torch.from_numpy(pairs).to(self.storage.device),
                        True, device_status=device_status, stream=stream)
        return pairs

    def swap_in(self, sid, device_status=None, stream=None):
        """Bring a swapped-out sequence back (host -> device copies)."""
        torch = _torch()
        pairs = self.pool.swap_in(sid)
        if pairs.shape[0]:
            swap_blocks(self.storage, self.host, torch.from_numpy(pairs).to(self.storage.device),
                        False, device_status=device_status, stream=stream)
        return pairs

    def attend(self, layer, q, block_tables, context_lens, max_context_len, out=None,
               workspace=None, partition=0, device_status=None, stream=None):
        ks = None if self.k_scale is None else self.k_scale[layer]
        vs = None if self.v_scale is None else self.v_scale[layer]
        return paged_attention_decode(q, self.k_cache(layer), self.v_cache(layer), block_tables,
                                      context_lens, self.scale, max_context_len, out=out,
                                      k_scale=ks, v_scale=vs, workspace=workspace,
                                      partition=partition, device_status=device_status,
                                      stream=stream)

    def append_attend(self, layer, q, k_new, v_new, slot_mapping, block_tables, context_lens,
                      max_context_len, out=None, workspace=None, partition=0, device_status=None,
                      stream=None):
        """One decode step of one layer: append each sequence's new token and
        attend, fused into the decode kernel where it runs the transposed
        tensor-core path."""
        ks = None if self.k_scale is None else self.k_scale[layer]
        vs = None if self.v_scale is None else self.v_scale[layer]
        return paged_attention_decode_append(q, k_new, v_new, slot_mapping, self.k_cache(layer),
                                             self.v_cache(layer), block_tables, context_lens,
                                             self.scale, max_context_len, out=out, k_scale=ks,
                                             v_scale=vs, workspace=workspace, partition=partition,
                                             device_status=device_status, stream=stream)

    def prefill(self, layer, q, query_start, block_tables, context_lens, max_query_len,
                max_context_len, causal=True, out=None, device_status=None, stream=None):
        ks = None if self.k_scale is None else self.k_scale[layer]
        vs = None if self.v_scale is None else self.v_scale[layer]
        return paged_attention_prefill(q, query_start, self.k_cache(layer), self.v_cache(layer),
                                       block_tables, context_lens, self.scale, max_query_len,
                                       max_context_len, causal=causal, out=out, k_scale=ks,
                                       v_scale=vs, device_status=device_status, stream=stream)

    def workspace_for(self, num_seqs, num_q_heads, max_context_len, partition=0, device="cuda"):
        torch = _torch()
        n = workspace_bytes(num_seqs, num_q_heads, self.num_kv_heads, self.head_dim,
                            max_context_len, partition)
        return torch.empty(max(n, 16), dtype=torch.uint8, device=device)


def build_prompts(pool, lens_after_step, prefix_tokens=0, prefix_seqs=0, owner_id=None):
    """Create every sequence and append its prompt (all but the step's token).

    Sequences ``0 .. prefix_seqs-1`` share the first ``prefix_tokens`` tokens of
    an owner sequence (id ``owner_id``, default ``len(lens)``) that is filled
    first.  Returns (owner id or None, list of per-sequence prompt slot arrays,
    owner prompt slots or None), in the order the rows were appended.
    """
    S = len(lens_after_step)
    owner = None
    owner_slots = None
    if prefix_tokens:
        owner = S if owner_id is None else owner_id
        pool.seq_create(owner)
        owner_slots = pool.append_tokens(owner, prefix_tokens)
    slots = []
    for s in range(S):
        L = int(lens_after_step[s]) - 1
        if prefix_tokens and s < prefix_seqs:
            pool.seq_fork_prefix(s, owner, prefix_tokens)
            slots.append(pool.append_tokens(s, L - prefix_tokens))
        else:
            pool.seq_create(s)
            slots.append(pool.append_tokens(s, L))
    return owner, slots, owner_slots
