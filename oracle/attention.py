"""Oracle for the cache append and PagedAttention decode (plain definition).

TEST INFRASTRUCTURE ONLY (see ``oracle/__init__``).

Storage (per layer): ``k_cache`` and ``v_cache`` are ``[num_blocks, block_size,
num_kv_heads, head_dim]``, i.e. one layer's K (or V) slice of the pool tensor
``[num_layers, 2, num_blocks, block_size, num_kv_heads, head_dim]`` in
"LLM inference tutorial" section 4.2.  Element storage types:

* ``"f32"``      - numpy float32;
* ``"bf16"``     - numpy uint16 holding bfloat16 bit patterns;
* ``"fp8_e4m3"`` - numpy uint8 holding E4M3 codes, with one float32 scale
                   per KV head (K and V separately);
* ``"int8"``     - numpy int8 holding symmetric 8-bit codes, with one float32
                   scale per KV head (K and V separately).

What the decode step computes is a plain definition: paging only decides where
the bytes of a sequence live, and the page's ``get_kv`` (section 4.2) gathers
them back into contiguous ``[seq_len, num_kv_heads, head_dim]`` K and V.  The
attention is then section 4.4's forward for one query token: for query head
``h`` with ``G = num_q_heads // num_kv_heads`` query heads per KV head,
KV head ``g = h // G`` (``repeat_interleave(G, dim=1)``), logits ``z = scale *
q_h . K_g^T``, ``p = softmax(z)``, ``out = p . V_g``.  All of it in float64.
A sequence of length 0 attends to nothing and its output is 0.
"""
from __future__ import annotations

import numpy as np

from . import fp8


# -- element decoding ---------------------------------------------------------
def bf16_bits_to_f64(bits: np.ndarray) -> np.ndarray:
    """bfloat16 bit patterns -> float64 (exact: bf16 is the top half of f32)."""
    b = np.asarray(bits, dtype=np.uint16).astype(np.uint32) << np.uint32(16)
    return b.view(np.float32).astype(np.float64)


def to_f64(x: np.ndarray, dtype: str) -> np.ndarray:
    """Decode a stored q or cache array (not FP8) to float64, exactly."""
    if dtype == "f32":
        return np.asarray(x, dtype=np.float32).astype(np.float64)
    if dtype == "bf16":
        return bf16_bits_to_f64(x)
    raise ValueError(dtype)


def fp8_dequant(codes: np.ndarray, scale_per_head: np.ndarray) -> np.ndarray:
    """FP8 cache rows ``[..., num_kv_heads, head_dim]`` -> float64.

    The dequantised value is ``f32(code) * f32(scale[head])`` as ONE float32
    multiply (the "LLM inference tutorial" section 3.1 dequant ``q * scale``,
    taken in float32 as the stored scale is float32), then widened to float64.
    """
    vals = fp8.decode(codes).astype(np.float32)          # exact: E4M3 fits f32
    s = np.asarray(scale_per_head, dtype=np.float32)[:, None]
    return (vals * s).astype(np.float64)


def int8_encode(x_f32: np.ndarray, scale_per_head: np.ndarray) -> np.ndarray:
    """"LLM inference tutorial" section 3.1 ``symmetric_quantize`` with bits =
    8 and a given scale: ``round(x / scale)`` clamped to [-128, 127].  The
    quotient is one IEEE float32 division and ``round`` is round-half-to-even
    (torch.round).  A NaN quotient (the page leaves it open) encodes as 0.
    ``x_f32 [..., num_kv_heads, head_dim]`` float32."""
    s = np.asarray(scale_per_head, dtype=np.float32)[:, None]
    with np.errstate(divide="ignore", invalid="ignore"):
        q = np.asarray(x_f32, dtype=np.float32) / s
    q = np.where(np.isnan(q), np.float32(0), q)
    return np.clip(np.rint(q), -128, 127).astype(np.int8)


def int8_dequant(codes: np.ndarray, scale_per_head: np.ndarray) -> np.ndarray:
    """INT8 cache rows -> float64 as ``f32(code) * f32(scale[head])`` (one
    float32 multiply, section 3.1 dequantisation), then widened."""
    s = np.asarray(scale_per_head, dtype=np.float32)[:, None]
    return (np.asarray(codes, dtype=np.int8).astype(np.float32) * s).astype(np.float64)


# -- append: section 4.2 append_token, write half ------------------------------
def reshape_and_cache(k_new, v_new, slot_mapping, k_cache, v_cache, src_dtype: str,
                      cache_dtype: str, k_scale=None, v_scale=None):
    """Write token ``i``'s K/V rows at ``slot_mapping[i]`` (in place).

    ``k_new``/``v_new`` are ``[num_tokens, num_kv_heads, head_dim]`` in the
    source storage type.  Slot ``s`` is physical block ``s // block_size`` at
    offset ``s % block_size`` (section 4.2 ``append_token``); a negative slot
    skips the token.  Same source and cache type: the bytes are copied.  FP8
    cache: ``code = E4M3_rne_satfinite(f32(x) / f32(scale[head]))`` with the
    quotient an IEEE float32 division (section 3.1 ``x / scale``).  INT8
    cache: ``int8_encode``.
    """
    bs = k_cache.shape[1]
    for i, slot in enumerate(np.asarray(slot_mapping, dtype=np.int64).tolist()):
        if slot < 0:
            continue
        blk, off = divmod(slot, bs)
        for src, dst, scale in ((k_new, k_cache, k_scale), (v_new, v_cache, v_scale)):
            row = src[i]
            if cache_dtype == src_dtype:
                dst[blk, off] = row
            elif cache_dtype == "fp8_e4m3":
                x = to_f64(row, src_dtype).astype(np.float32)   # exact widening
                q = x / np.asarray(scale, dtype=np.float32)[:, None]
                dst[blk, off] = fp8.encode_f32(q.astype(np.float32))
            elif cache_dtype == "int8":
                dst[blk, off] = int8_encode(to_f64(row, src_dtype).astype(np.float32), scale)
            else:
                raise ValueError(f"unsupported append {src_dtype}->{cache_dtype}")


# -- copy-on-write: section 4.2 class docstring --------------------------------
def copy_blocks(pool, pairs):
    """``pool [num_layers, 2, num_blocks, ...]`` (in place): for each (src,
    dst) pair in order, every layer's K and V rows of block ``dst`` become
    those of block ``src``."""
    for src, dst in pairs:
        pool[:, :, int(dst)] = pool[:, :, int(src)]


# -- swap: "ToPG framework" section 2.3 (pages beyond device memory) -----------
def swap_blocks(pool, host, pairs, to_host: bool):
    """``pool [num_layers, 2, num_blocks, ...]``, ``host [num_host_blocks,
    num_layers, 2, ...]`` (in place): each (source, destination) pair copies a
    whole block, every layer's K and V, from the pool to a host slot
    (``to_host``) or from a host slot to the pool."""
    for src, dst in pairs:
        if to_host:
            host[int(dst)] = pool[:, :, int(src)]
        else:
            pool[:, :, int(dst)] = host[int(src)]


# -- gather: section 4.2 get_kv ------------------------------------------------
def gather_sequence(cache, table, seq_len: int):
    """Concatenate the first ``seq_len`` rows of the table's blocks, in order."""
    num_blocks, bs = cache.shape[0], cache.shape[1]
    nb = -(-seq_len // bs)
    parts = []
    for j in range(nb):
        p = int(table[j])
        if not (0 <= p < num_blocks):
            raise IndexError(f"block table entry {p} out of range")
        take = min(bs, seq_len - j * bs)
        parts.append(cache[p, :take])
    if not parts:
        return cache[:0, 0]
    return np.concatenate(parts, axis=0)


def decode_kv(rows, kv_dtype: str, scale=None) -> np.ndarray:
    if kv_dtype == "fp8_e4m3":
        return fp8_dequant(rows, scale)
    if kv_dtype == "int8":
        return int8_dequant(rows, scale)
    return to_f64(rows, kv_dtype)


# -- attention: section 4.4 forward for one query token -------------------------
def attend_one(q_heads: np.ndarray, K: np.ndarray, V: np.ndarray, scale: float) -> np.ndarray:
    """``q_heads [Hq, D]``, ``K/V [L, Hkv, D]`` float64 -> ``[Hq, D]`` float64."""
    hq, d = q_heads.shape
    L, hkv, _ = K.shape
    out = np.zeros((hq, d), dtype=np.float64)
    if L == 0:
        return out
    groups = hq // hkv
    for h in range(hq):
        g = h // groups
        z = scale * (K[:, g, :] @ q_heads[h])
        z = z - z.max()
        p = np.exp(z)
        p = p / p.sum()
        out[h] = p @ V[:, g, :]
    return out


def paged_attention_decode(q, k_cache, v_cache, block_tables, context_lens, scale,
                           q_dtype: str, kv_dtype: str, k_scale=None, v_scale=None,
                           seqs=None) -> np.ndarray:
    """Decode attention for every sequence (or the listed ``seqs``).

    ``q [S, Hq, D]``; ``block_tables [S, max_blocks]``; ``context_lens [S]``;
    ``scale`` is the float32 logit scale, widened to float64.  Returns float64
    ``[S, Hq, D]`` (rows not in ``seqs`` are 0).
    """
    S, hq, d = q.shape
    hkv = k_cache.shape[2]
    if hq % hkv:
        raise ValueError("num_q_heads must be a multiple of num_kv_heads")
    scale64 = float(np.float32(scale))
    out = np.zeros((S, hq, d), dtype=np.float64)
    for s in (range(S) if seqs is None else seqs):
        L = int(context_lens[s])
        K = decode_kv(gather_sequence(k_cache, block_tables[s], L), kv_dtype, k_scale)
        V = decode_kv(gather_sequence(v_cache, block_tables[s], L), kv_dtype, v_scale)
        out[s] = attend_one(to_f64(q[s], q_dtype), K, V, scale64)
    return out
