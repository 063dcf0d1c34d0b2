"""Oracle for paged (chunked) prefill attention (plain definition).

TEST INFRASTRUCTURE ONLY (see ``oracle/__init__``).

Prefill is the first of the two inference phases in the "LLM inference
tutorial" (section 1.2): it processes all prompt tokens at once, computes
their attention and fills the KV cache.  The tutorial's chunked-prefill
scheduler (section 6.2, ``ChunkedPrefillScheduler``) splits a long prompt into
chunks of ``chunk_size`` tokens, so a chunk's queries attend to the cached
keys of the earlier chunks plus the chunk's own keys.

What one call computes, per sequence ``s``:

* the chunk's ``n_s = query_start[s+1] - query_start[s]`` query tokens are the
  LAST ``n_s`` positions of a context of ``ctx_s`` tokens whose K/V rows are
  already in the paged cache (appended before the attention, as the page's
  ``append_token`` precedes ``get_kv`` in section 4.2);
* query token ``i`` sits at position ``pos_i = ctx_s - n_s + i``; with the
  causal mask it attends to the keys at positions ``0 .. pos_i``, without it to
  all ``ctx_s`` keys;
* per query head ``h``: KV head ``g = h // G`` (section 4.4
  ``repeat_interleave``), ``z = scale * q . K^T``, ``p = softmax(z)``,
  ``out = p . V`` - section 4.4's forward, in float64.

The keys come from the sequence's blocks gathered in table order (section 4.2
``get_kv``), so paging changes only where the bytes live.
"""
from __future__ import annotations

import numpy as np

from .attention import decode_kv, gather_sequence, to_f64


def attend_rows(q_rows: np.ndarray, K: np.ndarray, V: np.ndarray, scale: float,
                limits) -> np.ndarray:
    """``q_rows [n, Hq, D]`` against ``K/V [L, Hkv, D]`` (float64).

    Row ``i`` sees the keys ``0 .. limits[i]`` (inclusive).  Returns float64
    ``[n, Hq, D]``.
    """
    n, hq, d = q_rows.shape
    hkv = K.shape[1]
    groups = hq // hkv
    out = np.zeros((n, hq, d), dtype=np.float64)
    for i in range(n):
        last = int(limits[i])
        if last < 0:
            continue
        for h in range(hq):
            g = h // groups
            z = scale * (K[: last + 1, g, :] @ q_rows[i, h])
            z = z - z.max()
            p = np.exp(z)
            p = p / p.sum()
            out[i, h] = p @ V[: last + 1, g, :]
    return out


def paged_attention_prefill(q, query_start, k_cache, v_cache, block_tables, context_lens,
                            scale, q_dtype: str, kv_dtype: str, causal: bool = True,
                            k_scale=None, v_scale=None, seqs=None) -> np.ndarray:
    """Prefill attention for every sequence (or the listed ``seqs``).

    ``q [T, Hq, D]`` holds the query tokens of all sequences back to back;
    sequence ``s`` owns rows ``query_start[s] .. query_start[s+1]-1``.
    ``block_tables [S, max_blocks]``, ``context_lens [S]`` (the chunk
    included).  ``scale`` is the float32 logit scale, widened to float64.
    Returns float64 ``[T, Hq, D]`` (rows of sequences not in ``seqs`` are 0).
    """
    T, hq, d = q.shape
    hkv = k_cache.shape[2]
    if hq % hkv:
        raise ValueError("num_q_heads must be a multiple of num_kv_heads")
    qs = np.asarray(query_start, dtype=np.int64)
    S = len(qs) - 1
    scale64 = float(np.float32(scale))
    out = np.zeros((T, hq, d), dtype=np.float64)
    for s in (range(S) if seqs is None else seqs):
        a, b = int(qs[s]), int(qs[s + 1])
        n, L = b - a, int(context_lens[s])
        if n == 0:
            continue
        if n > L:
            raise ValueError(f"sequence {s}: {n} query tokens but context {L}")
        K = decode_kv(gather_sequence(k_cache, block_tables[s], L), kv_dtype, k_scale)
        V = decode_kv(gather_sequence(v_cache, block_tables[s], L), kv_dtype, v_scale)
        limits = [(L - n + i) if causal else (L - 1) for i in range(n)]
        out[a:b] = attend_rows(to_f64(q[a:b], q_dtype), K, V, scale64, limits)
    return out

