"""Host-side accounting of bench.py, checked by brute force on small shapes."""
import numpy as np

import bench
import workloads as W


def test_prefill_flops_count_visible_keys():
    n = np.array([5, 1, 7, 0])
    ctx = np.array([5, 9, 30, 4])
    hq, d = 3, 8
    for causal in (True, False):
        keys = 0
        for ni, L in zip(n, ctx):
            for i in range(ni):
                keys += (L - ni + i + 1) if causal else L
        assert bench.prefill_alg_flops(n, ctx, hq, d, causal) == keys * hq * 4 * d


def test_prefill_workloads_respect_the_chunked_scheduler_limits():
    """Chunks of at most 512 tokens and at most 8192 tokens per batch ("LLM
    inference tutorial" section 6.2 defaults); prefix whole chunks."""
    for w in W.PREFILL:
        n, ctx = W.prefill_lens(w)
        assert (n <= ctx).all()
        if w.chunk_tokens:
            assert (n == w.chunk_tokens).all() and n.sum() <= 8192
            assert ((ctx - n) % w.chunk_tokens == 0).all()
