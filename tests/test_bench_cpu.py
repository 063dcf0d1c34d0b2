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


def test_model_tokens_per_s_extrapolates_from_one_layer():
    import bench
    import workloads as W
    r = bench.model_tokens_per_s(W.LLAMA7B_LAYER, 200e-6)      # 200 us per layer step
    assert r["layers"] == 32 and abs(r["value"] - 32 / (200e-6 * 32)) < 1e-6
    assert bench.model_tokens_per_s(W.LLAMA70B_GQA, 200e-6)["layers"] == 80
    assert bench.model_tokens_per_s(W.RAGGED_FP8, 1e-3) is None   # already 32 layers
