"""GPU parity of paged (chunked) prefill attention against the oracle.

Each case builds the same seeded step on both sides: the oracle pool and the C
pool hand out the same slots; the cached prefix rows are placed by the oracle's
append and uploaded; the chunk's rows are appended on the GPU by
reshape_and_cache (compared byte for byte with the oracle's append); then the
tcgen05 prefill kernel runs and its float32 output is compared with the
oracle's float64 result element by element.  Unused slots and padding table
entries hold NaN, so a kernel that touches them fails.
"""
import numpy as np
import pytest

import workloads as W
from oracle import attention as OA
from oracle import prefill as OPF
from tests.gpu_cases import from_torch
from tests.gpu_cases import make_prefill as build
from tests.gpu_cases import run_prefill_gpu as run_gpu

pytestmark = pytest.mark.gpu

TOL = 2e-3          # bf16 cache, float32 output (the decode bound)


def _w(hq, hkv, bs):
    return W.PrefillWorkload(f"t{hq}_{hkv}_{bs}", 0, 0, 0, hq, hkv, 128, bs, seed=31)


CASES = [  # (Hq, Hkv, bs, chunk lens, cached prefix lens)
    (4, 4, 16, [5, 130, 64], [0, 37, 300]),            # MHA: 2 query tiles, ragged tails
    (8, 2, 8, [33, 1, 70], [100, 0, 15]),              # G=4, blocks of 8, a decode-like row
    (16, 2, 128, [20, 17], [250, 0]),                  # G=8, 16 tokens per tile
    (16, 1, 32, [9, 40], [64, 3]),                     # G=16 (MQA-like), 8 tokens per tile
    (6, 2, 16, [50, 43], [7, 200]),                    # G=3: 42 tokens x 3 heads = 126 rows
    (4, 4, 64, [128, 0, 1], [128, 5, 0]),              # an empty chunk; exact tile sizes
    (8, 2, 4096, [70, 300], [4090, 4000]),             # the largest block: chunks across it
]


@pytest.mark.parametrize("causal", [True, False])
@pytest.mark.parametrize("hq,hkv,bs,chunk,prefix", CASES)
def test_prefill_matches_oracle(lib, hq, hkv, bs, chunk, prefix, causal):
    import torch
    w = _w(hq, hkv, bs)
    dev, host, max_q, max_ctx = build(w, chunk, prefix)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    got = run_gpu(w, dev, max_q, max_ctx, causal=causal, status=status)
    assert int(status.item()) == 0
    assert np.array_equal(from_torch(dev["kc"], "bf16"), host["kc"])   # chunk append, bytes
    assert np.array_equal(from_torch(dev["vc"], "bf16"), host["vc"])
    ref = OPF.paged_attention_prefill(host["q"], host["qs"], host["kc"], host["vc"],
                                      host["tables"], host["ctx"], w.scale, "bf16", "bf16",
                                      causal=causal)
    assert np.isfinite(got).all()
    err = np.abs(got - ref).max() if got.size else 0.0
    assert err <= TOL, err


FP8_CASES = [  # (Hq, Hkv, bs, chunk lens, cached prefix lens)
    (4, 4, 16, [5, 130, 64], [0, 37, 300]),            # MHA, 16-row boxes, ragged tails
    (16, 2, 128, [20, 17], [250, 0]),                  # G=8, one box per tile
    (8, 2, 8, [33, 1, 70], [100, 0, 15]),              # blocks of 8: 8 boxes per tile
    (8, 1, 64, [200, 64], [0, 600]),                   # G=8 (MQA-like), many tiles
]


@pytest.mark.parametrize("kv", ["fp8_e4m3", "int8"])
@pytest.mark.parametrize("causal", [True, False])
@pytest.mark.parametrize("hq,hkv,bs,chunk,prefix", FP8_CASES)
def test_8bit_prefill_matches_oracle(lib, hq, hkv, bs, chunk, prefix, causal, kv):
    """FP8-E4M3 and INT8 caches: the chunk's codes bit-exact with the oracle's
    append, the output within the 8-bit bound (the oracle dequantises the same
    codes)."""
    import torch
    w = _w(hq, hkv, bs)
    dev, host, max_q, max_ctx = build(w, chunk, prefix, kv=kv)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    got = run_gpu(w, dev, max_q, max_ctx, causal=causal, status=status)
    assert int(status.item()) == 0
    assert np.array_equal(from_torch(dev["kc"], kv), host["kc"])
    assert np.array_equal(from_torch(dev["vc"], kv), host["vc"])
    ref = OPF.paged_attention_prefill(host["q"], host["qs"], host["kc"], host["vc"],
                                      host["tables"], host["ctx"], w.scale, "bf16", kv,
                                      causal=causal, k_scale=host["ks"], v_scale=host["vs"])
    assert np.isfinite(got).all()
    err = np.abs(got - ref).max() if got.size else 0.0
    assert err <= 1e-2, err


@pytest.mark.parametrize("kv", ["bf16", "fp8_e4m3", "int8"])
def test_prefill_q_far_outside_fp16_range(lib, kv):
    """q rows of magnitude 3e5 (past fp16's 65504), 1e-5 (fp16 subnormal) and 1:
    the FP8 path carries q in fp16 scaled per row by a power of two, so every
    row stays finite and exact; both paths match the oracle."""
    import torch
    w = _w(8, 2, 16)
    dev, host, max_q, max_ctx = build(w, [40, 17], [100, 3], kv=kv, q_mul=[3e5, 1e-5, 1.0])
    assert np.abs(OA.to_f64(host["q"], "bf16")).max() > 65504.0
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    got = run_gpu(w, dev, max_q, max_ctx, causal=True, status=status)
    assert int(status.item()) == 0
    ref = OPF.paged_attention_prefill(host["q"], host["qs"], host["kc"], host["vc"],
                                      host["tables"], host["ctx"], w.scale, "bf16", kv,
                                      causal=True, k_scale=host["ks"], v_scale=host["vs"])
    assert np.isfinite(got).all()
    assert np.abs(got - ref).max() <= (TOL if kv == "bf16" else 1e-2)


def attention_sink(k0):
    """Key 0 of every sequence far above the rest: q is 3 on dimension 0 and
    that key k0 there (0 elsewhere), the other keys are scaled by 1/4, so its
    logit sits about 0.265 k0 nats above theirs, which spread a few tenths of a
    nat around 0: k0 = 67 puts their P near 2^-25.6 (below every fp16 value),
    k0 = 49 near 2^-18.7 (fp16 subnormals)."""
    def shape(k, v, q, starts):
        q[:, :, 0] = 3.0
        k *= 0.25
        for s0 in starts:
            k[s0] = 0.0
            k[s0, :, 0] = k0
    return shape


@pytest.mark.parametrize("k0", [67, 49])
@pytest.mark.parametrize("kv", ["int8", "fp8_e4m3", "bf16"])
def test_prefill_long_context_with_an_attention_sink(lib, kv, k0):
    """32K cached tokens and one key far above the rest: every other key's P
    is far below the largest, where fp16 keeps few bits or none, so the P the
    MMA sees sums short of the float32 row sum.  The INT8 path widens V
    exactly: a +1152 offset kept in V and taken off in the epilogue would be
    off by about 0.03 at k0 = 67.  The 8-bit bound (1e-2) and the bf16 one
    (2e-3) hold."""
    import torch
    w = _w(8, 2, 16)
    dev, host, max_q, max_ctx = build(w, [64, 40], [32768, 32000], kv=kv,
                                      shape_rows=attention_sink(k0))
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    got = run_gpu(w, dev, max_q, max_ctx, causal=True, status=status)
    assert int(status.item()) == 0
    ref = OPF.paged_attention_prefill(host["q"], host["qs"], host["kc"], host["vc"],
                                      host["tables"], host["ctx"], w.scale, "bf16", kv,
                                      causal=True, k_scale=host["ks"], v_scale=host["vs"])
    assert np.isfinite(got).all()
    err = np.abs(got - ref).max()
    print(f"prefill sink {kv} k0={k0}: max abs err {err:.3e}")
    assert err <= (TOL if kv == "bf16" else 1e-2)


@pytest.mark.parametrize("kv", ["bf16", "fp8_e4m3"])
@pytest.mark.parametrize("chunk,prefix", [
    ([10, 30, 10, 30, 20], [50, 30, 50, 30, 40]),   # equal contexts: ties in the work order
    ([3, 1, 2] * 44, [(7 * i) % 61 for i in range(132)]),   # 132 sequences: not ranked
])
def test_work_order_covers_every_sequence(lib, kv, chunk, prefix):
    """The kernel maps its blocks to (sequence, pair, KV head) longest context
    first, ranking up to 128 sequences itself: with tied contexts and with
    more sequences than it ranks, every row of every chunk still matches the
    oracle (a sequence left out or done twice would not)."""
    import torch
    w = _w(8, 2, 16)
    dev, host, max_q, max_ctx = build(w, chunk, prefix, kv=kv)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    got = run_gpu(w, dev, max_q, max_ctx, causal=True, status=status)
    assert int(status.item()) == 0
    ref = OPF.paged_attention_prefill(host["q"], host["qs"], host["kc"], host["vc"],
                                      host["tables"], host["ctx"], w.scale, "bf16", kv,
                                      causal=True, k_scale=host["ks"], v_scale=host["vs"])
    assert np.isfinite(got).all()
    assert np.abs(got - ref).max() <= (TOL if kv == "bf16" else 1e-2)


def test_single_token_chunks_match_decode_kernel(lib):
    """A chunk of one token is a decode step: both kernels, both within tolerance
    of the oracle, on the same cache."""
    import torch
    import paged_kv_cache_295_gb300 as pkv
    w = _w(8, 2, 16)
    dev, host, max_q, max_ctx = build(w, [1, 1, 1, 1], [0, 63, 200, 17])
    pre = run_gpu(w, dev, max_q, max_ctx)
    dec = pkv.paged_attention_decode(dev["q"], dev["kc"], dev["vc"], dev["tables"], dev["ctx"],
                                     w.scale, max_ctx)
    torch.cuda.synchronize()
    ref = OA.paged_attention_decode(host["q"], host["kc"], host["vc"], host["tables"],
                                    host["ctx"], w.scale, "bf16", "bf16")
    assert np.abs(pre - ref).max() <= TOL
    assert np.abs(dec.cpu().numpy() - ref).max() <= TOL


def test_bad_block_is_flagged_and_skipped(lib):
    """An out-of-range table entry is flagged; its keys are left out, which is
    the oracle's result on a cache whose block holds no key (checked on the
    rows that cannot see the block)."""
    import torch
    w = _w(4, 4, 16)
    dev, host, max_q, max_ctx = build(w, [40], [60], bad_block=(0, 5))   # keys 80..95
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    got = run_gpu(w, dev, max_q, max_ctx, status=status)
    assert int(status.item()) & 0x1
    tables = host["tables"].copy()
    tables[0, 5] = 0                     # any real block; rows below 80 never see it
    ref = OPF.paged_attention_prefill(host["q"], host["qs"], host["kc"], host["vc"], tables,
                                      host["ctx"], w.scale, "bf16", "bf16")
    # query i sits at position 60 + i: rows 0..19 see keys 0..79 only
    assert np.abs(got[:20] - ref[:20]).max() <= TOL
    assert np.isfinite(got).all()


def test_bad_query_start_is_flagged(lib):
    import torch
    import paged_kv_cache_295_gb300 as pkv
    w = _w(4, 4, 16)
    dev, host, max_q, max_ctx = build(w, [10, 10], [0, 0])
    dev["qs"] = torch.tensor([0, 10, 25], dtype=torch.int32, device="cuda")   # 25 > T = 20
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    out = torch.zeros((20, 4, 128), dtype=torch.float32, device="cuda")
    pkv.paged_attention_prefill(dev["q"], dev["qs"], dev["kc"], dev["vc"], dev["tables"],
                                dev["ctx"], w.scale, 15, max_ctx, out=out, device_status=status)
    torch.cuda.synchronize()
    assert int(status.item()) & 0x4


def test_argument_errors(lib):
    import torch
    import paged_kv_cache_295_gb300 as pkv
    w = _w(4, 4, 16)
    dev, host, max_q, max_ctx = build(w, [8], [8])
    with pytest.raises(pkv.PagedKVError):  # head_dim 64 is not built for prefill
        pkv.paged_attention_prefill(dev["q"][..., :64].contiguous(), dev["qs"],
                                    dev["kc"][..., :64].contiguous(),
                                    dev["vc"][..., :64].contiguous(), dev["tables"], dev["ctx"],
                                    0.1, max_q, max_ctx)
    with pytest.raises(pkv.PagedKVError):  # max_query_len above the token count
        pkv.paged_attention_prefill(dev["q"], dev["qs"], dev["kc"], dev["vc"], dev["tables"],
                                    dev["ctx"], 0.1, 9, max_ctx)


@pytest.mark.parametrize("name", [w.name for w in W.PREFILL if w.chunk_tokens])
def test_fullsize_sampled_rows(lib, name):
    """The bench's full-size step, in the launch configuration bench.py times,
    against the oracle on sampled query rows: the first, the last and a middle
    row of the sequences with the shortest and the longest context."""
    import torch
    import bench
    w = bench.WORKLOADS[name]
    st = bench.PrefillStep(w, torch.device("cuda", 0), keep_src=True)
    st.run()
    torch.cuda.synchronize()
    assert int(st.status.item()) == 0
    k_src, v_src, off = st.src
    got = st.out
    codes8 = w.kv_dtype in ("fp8_e4m3", "int8")
    for s in sorted({int(np.argmin(st.lens)), int(np.argmax(st.lens))}):
        L, n = int(st.lens[s]), int(st.n[s])
        rows = sorted({0, n // 2, n - 1})
        if codes8:   # the cache's codes through the block table, dequantised by the oracle
            blocks = torch.from_numpy(st.tables_h[s, :-(-L // w.block_size)]).cuda()
            ks, vs = (x[0].cpu().numpy() for x in (st.eng.k_scale, st.eng.v_scale))
            kc = from_torch(st.eng.k_cache(0)[blocks], w.kv_dtype).reshape(-1, *k_src.shape[1:])
            vc = from_torch(st.eng.v_cache(0)[blocks], w.kv_dtype).reshape(-1, *v_src.shape[1:])
            K = OA.decode_kv(kc[:L], w.kv_dtype, ks)
            V = OA.decode_kv(vc[:L], w.kv_dtype, vs)
        else:
            K = OA.to_f64(from_torch(k_src[off[s]:off[s] + L], "bf16"), "bf16")
            V = OA.to_f64(from_torch(v_src[off[s]:off[s] + L], "bf16"), "bf16")
        a = int(st.qs_h[s])
        q = OA.to_f64(from_torch(st.q[a:a + n], "bf16"), "bf16")
        ref = OPF.attend_rows(q[rows], K, V, w.scale, [L - n + i for i in rows])
        g = got[[a + i for i in rows]].cpu().numpy()
        assert np.abs(g - ref).max() <= (1e-2 if codes8 else TOL)
