"""GPU parity of swapping blocks to host memory and back: swap_blocks against
the oracle's copy, and a decode after swap-outs, block reuse by other
sequences and swap-ins, against the oracle pool + oracle attention."""
import numpy as np
import pytest

import workloads as W
from oracle import attention as OA
from oracle import pool as OP
from tests.gpu_cases import from_torch, to_torch

pytestmark = pytest.mark.gpu


def test_swap_blocks_bit_exact_both_ways(lib):
    import torch
    import paged_kv_cache_295_gb300 as pkv
    r = np.random.default_rng(0)
    L, nb, bs, hkv, d, H = 2, 12, 16, 2, 128, 6
    pool = W.store(r.standard_normal((L, 2, nb, bs, hkv, d), dtype=np.float32), "bf16")
    host = W.store(r.standard_normal((H, L, 2, bs, hkv, d), dtype=np.float32), "bf16")
    dev = to_torch(pool, "bf16")
    h = to_torch(host, "bf16", device="cpu").pin_memory()
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    out_pairs = np.array([[3, 0], [7, 4], [0, 5]], dtype=np.int32)
    pkv.swap_blocks(dev, h, torch.from_numpy(out_pairs).cuda(), True, device_status=status)
    torch.cuda.synchronize()
    OA.swap_blocks(pool, host, out_pairs.tolist(), True)
    assert np.array_equal(h.view(torch.int16).numpy().view(np.uint16), host)
    in_pairs = np.array([[4, 1], [2, 9]], dtype=np.int32)
    pkv.swap_blocks(dev, h, torch.from_numpy(in_pairs).cuda(), False, device_status=status)
    torch.cuda.synchronize()
    OA.swap_blocks(pool, host, in_pairs.tolist(), False)
    assert np.array_equal(from_torch(dev, "bf16"), pool)
    assert int(status.item()) == 0


def test_decode_after_swap_round_trip_matches_oracle(lib):
    import torch
    import paged_kv_cache_295_gb300 as pkv
    from paged_kv_cache_295_gb300.engine import PagedKVCache
    L, hq, hkv, d, bs, nb, H = 2, 8, 2, 128, 16, 40, 32
    r = np.random.default_rng(5)
    order = r.permutation(nb).astype(np.int32)
    eng = PagedKVCache(L, hkv, d, bs, nb, pkv.BF16, device="cuda", initial_free_order=order)
    eng.host_area(H)
    op = OP.Pool(L, hkv, d, bs, 2, nb, initial_free_order=order.tolist())
    op.host_init(H)
    ocache = np.full((L, 2, nb, bs, hkv, d), 0x7FC0, dtype=np.uint16)
    ohost = np.zeros((H, L, 2, bs, hkv, d), dtype=np.uint16)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")

    def append(sid, n):
        sl = eng.pool.append_tokens(sid, n)
        assert sl.tolist() == op.seq_append_tokens(sid, n)
        for l in range(L):
            k = W.store(r.standard_normal((n, hkv, d), dtype=np.float32), "bf16")
            v = W.store(r.standard_normal((n, hkv, d), dtype=np.float32), "bf16")
            OA.reshape_and_cache(k, v, sl, ocache[l, 0], ocache[l, 1], "bf16", "bf16")
            eng.append(l, to_torch(k, "bf16"), to_torch(v, "bf16"),
                       torch.from_numpy(sl).cuda(), device_status=status)

    for s, n in enumerate([70, 33, 100]):
        eng.pool.seq_create(s)
        op.seq_create(s)
        append(s, n)
    eng.pool.seq_fork_prefix(3, 0, 64)               # shares 4 whole blocks of sequence 0
    op.seq_fork_prefix(3, 0, 64)
    append(3, 5)
    assert eng.pool.lru_order() == op.lru_order() == [0, 1, 2, 3]
    for s in (1, 0):                                   # the two least recent, 0 with shared blocks
        pairs = eng.swap_out(s, device_status=status)
        opairs = op.seq_swap_out(s)
        assert [tuple(x) for x in pairs.tolist()] == opairs
        OA.swap_blocks(ocache, ohost, opairs, True)
    for s, n in ((4, 90), (5, 40)):                    # new sequences reuse the freed blocks
        eng.pool.seq_create(s)
        op.seq_create(s)
        append(s, n)
    for s in (0, 1):
        pairs = eng.swap_in(s, device_status=status)
        opairs = op.seq_swap_in(s)
        assert [tuple(x) for x in pairs.tolist()] == opairs
        OA.swap_blocks(ocache, ohost, opairs, False)
    seqs = [0, 1, 2, 3, 4, 5]
    mb = max(len(op.tables[s]) for s in seqs)
    tables, lens = eng.pool.batch_tables(seqs, mb)
    t_o, l_o = op.padded_tables(seqs, mb)
    assert np.array_equal(tables, np.asarray(t_o)) and np.array_equal(lens, l_o)
    for l in range(L):
        q = W.store(r.standard_normal((len(seqs), hq, d), dtype=np.float32), "bf16")
        out = eng.attend(l, to_torch(q, "bf16"), torch.from_numpy(tables).cuda(),
                         torch.from_numpy(lens).cuda(), int(lens.max()), device_status=status)
        torch.cuda.synchronize()
        ref = OA.paged_attention_decode(q, ocache[l, 0], ocache[l, 1], np.asarray(t_o), l_o,
                                        eng.scale, "bf16", "bf16")
        assert np.abs(out.cpu().numpy() - ref).max() <= 2e-3
    assert int(status.item()) == 0
    assert np.array_equal(from_torch(eng.storage, "bf16"), ocache)
