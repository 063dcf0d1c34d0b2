"""GPU tests of the CUDA-graph decode step (buckets + padding): replaying the
captured step equals the same calls made eagerly (bit for bit, same partition),
padded rows stay untouched and output 0, and the result matches the oracle."""
import numpy as np
import pytest

from oracle import attention as OA
from oracle import pool as OP
from tests.gpu_cases import from_torch, to_torch

pytestmark = pytest.mark.gpu


def _setup(L=3, hq=8, hkv=2, d=128, bs=16, nb=160, seqs=8, seed=0):
    import torch
    import paged_kv_cache_295_gb300 as pkv
    from paged_kv_cache_295_gb300.engine import PagedKVCache
    r = np.random.default_rng(seed)
    order = r.permutation(nb).astype(np.int32)
    eng = PagedKVCache(L, hkv, d, bs, nb, pkv.BF16, device="cuda", initial_free_order=order)
    op = OP.Pool(L, hkv, d, bs, 2, nb, initial_free_order=order.tolist())
    lens = r.integers(1, 200, size=seqs)
    host = np.full((L, 2, nb, bs, hkv, d), 0x7FC0, dtype=np.uint16)
    for s, n in enumerate(lens):
        eng.pool.seq_create(s)
        op.seq_create(s)
        sl = eng.pool.append_tokens(s, int(n))
        assert sl.tolist() == op.seq_append_tokens(s, int(n))
        for l in range(L):
            k = W_store(r, (int(n), hkv, d))
            v = W_store(r, (int(n), hkv, d))
            OA.reshape_and_cache(k, v, sl, host[l, 0], host[l, 1], "bf16", "bf16")
    eng.storage.copy_(to_torch(host, "bf16"))
    torch.cuda.synchronize()
    return eng, op, host, r


def W_store(r, shape):
    import workloads as W
    return W.store(r.standard_normal(shape, dtype=np.float32), "bf16")


@pytest.mark.parametrize("batch", [1, 3, 8])
def test_graph_replay_equals_eager_and_oracle(lib, batch):
    import torch
    import paged_kv_cache_295_gb300 as pkv
    eng, op, host, r = _setup()
    L, hq, hkv, d = eng.num_layers, 8, eng.num_kv_heads, eng.head_dim
    mb = 16
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    g = pkv.DecodeGraph(eng, hq, mb, [1, 2, 4, 8], device_status=status)
    before = eng.storage.clone()
    sids = list(range(batch))
    slots = eng.pool.append_slots(sids)
    assert slots.tolist() == op.seq_append_slots(sids)
    tables, lens = eng.pool.batch_tables(sids, mb)
    q = W_store(r, (L, batch, hq, d))
    kn = W_store(r, (L, batch, hkv, d))
    vn = W_store(r, (L, batch, hkv, d))
    g.q[:, :batch] = to_torch(q, "bf16")
    g.k_new[:, :batch] = to_torch(kn, "bf16")
    g.v_new[:, :batch] = to_torch(vn, "bf16")
    g.slots[:batch] = torch.from_numpy(slots).cuda()
    g.tables[:batch] = torch.from_numpy(tables).cuda()
    g.lens[:batch] = torch.from_numpy(lens).cuda()
    g.out.fill_(float("nan"))
    bucket = g.launch(batch)
    torch.cuda.synchronize()
    assert bucket == min(b for b in (1, 2, 4, 8) if b >= batch)
    assert int(status.item()) == 0
    got = g.out.cpu().numpy()
    assert (got[:, batch:bucket] == 0).all()          # padded rows: context 0
    after_graph = eng.storage.clone()

    # the same calls made eagerly on the cache as it was, with the graph's partition
    eng.storage.copy_(before)
    eager = []
    for l in range(L):
        eng.append(l, g.k_new[l, :batch], g.v_new[l, :batch], g.slots[:batch])
        eager.append(eng.attend(l, g.q[l, :batch], g.tables[:batch], g.lens[:batch], mb * 16,
                                workspace=g.ws).cpu().numpy())
    torch.cuda.synchronize()
    assert torch.equal(eng.storage.view(torch.int16), after_graph.view(torch.int16))
    for l in range(L):
        assert np.array_equal(got[l, :batch], eager[l])

    # the oracle: same appends, float64 attention
    for l in range(L):
        OA.reshape_and_cache(kn[l], vn[l], slots, host[l, 0], host[l, 1], "bf16", "bf16")
        ref = OA.paged_attention_decode(q[l], host[l, 0], host[l, 1], tables, lens, eng.scale,
                                        "bf16", "bf16")
        assert np.abs(got[l, :batch] - ref).max() <= 2e-3
    assert np.array_equal(from_torch(eng.storage, "bf16"), host)
    g.close()


def test_graph_batch_out_of_range_is_refused(lib):
    import paged_kv_cache_295_gb300 as pkv
    eng, _, _, _ = _setup(L=1, seqs=2)
    g = pkv.DecodeGraph(eng, 8, 16, [2, 4])
    for bad in (0, 5):
        with pytest.raises(pkv.PagedKVError):
            g.launch(bad)
    g.close()


def test_step_from_host_memory_equals_graph_launch(lib):
    """decode_graph_step_host (tables from the pool, host inputs in, output out)
    gives the same bytes as filling the buffers and launching."""
    import torch
    import paged_kv_cache_295_gb300 as pkv
    eng, op, host, r = _setup(seed=3)
    L, hq, hkv, d = eng.num_layers, 8, eng.num_kv_heads, eng.head_dim
    g = pkv.DecodeGraph(eng, hq, 16, [1, 2, 4, 8])
    sids = [0, 2, 5]
    slots = eng.pool.append_slots(sids)
    q = torch.from_numpy(W_store(r, (L, 3, hq, d)).view(np.int16)).view(torch.bfloat16)
    kn = torch.from_numpy(W_store(r, (L, 3, hkv, d)).view(np.int16)).view(torch.bfloat16)
    vn = torch.from_numpy(W_store(r, (L, 3, hkv, d)).view(np.int16)).view(torch.bfloat16)
    q_h, kn_h, vn_h = q.pin_memory(), kn.pin_memory(), vn.pin_memory()
    slots_h = torch.from_numpy(slots).pin_memory()
    out_h = torch.empty((L, 3, hq, d), dtype=torch.float32).pin_memory()
    before = eng.storage.clone()
    g.step_host(eng.pool, sids, q_h, kn_h, vn_h, slots_h, out_h)
    via_host = out_h.numpy().copy()
    after = eng.storage.clone()
    eng.storage.copy_(before)
    tables, lens = eng.pool.batch_tables(sids, 16)
    g.q[:, :3] = q.cuda()
    g.k_new[:, :3] = kn.cuda()
    g.v_new[:, :3] = vn.cuda()
    g.slots[:3] = torch.from_numpy(slots).cuda()
    g.tables[:3] = torch.from_numpy(tables).cuda()
    g.lens[:3] = torch.from_numpy(lens).cuda()
    g.launch(3)
    torch.cuda.synchronize()
    assert np.array_equal(g.out[:, :3].cpu().numpy(), via_host)
    assert torch.equal(eng.storage.view(torch.int16), after.view(torch.int16))
    with pytest.raises(pkv.PagedKVError):
        g.step_host(eng.pool, [0, 99], q_h[:, :2].contiguous(), kn_h[:, :2].contiguous(),
                    vn_h[:, :2].contiguous(), slots_h[:2].contiguous(), out_h[:, :2].contiguous())
    g.close()


def test_step_from_pageable_host_memory_equals_page_locked(lib):
    """Page-locked inputs are gathered by the staging kernel; pageable ones go
    through one copy per buffer.  Both give the same cache and output bytes."""
    import torch
    import paged_kv_cache_295_gb300 as pkv
    results = []
    for pinned in (True, False):
        eng, op, host, r = _setup(seed=4)
        L, hq, hkv, d = eng.num_layers, 8, eng.num_kv_heads, eng.head_dim
        g = pkv.DecodeGraph(eng, hq, 16, [1, 2, 4, 8])
        sids = [1, 4, 6, 7]
        slots = eng.pool.append_slots(sids)
        r2 = np.random.default_rng(11)
        mk = lambda shape: torch.from_numpy(W_store(r2, shape).view(np.int16)).view(torch.bfloat16)
        q, kn, vn = mk((L, 4, hq, d)), mk((L, 4, hkv, d)), mk((L, 4, hkv, d))
        sl = torch.from_numpy(slots)
        out = torch.empty((L, 4, hq, d), dtype=torch.float32)
        if pinned:
            q, kn, vn, sl, out = (x.pin_memory() for x in (q, kn, vn, sl, out))
        g.step_host(eng.pool, sids, q, kn, vn, sl, out)
        results.append((out.numpy().copy(), eng.storage.view(torch.int16).cpu().numpy()))
        g.close()
    assert results[0][0].tobytes() == results[1][0].tobytes()
    assert results[0][1].tobytes() == results[1][1].tobytes()
