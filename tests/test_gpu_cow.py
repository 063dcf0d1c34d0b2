"""GPU parity of copy-on-write: copy_blocks against the oracle's copy, and a
beam-search decode (forked sequences, copy-on-write appends, decode) run on
the C pool + CUDA kernels and on the oracle pool + oracle, step by step."""
import numpy as np
import pytest

import workloads as W
from oracle import attention as OA
from oracle import pool as OP
from tests.gpu_cases import from_torch, to_torch

pytestmark = pytest.mark.gpu


def _pairs(r, nb, k):
    ids = r.permutation(nb)
    return np.stack([ids[:k], ids[k:2 * k]], axis=1).astype(np.int32)   # dst never a src


@pytest.mark.parametrize("L,bs,hkv,d,k", [(2, 16, 4, 64, 5), (3, 8, 2, 128, 17),
                                          (1, 128, 8, 128, 3)])
def test_copy_blocks_bit_exact(lib, L, bs, hkv, d, k):
    import torch
    import paged_kv_cache_295_gb300 as pkv
    r = np.random.default_rng(L * 100 + k)
    nb = 3 * k + 4
    host = W.store(r.standard_normal((L, 2, nb, bs, hkv, d), dtype=np.float32), "bf16")
    dev = to_torch(host, "bf16")
    pairs = _pairs(r, nb, k)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    pkv.copy_blocks(dev, torch.from_numpy(pairs).cuda(), device_status=status)
    torch.cuda.synchronize()
    OA.copy_blocks(host, pairs.tolist())
    assert int(status.item()) == 0
    assert np.array_equal(from_torch(dev, "bf16"), host)


def test_copy_blocks_bad_ids_are_flagged_and_skipped(lib):
    import torch
    import paged_kv_cache_295_gb300 as pkv
    r = np.random.default_rng(3)
    host = W.store(r.standard_normal((1, 2, 8, 16, 2, 64), dtype=np.float32), "bf16")
    dev = to_torch(host, "bf16")
    pairs = np.array([[1, 2], [9, 3], [4, -1]], dtype=np.int32)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    pkv.copy_blocks(dev, torch.from_numpy(pairs).cuda(), device_status=status)
    torch.cuda.synchronize()
    assert int(status.item()) & 0x1
    OA.copy_blocks(host, [(1, 2)])
    assert np.array_equal(from_torch(dev, "bf16"), host)


@pytest.mark.parametrize("bs,hq,hkv", [(16, 8, 2), (8, 4, 4)])
def test_beam_search_decode_matches_oracle(lib, bs, hq, hkv):
    """Prompts, then beams forked from them (full forks, so the partly filled
    last block is shared), then several decode steps with copy-on-write."""
    import torch
    import paged_kv_cache_295_gb300 as pkv
    from paged_kv_cache_295_gb300.engine import PagedKVCache
    L, d, nb = 2, 128, 96
    r = np.random.default_rng(bs + hq)
    order = r.permutation(nb).astype(np.int32)
    eng = PagedKVCache(L, hkv, d, bs, nb, pkv.BF16, device="cuda", initial_free_order=order)
    op = OP.Pool(L, hkv, d, bs, 2, nb, initial_free_order=order.tolist())
    ocache = np.full((L, 2, nb, bs, hkv, d), 0x7FC0, dtype=np.uint16)    # NaN, like the engine
    status = torch.zeros(1, dtype=torch.int32, device="cuda")

    def write(slots, k_rows, v_rows, layer):
        OA.reshape_and_cache(k_rows, v_rows, slots, ocache[layer, 0], ocache[layer, 1],
                             "bf16", "bf16")
        eng.append(layer, to_torch(k_rows, "bf16"), to_torch(v_rows, "bf16"),
                   torch.from_numpy(np.asarray(slots, dtype=np.int64)).cuda(),
                   device_status=status)

    prompts = [37, 21, 50]
    for s, n in enumerate(prompts):
        eng.pool.seq_create(s)
        op.seq_create(s)
        sl = eng.pool.append_tokens(s, n)
        assert sl.tolist() == op.seq_append_tokens(s, n)
        for layer in range(L):
            write(sl, W.store(r.standard_normal((n, hkv, d), dtype=np.float32), "bf16"),
                  W.store(r.standard_normal((n, hkv, d), dtype=np.float32), "bf16"), layer)
    beams = list(range(len(prompts)))
    nid = len(prompts)
    for s in range(len(prompts)):               # two more beams per prompt
        for _ in range(2):
            eng.pool.seq_fork_prefix(nid, s, prompts[s])
            op.seq_fork_prefix(nid, s, prompts[s])
            beams.append(nid)
            nid += 1
    checked = 0
    for step in range(bs + 2):                  # crosses a block boundary
        slots = eng.pool.append_slots(beams)
        assert slots.tolist() == op.seq_append_slots(beams)
        pairs = eng.run_copies(device_status=status)
        opairs = op.take_copies()
        assert [tuple(x) for x in pairs.tolist()] == opairs
        OA.copy_blocks(ocache, opairs)
        if step == 0:
            assert len(opairs) == 2 * len(prompts)   # every prompt's partial block, twice
        mb = max(len(op.tables[b]) for b in beams)
        tables, lens = eng.pool.batch_tables(beams, mb)
        t_o, l_o = op.padded_tables(beams, mb)
        assert np.array_equal(tables, np.asarray(t_o)) and np.array_equal(lens, l_o)
        tables_d = torch.from_numpy(tables).cuda()
        lens_d = torch.from_numpy(lens).cuda()
        for layer in range(L):
            k_rows = W.store(r.standard_normal((len(beams), hkv, d), dtype=np.float32), "bf16")
            v_rows = W.store(r.standard_normal((len(beams), hkv, d), dtype=np.float32), "bf16")
            write(slots, k_rows, v_rows, layer)
            q = W.store(r.standard_normal((len(beams), hq, d), dtype=np.float32), "bf16")
            out = eng.attend(layer, to_torch(q, "bf16"), tables_d, lens_d, int(lens.max()),
                             device_status=status)
            torch.cuda.synchronize()
            ref = OA.paged_attention_decode(q, ocache[layer, 0], ocache[layer, 1],
                                            np.asarray(t_o), l_o, eng.scale, "bf16", "bf16")
            assert np.abs(out.cpu().numpy() - ref).max() <= 2e-3
            checked += 1
    assert int(status.item()) == 0
    assert np.array_equal(from_torch(eng.storage, "bf16"), ocache)      # every byte
    assert checked == (bs + 2) * L
