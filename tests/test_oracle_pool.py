"""Pins for the pool oracle: the pages' worked example, hand-derived traces, invariants."""
import json
import os

import numpy as np
import pytest

from oracle import pool as P

GOLD = os.path.join(os.path.dirname(__file__), "golden")


def test_worked_example_memory_usage():
    g = json.load(open(os.path.join(GOLD, "pool_worked_example.json")))
    pool = P.Pool(g["num_layers"], g["num_kv_heads"], g["head_dim"], g["block_size"],
                  g["dtype_size"], g["num_blocks"])
    for sid in range(g["num_seqs"]):
        pool.seq_create(sid)
        for _ in range(g["tokens_per_seq"]):
            pool.seq_append_slots([sid])
    st = pool.stats()
    e = g["expected"]
    assert st["total_blocks"] == e["total_blocks"]
    assert st["used_blocks"] == e["used_blocks"]
    assert st["free_blocks"] == e["free_blocks"]
    assert st["utilization"] == pytest.approx(e["utilization"], rel=0, abs=1e-12)
    assert st["block_bytes"] == e["block_bytes_per_layer"] * g["num_layers"]
    assert st["total_memory_gb"] == pytest.approx(e["total_memory_gb"], rel=1e-15)
    assert st["used_memory_gb"] == pytest.approx(e["used_memory_gb"], rel=1e-15)
    for sid in range(g["num_seqs"]):
        assert len(pool.block_table(sid)) == e["blocks_per_seq"]
    # FIFO hand-out of an unshuffled pool: sequence i owns blocks 7i .. 7i+6
    assert pool.block_table(3) == list(range(21, 28))


def test_kv_size_printouts():
    g = json.load(open(os.path.join(GOLD, "kv_cache_sizes.json")))
    mha = None
    for c in g["cases"]:
        b = P.block_bytes(1, g["seq_len"], c["kv_heads"], g["head_dim"], g["dtype_size"])
        assert f"{b / 1e6:.1f}" == c["mb_1dp"]
        if mha is None:
            mha = b
        else:
            assert f"{(1 - b / mha) * 100:.0f}" == c["saving_pct"]


def test_available_blocks_floor():
    bb = P.block_bytes(32, 16, 32, 128, 2)
    assert bb == 8 * 1024 * 1024                 # 8 MiB per all-layer block (7B, fp16)
    assert P.available_blocks(80 * 2**30, bb) == 10240
    assert P.available_blocks(bb - 1, bb) == 0


def test_hand_trace_fifo_slots_and_free_order():
    # block_size 4, free list starts [5, 2, 0, 4, 1, 3]
    pool = P.Pool(1, 1, 8, 4, 2, 6, initial_free_order=[5, 2, 0, 4, 1, 3])
    pool.seq_create(10)                          # takes 5
    pool.seq_create(11)                          # takes 2
    assert pool.seq_append_tokens(10, 5) == [20, 21, 22, 23, 0]   # 5*4+0..3, then block 0
    assert pool.seq_append_slots([11, 10]) == [8, 1]
    assert pool.block_table(10) == [5, 0] and pool.lens[10] == 6
    pool.seq_free(10)                            # tail gets 5 then 0
    assert list(pool.free) == [4, 1, 3, 5, 0]
    pool.seq_create(12)                          # takes 4
    assert pool.seq_append_tokens(12, 4) == [16, 17, 18, 19]
    assert pool.seq_append_slots([12]) == [4]    # block 1, offset 0
    assert pool.stats()["used_blocks"] == 3      # blocks 2, 4, 1


def test_prefix_sharing_refcounts():
    pool = P.Pool(1, 1, 8, 4, 2, 8)
    pool.seq_create(0)
    pool.seq_append_tokens(0, 8)                 # blocks 0, 1 full
    pool.seq_fork_prefix(1, 0, 8)
    pool.seq_fork_prefix(2, 0, 4)
    assert pool.ref[0] == 3 and pool.ref[1] == 2
    assert pool.seq_append_slots([1, 2]) == [2 * 4 + 0, 3 * 4 + 0]
    pool.seq_free(0)
    assert pool.ref[0] == 2 and pool.ref[1] == 1 and 0 not in pool.free
    pool.seq_free(1)
    assert pool.ref[1] == 0 and list(pool.free)[-2:] == [1, 2]
    pool.seq_free(2)
    assert pool.stats()["used_blocks"] == 0
    assert sorted(pool.free) == list(range(8))


def test_errors():
    pool = P.Pool(1, 1, 8, 4, 2, 2)
    pool.seq_create(0)
    pool.seq_create(1)
    with pytest.raises(P.PoolError) as e:
        pool.seq_create(2)
    assert e.value.status == P.NO_FREE_BLOCK
    pool.seq_append_tokens(0, 4)
    with pytest.raises(P.PoolError) as e:        # needs a block, none free: no change
        pool.seq_append_slots([1, 0])
    assert e.value.status == P.NO_FREE_BLOCK and pool.lens[1] == 0
    with pytest.raises(P.PoolError) as e:
        pool.block_free(7)
    assert e.value.status == P.BAD_BLOCK
    pool.seq_free(1)
    with pytest.raises(P.PoolError) as e:
        pool.block_free(1)
    assert e.value.status == P.REFCOUNT
    with pytest.raises(P.PoolError) as e:
        pool.block_ref(1)
    assert e.value.status == P.REFCOUNT
    with pytest.raises(P.PoolError) as e:
        pool.seq_fork_prefix(3, 0, 3)            # not whole blocks
    assert e.value.status == P.INVALID_ARG
    with pytest.raises(P.PoolError) as e:
        pool.seq_append_slots([0, 0])
    assert e.value.status == P.INVALID_ARG
    with pytest.raises(P.PoolError):
        P.Pool(1, 1, 8, 4, 2, 3, initial_free_order=[0, 0, 1])


def test_brute_force_slots_against_position_rule():
    """Random traffic: every live token's slot equals table[pos//bs]*bs + pos%bs,
    no two live tokens share a slot, and used + free = total."""
    r = np.random.default_rng(7)
    bs, nb = 8, 64
    pool = P.Pool(1, 1, 8, bs, 2, nb, initial_free_order=r.permutation(nb).tolist())
    owner = {}
    live = set()
    next_id = 0
    for _ in range(400):
        op = r.integers(0, 4)
        if op == 0 or not live:
            try:
                pool.seq_create(next_id)
                live.add(next_id)
            except P.PoolError:
                pass
            next_id += 1
        elif op in (1, 2):
            sids = sorted(r.choice(sorted(live), size=min(len(live), 3), replace=False).tolist())
            try:
                slots = pool.seq_append_slots(sids)
            except P.PoolError:
                continue
            for s, sl in zip(sids, slots):
                pos = pool.lens[s] - 1
                t = pool.tables[s]
                assert sl == t[pos // bs] * bs + pos % bs
                assert sl not in owner
                owner[sl] = s
        else:
            s = int(r.choice(sorted(live)))
            for sl in [k for k, v in owner.items() if v == s]:
                del owner[sl]
            pool.seq_free(s)
            live.discard(s)
        st = pool.stats()
        assert st["used_blocks"] + st["free_blocks"] == nb
        assert st["used_blocks"] == sum(len(pool.tables[s]) for s in live)
