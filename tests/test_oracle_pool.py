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
    for bad in (0, 5):                           # nothing to share / beyond the length
        with pytest.raises(P.PoolError) as e:
            pool.seq_fork_prefix(3, 0, bad)
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


def test_copy_on_write_trace():
    """Hand-derived: a beam fork shares a partly filled block; the first write
    into it moves the writer to the free-list front and queues (old, new)."""
    pool = P.Pool(1, 1, 8, 4, 2, 8)
    pool.seq_create(0)                                   # block 0
    assert pool.seq_append_tokens(0, 6) == [0, 1, 2, 3, 4, 5]   # block 1 opened at token 4
    pool.seq_fork_prefix(1, 0, 6)                        # full fork: [0, 1], len 6
    assert pool.ref[0] == 2 and pool.ref[1] == 2
    assert pool.seq_append_slots([1]) == [2 * 4 + 2]     # block 1 shared -> copy into 2
    assert pool.block_table(1) == [0, 2] and pool.ref[1] == 1 and pool.ref[2] == 1
    assert pool.seq_append_slots([0]) == [1 * 4 + 2]     # block 1 is 0's alone now
    assert pool.take_copies() == [(1, 2)] and pool.take_copies() == []
    assert pool.seq_append_tokens(1, 2) == [11, 12]      # block 2 offset 3, then block 3
    pool.seq_free(0)
    assert pool.ref[0] == 1 and pool.ref[1] == 0 and list(pool.free)[-1] == 1


def test_copy_on_write_counts_in_all_or_nothing():
    pool = P.Pool(1, 1, 8, 4, 2, 3)
    pool.seq_create(0)
    pool.seq_append_tokens(0, 2)
    pool.seq_fork_prefix(1, 0, 2)
    pool.seq_create(2)                                   # last free block
    with pytest.raises(P.PoolError) as e:                # both would copy: one block short
        pool.seq_append_slots([0, 1])
    assert e.value.status == P.NO_FREE_BLOCK and pool.lens[0] == 2 and pool.copies == []
    with pytest.raises(P.PoolError) as e:
        pool.seq_append_tokens(1, 3)                     # 1 copy + 1 new block, 1 free
    assert e.value.status == P.NO_FREE_BLOCK and pool.lens[1] == 2
    pool.seq_free(2)
    assert pool.seq_append_tokens(1, 3) and pool.lens[1] == 5 and len(pool.copies) == 1


def _check_beams(seed, bs, nb, steps, drain=True, swaps=False, swap_in_copy=True):
    """Random forks, appends, frees (and swaps) with a cache of token values;
    after every append the copy queue is executed before the writes, and every
    swap's pairs are copied at once.  Returns the largest mismatch between each
    live sequence's gathered cache and its own history."""
    from oracle import attention as A
    r = np.random.default_rng(seed)
    pool = P.Pool(1, 1, 1, bs, 4, nb, initial_free_order=r.permutation(nb).tolist())
    cache = np.full((1, 2, nb, bs, 1, 1), np.nan)
    host = np.full((nb, 1, 2, bs, 1, 1), np.nan)
    if swaps:
        pool.host_init(nb)
    hist, nid, val = {}, 0, 0.0
    for _ in range(steps):
        op = r.integers(0, 8 if swaps else 6)
        live = sorted(s for s in hist if s not in pool.on_host)
        try:
            if op == 6:
                if live:
                    A.swap_blocks(cache, host, pool.seq_swap_out(int(r.choice(live))), True)
                continue
            if op == 7:
                out = sorted(pool.on_host)
                if out:
                    pairs = pool.seq_swap_in(int(r.choice(out)))
                    if swap_in_copy:
                        A.swap_blocks(cache, host, pairs, False)
                continue
            if op == 0 or not live:
                pool.seq_create(nid)
                hist[nid] = []
                nid += 1
            elif op == 1:                                 # fork (beam or prefix)
                src = int(r.choice(live))
                if hist[src]:
                    ntok = int(r.integers(1, len(hist[src]) + 1))
                    pool.seq_fork_prefix(nid, src, ntok)
                    hist[nid] = hist[src][:ntok]
                    nid += 1
            elif op in (2, 3, 4):
                sids = r.choice(live, size=int(r.integers(1, len(live) + 1)),
                                replace=False).tolist()
                slots = pool.seq_append_slots(sids)
                if drain:
                    A.copy_blocks(cache, pool.take_copies())
                for sid, sl in zip(sids, slots):
                    val += 1.0
                    cache[0, :, sl // bs, sl % bs] = val
                    hist[sid].append(val)
            else:
                sid = int(r.choice(live))
                pool.seq_free(sid)
                del hist[sid]
        except P.PoolError as e:
            assert e.status == P.NO_FREE_BLOCK
    for sid in sorted(pool.on_host):
        try:
            A.swap_blocks(cache, host, pool.seq_swap_in(sid), False)
        except P.PoolError:
            pass                        # read from the host slots below
    worst = 0.0
    for sid, h in hist.items():
        on_host = pool.on_host.get(sid, set())
        for kv in (0, 1):
            rows = [host[b, 0, kv] if j in on_host else cache[0, kv, b]
                    for j, b in enumerate(pool.tables[sid])]
            got = (np.concatenate(rows)[: len(h), 0, 0] if rows else np.zeros(0))
            d = np.abs(got - np.asarray(h)) if h else np.zeros(1)
            worst = max(worst, float(np.nan_to_num(d, nan=1e9).max()))
    return worst


@pytest.mark.parametrize("seed,bs", [(0, 4), (1, 1), (2, 16), (3, 3)])
def test_beams_read_back_their_own_history(seed, bs):
    """Every sequence gathers exactly the tokens it appended, whatever was
    forked from it or written by its beams later (copy-on-write invariant)."""
    assert _check_beams(seed, bs, 64, 800) == 0.0


def test_skipping_the_copies_is_caught():
    assert _check_beams(0, 4, 64, 800, drain=False) > 0.0


def test_prefix_cache_trace():
    """Section 4.3: insert with count 1, longest-prefix lookup adds one per hit,
    release takes one off; at zero the entry and its block references go."""
    pool = P.Pool(1, 1, 8, 4, 2, 16)
    toks = [5, 6, 7, 8, 9, 10]
    pool.seq_create(0)
    pool.seq_append_tokens(0, 6)                          # blocks 0, 1
    pool.prefix_insert(toks[:4], 0)                       # block 0
    pool.prefix_insert(toks, 0)                           # blocks 0, 1
    assert pool.ref[0] == 3 and pool.ref[1] == 2
    assert pool.prefix_count(toks[:4]) == 1 and pool.prefix_count(toks) == 1
    assert pool.prefix_lookup(toks + [11, 12]) == ([0, 1], 6)
    assert pool.prefix_lookup([5, 6, 7, 8, 0]) == ([0], 4)
    assert pool.prefix_lookup([5, 6, 7]) is None and pool.prefix_lookup([1]) is None
    assert pool.prefix_count(toks) == 2 and pool.prefix_count(toks[:4]) == 2
    assert pool.seq_create_from_prefix(1, toks + [42]) == 6
    assert pool.block_table(1) == [0, 1] and pool.lens[1] == 6 and pool.ref[1] == 3
    assert pool.seq_append_slots([1]) == [2 * 4 + 2]      # partly filled block 1: copied
    assert pool.take_copies() == [(1, 2)]
    assert pool.seq_create_from_prefix(2, [99]) == 0 and pool.block_table(2) == [3]
    pool.seq_free(0)
    for _ in range(3):
        pool.prefix_release(toks)                         # 3 -> 0: entry dropped
    assert pool.prefix_count(toks) == 0 and pool.ref[1] == 0 and pool.ref[0] == 2   # [:4] entry + seq 1
    with pytest.raises(P.PoolError):
        pool.prefix_release(toks)
    with pytest.raises(P.PoolError):
        pool.prefix_insert(toks[:4], 1)                   # already cached


def test_prefix_lookup_equals_brute_force_scan():
    """The longest cached prefix found by the page's descending loop equals a
    direct scan of every entry."""
    r = np.random.default_rng(5)
    pool = P.Pool(1, 1, 8, 4, 2, 256)
    pool.seq_create(0)
    pool.seq_append_tokens(0, 40)
    entries = set()
    for _ in range(30):
        n = int(r.integers(1, 12))
        e = tuple(int(x) for x in r.integers(0, 3, size=n))
        if e not in entries:
            pool.prefix_insert(list(e), 0)
            entries.add(e)
    for _ in range(300):
        q = [int(x) for x in r.integers(0, 3, size=int(r.integers(0, 15)))]
        best = max((len(e) for e in entries if tuple(q[:len(e)]) == e), default=0)
        hit = pool.prefix_lookup(q)
        assert (hit[1] if hit else 0) == best


@pytest.mark.parametrize("seed,bs", [(0, 4), (1, 1), (2, 16)])
def test_swapped_sequences_read_back_their_history(seed, bs):
    """Swapping out (device -> host copies) and back in (host -> device) in the
    middle of forks and appends never changes what a sequence reads."""
    assert _check_beams(seed, bs, 96, 900, swaps=True) == 0.0


def test_skipping_the_swap_in_copy_is_caught():
    assert _check_beams(0, 4, 96, 900, swaps=True, swap_in_copy=False) > 0.0


def test_swap_trace_and_lru_order():
    """Hand-derived: private blocks go to host slots (FIFO), shared ones stay;
    swap-in takes device blocks from the free-list front; LRU = last append."""
    pool = P.Pool(1, 1, 8, 4, 2, 8)
    pool.host_init(3)
    pool.seq_create(0)
    pool.seq_append_tokens(0, 6)            # blocks 0, 1
    pool.seq_fork_prefix(1, 0, 4)           # shares block 0
    pool.seq_create(2)                      # block 2
    assert pool.lru_order() == [0, 1, 2]
    pool.seq_append_slots([0])
    assert pool.lru_order() == [1, 2, 0]
    assert pool.seq_swap_out(0) == [(1, 0)]          # block 1 private, block 0 shared
    assert pool.tables[0] == [0, 0] and pool.on_host[0] == {1}
    assert list(pool.free)[-1] == 1 and pool.lru_order() == [1, 2]
    with pytest.raises(P.PoolError):
        pool.seq_append_slots([0])                  # swapped out: no appends
    with pytest.raises(P.PoolError):
        pool.padded_tables([0], 4)
    assert pool.seq_swap_in(0) == [(0, 3)]           # free list front is block 3
    assert pool.tables[0] == [0, 3] and list(pool.host_free) == [1, 2, 0]
    assert pool.lru_order() == [1, 2, 0]
    pool.seq_swap_out(2)
    pool.seq_free(2)                                 # its host slot goes back
    assert list(pool.host_free) == [2, 0, 1]


def test_swap_out_is_all_or_nothing():
    pool = P.Pool(1, 1, 8, 4, 2, 8)
    pool.host_init(1)
    pool.seq_create(0)
    pool.seq_append_tokens(0, 8)
    with pytest.raises(P.PoolError) as e:
        pool.seq_swap_out(0)
    assert e.value.status == P.NO_FREE_BLOCK and pool.tables[0] == [0, 1]
