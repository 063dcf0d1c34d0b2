"""CPU tests of the C ABI: exported symbols, the C++ pool against the oracle pool,
and host-side argument validation (no kernel launches)."""
import ctypes as C
import os
import re

import numpy as np
import pytest

import workloads as W
from oracle import pool as OP

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def header_functions():
    txt = open(os.path.join(ROOT, "include", "pagedkv.h")).read()
    txt = re.sub(r"/\*.*?\*/", "", txt, flags=re.S)
    names = re.findall(r"^\s*(?:const\s+)?[a-z_0-9]+\s*\*?\s+([a-z_0-9]+)\s*\(", txt, flags=re.M)
    return sorted(set(names))


def test_library_exports_every_header_symbol(lib):
    names = header_functions()
    assert len(names) >= 20
    so = C.CDLL(lib.LIB_PATH)
    missing = [n for n in names if not hasattr(so, n)]
    assert not missing, missing
    assert set(names) <= set(lib._SIGS), set(names) - set(lib._SIGS)


def test_block_bytes_formula(lib):
    assert lib.block_bytes(32, 16, 32, 128, lib.BF16) == 2 * 32 * 16 * 32 * 128 * 2
    assert lib.block_bytes(1, 256, 8, 128, lib.FP8_E4M3) == 2 * 256 * 8 * 128
    assert lib.block_bytes(0, 16, 32, 128, lib.BF16) == -1


def test_pool_sized_from_free_bytes(lib):
    bb = lib.block_bytes(32, 16, 32, 128, lib.BF16)
    p = lib.Pool(32, 32, 128, 16, lib.BF16, num_blocks=0, free_bytes=10 * bb + bb // 2)
    assert p.stats()["total_blocks"] == 10


def test_worked_example_through_c_pool(lib):
    p = lib.Pool(32, 32, 128, 16, lib.BF16, num_blocks=500)
    for s in range(5):
        p.seq_create(s)
        for _ in range(100):
            p.append_slots([s])
    st = p.stats()
    assert (st["used_blocks"], st["free_blocks"]) == (35, 465)
    assert st["utilization"] == pytest.approx(7.0, abs=1e-12)
    assert st["total_bytes"] / 1e9 == pytest.approx(4.194304, rel=1e-15)
    assert st["used_bytes"] / 1e9 == pytest.approx(0.29360128, rel=1e-15)


def _status_of(fn):
    try:
        fn()
        return OP.OK
    except OP.PoolError as e:
        return e.status


def _c_status_of(lib, fn):
    try:
        fn()
        return OP.OK
    except lib.PagedKVError as e:
        return e.status


@pytest.mark.parametrize("seed", [0, 1, 2])
def test_c_pool_replays_oracle_bit_exact(lib, seed):
    """Random op streams on both pools: every outcome, slot, table, refcount and
    the free-list order must match exactly."""
    r = np.random.default_rng(100 + seed)
    bs, nb = [4, 16, 1][seed], 48
    order = r.permutation(nb).tolist()
    o = OP.Pool(1, 2, 16, bs, 2, nb, initial_free_order=order)
    c = lib.Pool(1, 2, 16, bs, lib.BF16, num_blocks=nb, initial_free_order=order)
    o.host_init(24)
    c.host_init(24)
    live, nid = [], 0
    prompts = {}                       # token ids of a few cached prefixes
    for _ in range(600):
        op = int(r.integers(0, 12))
        if op == 10 and live:            # swap a sequence out or back in
            s = int(r.choice(live))
            if s in o.on_host:
                fo, fc = o.seq_swap_in, c.swap_in
            else:
                fo, fc = o.seq_swap_out, c.swap_out
            res_o, res_c = {}, {}
            a = _status_of(lambda: res_o.setdefault("v", fo(s)))
            b = _c_status_of(lib, lambda: res_c.setdefault("v", fc(s)))
            assert a == b
            if a == OP.OK:
                assert [tuple(x) for x in res_o["v"]] == [tuple(x) for x in res_c["v"].tolist()]
            assert (s in o.on_host) == c.is_swapped(s)
            continue
        if op == 11:
            assert o.lru_order() == c.lru_order()
            continue
        if op == 0 or not live:
            a = _status_of(lambda: o.seq_create(nid))
            b = _c_status_of(lib, lambda: c.seq_create(nid))
            assert a == b
            if a == OP.OK:
                live.append(nid)
            nid += 1
        elif op in (1, 2):
            k = int(r.integers(1, len(live) + 1))
            sids = r.choice(live, size=k, replace=False).tolist()
            res_o, res_c = {}, {}
            a = _status_of(lambda: res_o.setdefault("v", o.seq_append_slots(sids)))
            b = _c_status_of(lib, lambda: res_c.setdefault("v", c.append_slots(sids)))
            assert a == b
            if a == OP.OK:
                assert res_o["v"] == res_c["v"].tolist()
        elif op == 3:
            s = int(r.choice(live))
            n = int(r.integers(0, 3 * bs + 2))
            res_o, res_c = {}, {}
            a = _status_of(lambda: res_o.setdefault("v", o.seq_append_tokens(s, n)))
            b = _c_status_of(lib, lambda: res_c.setdefault("v", c.append_tokens(s, n)))
            assert a == b
            if a == OP.OK:
                assert res_o["v"] == res_c["v"].tolist()
        elif op == 4:
            src = int(r.choice(live))
            ntok = int(r.integers(0, o.lens[src] + 2))       # 0 and len+1 are refused
            a = _status_of(lambda: o.seq_fork_prefix(nid, src, ntok))
            b = _c_status_of(lib, lambda: c.seq_fork_prefix(nid, src, ntok))
            assert a == b
            if a == OP.OK:
                live.append(nid)
            nid += 1
        elif op == 5:
            s = int(r.choice(live))
            o.seq_free(s)
            c.seq_free(s)
            live.remove(s)
        elif op == 7:                    # the copy-on-write queue, drained on both
            assert [tuple(x) for x in o.take_copies()] == [tuple(x) for x in
                                                           c.take_copies().tolist()]
        elif op == 8:                    # cache a prefix of a live sequence
            s = int(r.choice(live))
            if o.lens[s]:
                toks = r.integers(0, 4, size=int(r.integers(1, o.lens[s] + 1))).tolist()
                a = _status_of(lambda: o.prefix_insert(toks, s))
                b = _c_status_of(lib, lambda: c.prefix_insert(toks, s))
                assert a == b
                if a == OP.OK:
                    prompts[tuple(toks)] = True
        elif op == 9 and prompts:        # look up / start from / release a prefix
            key = list(list(prompts)[int(r.integers(0, len(prompts)))])
            q = key + r.integers(0, 4, size=int(r.integers(0, 3))).tolist()
            kind = int(r.integers(0, 3))
            if kind == 0:
                hit = o.prefix_lookup(q)
                assert c.prefix_lookup(q) == ((hit[1], hit[0]) if hit else (0, []))
            elif kind == 1:
                res_o, res_c = {}, {}
                a = _status_of(lambda: res_o.setdefault("v", o.seq_create_from_prefix(nid, q)))
                b = _c_status_of(lib, lambda: res_c.setdefault("v",
                                                              c.seq_create_from_prefix(nid, q)))
                assert a == b and res_o.get("v") == res_c.get("v")
                if a == OP.OK:
                    live.append(nid)
                nid += 1
            else:
                a = _status_of(lambda: o.prefix_release(key))
                b = _c_status_of(lib, lambda: c.prefix_release(key))
                assert a == b
                if o.prefix_count(key) == 0:
                    prompts.pop(tuple(key), None)
            assert o.prefix_count(key) == c.prefix_count(key)
        else:
            b_id = int(r.integers(-1, nb + 1))
            if r.integers(0, 2):
                a = _status_of(lambda: o.block_ref(b_id))
                b = _c_status_of(lib, lambda: c.block_ref(b_id))
            else:
                a = _status_of(lambda: o.block_free(b_id)) if b_id < 0 or b_id >= nb or \
                    o.ref[b_id] == 0 else "skip"
                b = _c_status_of(lib, lambda: c.block_free(b_id)) if a != "skip" else "skip"
            assert a == b
        assert list(o.free) == c.free_list()
        for s in live:
            assert o.tables[s] == c.block_table(s)
            assert o.lens[s] == c.seq_length(s)
        assert o.lru_order() == c.lru_order()
        so, sc = o.stats(), c.stats()
        assert (so["used_blocks"], so["free_blocks"]) == (sc["used_blocks"], sc["free_blocks"])
    for b_id in range(nb):
        assert o.ref[b_id] == c.refcount(b_id)
    live = [s for s in live if s not in o.on_host]
    if live:
        mb = max(len(o.tables[s]) for s in live)
        t_c, l_c = c.batch_tables(live, mb)
        t_o, l_o = o.padded_tables(live, mb)
        assert (t_c == np.asarray(t_o)).all() and (l_c == np.asarray(l_o)).all()


def test_tiny_workload_slots_match_hand_reading(lib):
    """Tiny workload: after the prompts, the step's slots are table[2]*16+4 and table[4]*16+5."""
    w = W.TINY
    lens = W.context_lens(w)
    order = W.free_order(w, 16)
    p = lib.Pool(1, w.num_kv_heads, w.head_dim, w.block_size, lib.F32, num_blocks=16,
                 initial_free_order=order)
    for s, L in enumerate(lens):
        p.seq_create(s)
        p.append_tokens(s, int(L) - 1, want_slots=False)
    slots = p.append_slots([0, 1])
    assert slots.tolist() == [int(order[2]) * 16 + 4, int(order[7]) * 16 + 5]
    assert p.stats()["used_blocks"] == 8


def test_pool_error_codes(lib):
    p = lib.Pool(1, 1, 16, 4, lib.BF16, num_blocks=2)
    p.seq_create(0)
    p.seq_create(1)
    with pytest.raises(lib.PagedKVError) as e:
        p.seq_create(2)
    assert e.value.status == "no_free_block"
    with pytest.raises(lib.PagedKVError) as e:
        p.block_free(9)
    assert e.value.status == "bad_block"
    with pytest.raises(lib.PagedKVError) as e:
        p.append_slots([0, 0])
    assert e.value.status == "invalid_arg"
    p.seq_free(1)
    with pytest.raises(lib.PagedKVError) as e:
        p.block_free(1)
    assert e.value.status == "refcount"
    with pytest.raises(lib.PagedKVError):
        lib.Pool(1, 1, 16, 4, lib.BF16, num_blocks=3, initial_free_order=[0, 0, 1])


def test_device_calls_reject_bad_arguments_before_launch(lib):
    so = lib.library()
    # group not a divisor, no pointers touched
    st = so.paged_attention_decode(None, None, None, None, None, 2, 6, 4, 128, 16, 10, 4, 64,
                                   0.1, lib.BF16, lib.BF16, None, None, None, None, 0, 0, None,
                                   None)
    assert st == 1
    # block size not a power of two
    st = so.paged_attention_decode(None, None, None, None, None, 2, 4, 4, 128, 12, 10, 4, 48,
                                   0.1, lib.BF16, lib.BF16, None, None, None, None, 0, 0, None,
                                   None)
    assert st == 5
    # unsupported group size 3
    st = so.paged_attention_decode(None, None, None, None, None, 2, 12, 4, 128, 16, 10, 4, 64,
                                   0.1, lib.BF16, lib.BF16, None, None, None, None, 0, 0, None,
                                   None)
    assert st == 5
    # context longer than the table
    st = so.paged_attention_decode(None, None, None, None, None, 2, 4, 4, 128, 16, 10, 4, 65,
                                   0.1, lib.BF16, lib.BF16, None, None, None, None, 0, 0, None,
                                   None)
    assert st == 1
    # unsupported append dtype pair (fp8 -> bf16)
    st = so.reshape_and_cache(None, None, None, None, None, 1, 1, 128, 16, 4, lib.FP8_E4M3,
                              lib.BF16, None, None, None, None)
    assert st in (1, 5)


def test_workspace_formula(lib):
    # explicit partition: S * Hq * ceil(ctx/P) * (D+2) * 4
    assert lib.workspace_bytes(8, 32, 8, 128, 131072, 2048) == 8 * 32 * 64 * 130 * 4
    assert lib.workspace_bytes(8, 32, 8, 128, 2048, 2048) == 0
    assert lib.partition_tokens(8, 32, 8, 1000, 192) == 192
    assert lib.partition_tokens(8, 32, 8, 1000, 100) == 0
    assert lib.partition_tokens(8, 30, 8, 1000, 0) == 0          # Hq not a multiple of Hkv


def test_auto_partition_floor_grows_with_group(lib):
    """The automatic partition is a power of two in [256, 4096] and at least
    256 * G tokens (the partials' share of the traffic grows with G)."""
    for S, hq, hkv, ctx in [(32, 32, 32, 4085), (64, 64, 8, 8117), (8, 32, 8, 128932),
                            (1, 8, 8, 10), (256, 32, 32, 16384), (4, 128, 8, 300)]:
        P = lib.partition_tokens(S, hq, hkv, ctx, 0)
        G = hq // hkv
        assert 256 <= P <= 4096 and P & (P - 1) == 0
        assert P >= min(256 * G, 4096)
    assert lib.partition_tokens(64, 64, 8, 8117, 0) >= 2048        # 70B-shaped GQA-8 layer


def test_auto_partition_long_contexts_take_longer_partitions(lib):
    """Past 32 partitions per sequence the partition doubles (up to 4096)
    while the doubled grid keeps two waves of three CTAs per SM (152 SMs)."""
    assert lib.partition_tokens(8, 32, 8, 128932, 0) == 4096        # 64 -> 32 partitions
    assert lib.partition_tokens(1, 32, 8, 128932, 0) == 1024        # too few CTAs to double
    assert lib.partition_tokens(32, 32, 32, 4085, 0) == 1024        # 4 partitions: unchanged
    assert lib.partition_tokens(64, 64, 8, 8117, 0) == 2048         # 4 partitions: unchanged


def test_auto_partition_small_batches_fill_one_wave(lib):
    """Below 1024 tokens the partition doubles while the grid still fills one
    wave of three CTAs per SM (152 SMs here and without a device)."""
    assert lib.partition_tokens(2, 32, 32, 974, 0) == 256          # 256 items at 256 already
    assert lib.partition_tokens(8, 32, 32, 974, 0) == 512          # 512 items at 512
    assert lib.partition_tokens(32, 32, 32, 974, 0) == 1024        # one partition each
    assert lib.partition_tokens(32, 32, 32, 4085, 0) == 1024       # large work: unchanged


def test_prefill_argument_checks(lib):
    """paged_attention_prefill's checks, all before any device work: an fp32 cache
    is unsupported; an INT8 cache is accepted (an empty chunk returns OK right
    after the type checks); 8-bit caches (FP8 and INT8) need both scales.  The
    calls run in a child process that sees no GPU, so the 16-byte aligned
    placeholder addresses could never reach a kernel even if a check moved
    behind a launch (that call would return CUDA instead)."""
    import subprocess
    import sys
    code = f"""
import sys
sys.path.insert(0, {ROOT!r})
import paged_kv_cache_295_gb300 as lib
so = lib.library()
fake = 0x100000
def call(kv, scales, max_q=8):
    ks = fake if scales else None
    return so.paged_attention_prefill(fake, fake, fake, fake, fake, fake, 1, 8, max_q, 8, 2,
                                      128, 16, 64, 4, 64, 0.1, 1, lib.BF16, kv, ks, ks, fake,
                                      None, None)
print(call(lib.F32, True), call(lib.INT8, True, max_q=0), call(lib.FP8_E4M3, False),
      call(lib.INT8, False))
"""
    env = dict(os.environ, CUDA_VISIBLE_DEVICES="")
    r = subprocess.run([sys.executable, "-c", code], env=env, capture_output=True, text=True,
                       timeout=120)
    assert r.returncode == 0, r.stderr
    # UNSUPPORTED; accepted (nothing to do); INVALID_ARG twice (scales required)
    assert r.stdout.split() == ["5", "0", "1", "1"]


def test_decode_test_hooks_check_their_arguments(lib):
    """The kernel choice and the barrier stall used by the GPU tests refuse
    unknown values and leave the setting unchanged (host only)."""
    so = lib.library()
    assert lib.STATUS[so.pkv_test_force_decode_kernel(3)] == "invalid_arg"
    assert lib.STATUS[so.pkv_test_force_decode_kernel(-1)] == "invalid_arg"
    for k in (1, 2, 0):
        assert so.pkv_test_force_decode_kernel(k) == 0
    assert lib.STATUS[so.pkv_test_decode_stall(8)] == "invalid_arg"
    assert lib.STATUS[so.pkv_test_decode_stall(65552)] == "invalid_arg"
    assert so.pkv_test_decode_stall(0) == 0
