"""Pins for the attention and append oracle.

What pins it (none of these re-types the oracle's formula):
* equality with unpaged contiguous attention computed by torch's
  scaled_dot_product_attention in float64 (a library routine; enable_gqa maps
  query head h to KV head h // G, the page's repeat_interleave);
* bit-identical output under a random permutation of the physical blocks;
* context length 1 -> the output is that token's V row, exactly;
* constant V rows -> the output is that row;
* brute force with explicit loops and math.exp on the tiny workload;
* planted mistakes (in a copy of the oracle, on the CPU) are caught.
"""
import math

import numpy as np
import pytest
import torch

import workloads as W
from oracle import attention as A
from oracle import fp8
from oracle import pool as P


def paged_from_contiguous(K, V, lens, bs, nb, order, fill=np.nan):
    """Scatter contiguous per-sequence rows into a paged cache (test-side).

    ``K``/``V``: list of ``[L_s, Hkv, D]`` arrays (any dtype).  Slots come from
    the oracle allocator fed one prompt per sequence.
    """
    hkv, d = K[0].shape[1], K[0].shape[2]
    pool = P.Pool(1, hkv, d, bs, 2, nb, initial_free_order=order)
    kc = np.full((nb, bs, hkv, d), fill, dtype=K[0].dtype)
    vc = np.full((nb, bs, hkv, d), fill, dtype=K[0].dtype)
    for s, L in enumerate(lens):
        pool.seq_create(s)
        slots = pool.seq_append_tokens(s, int(L))
        for i, sl in enumerate(slots):
            kc[sl // bs, sl % bs] = K[s][i]
            vc[sl // bs, sl % bs] = V[s][i]
    mb = max(len(pool.tables[s]) for s in range(len(lens)))
    rows, _ = pool.padded_tables(list(range(len(lens))), mb, pad=-1)
    return kc, vc, np.asarray(rows, dtype=np.int64)


def sdpa_contiguous(q64, K64, V64, scale):
    """torch SDPA, float64, one query token, GQA by enable_gqa."""
    out = []
    for s in range(len(K64)):
        q = torch.from_numpy(q64[s])[None, :, None, :]
        k = torch.from_numpy(K64[s]).permute(1, 0, 2)[None]
        v = torch.from_numpy(V64[s]).permute(1, 0, 2)[None]
        o = torch.nn.functional.scaled_dot_product_attention(q, k, v, scale=scale,
                                                             enable_gqa=True)
        out.append(o[0, :, 0, :].numpy())
    return np.stack(out)


CASES = [  # (S, Hq, Hkv, D, bs, dtype, lens)
    (3, 4, 4, 16, 4, "f32", [1, 9, 16]),
    (2, 8, 2, 32, 8, "bf16", [23, 40]),
    (4, 8, 1, 16, 16, "bf16", [5, 16, 17, 33]),
    (2, 6, 3, 8, 2, "f32", [7, 1]),
]


@pytest.mark.parametrize("S,hq,hkv,d,bs,dt,lens", CASES)
def test_equals_unpaged_sdpa(S, hq, hkv, d, bs, dt, lens):
    r = np.random.default_rng(11)
    K = [W.store(r.standard_normal((L, hkv, d), dtype=np.float32), dt) for L in lens]
    V = [W.store(r.standard_normal((L, hkv, d), dtype=np.float32), dt) for L in lens]
    q = W.store(r.standard_normal((S, hq, d), dtype=np.float32), dt)
    nb = sum(-(-L // bs) for L in lens) + 3
    kc, vc, bt = paged_from_contiguous(K, V, lens, bs, nb, r.permutation(nb).tolist(),
                                       fill=0)
    scale = 1.0 / math.sqrt(d)
    got = A.paged_attention_decode(q, kc, vc, bt, lens, scale, dt, dt)
    ref = sdpa_contiguous(A.to_f64(q, dt), [A.to_f64(k, dt) for k in K],
                          [A.to_f64(v, dt) for v in V], float(np.float32(scale)))
    np.testing.assert_allclose(got, ref, rtol=0, atol=1e-12)


def test_fp8_equals_unpaged_sdpa_on_dequantised():
    r = np.random.default_rng(12)
    S, hq, hkv, d, bs, lens = 3, 4, 2, 32, 8, [9, 30, 64]
    K32 = [r.standard_normal((L, hkv, d), dtype=np.float32) for L in lens]
    V32 = [r.standard_normal((L, hkv, d), dtype=np.float32) for L in lens]
    ks = np.array([0.011, 0.007], dtype=np.float32)
    vs = np.array([0.009, 0.013], dtype=np.float32)
    # codes via torch's float8 conversion (independent of the oracle encoder)
    enc = lambda x, s: torch.from_numpy((x / s[None, :, None]).astype(np.float32)).to(
        torch.float8_e4m3fn).view(torch.uint8).numpy()
    Kc = [enc(k, ks) for k in K32]
    Vc = [enc(v, vs) for v in V32]
    q = W.store(r.standard_normal((S, hq, d), dtype=np.float32), "bf16")
    nb = sum(-(-L // bs) for L in lens)
    kc, vc, bt = paged_from_contiguous(Kc, Vc, lens, bs, nb, r.permutation(nb).tolist(),
                                       fill=0x7F)
    got = A.paged_attention_decode(q, kc, vc, bt, lens, 0.125, "bf16", "fp8_e4m3", ks, vs)
    deq = lambda c, s: (torch.from_numpy(c).view(torch.float8_e4m3fn).float()
                        * torch.from_numpy(s)[None, :, None]).double().numpy()
    ref = sdpa_contiguous(A.to_f64(q, "bf16"), [deq(k, ks) for k in Kc],
                          [deq(v, vs) for v in Vc], 0.125)
    np.testing.assert_allclose(got, ref, rtol=0, atol=1e-12)


def _random_paged(seed, S=3, hq=8, hkv=2, d=16, bs=4, lens=(5, 12, 3), dt="bf16"):
    r = np.random.default_rng(seed)
    K = [W.store(r.standard_normal((L, hkv, d), dtype=np.float32), dt) for L in lens]
    V = [W.store(r.standard_normal((L, hkv, d), dtype=np.float32), dt) for L in lens]
    q = W.store(r.standard_normal((S, hq, d), dtype=np.float32), dt)
    nb = sum(-(-L // bs) for L in lens) + 2
    kc, vc, bt = paged_from_contiguous(K, V, list(lens), bs, nb, list(range(nb)), fill=0)
    return q, kc, vc, bt, list(lens), K, V


def test_block_permutation_invariance_bit_identical():
    q, kc, vc, bt, lens, _, _ = _random_paged(21)
    base = A.paged_attention_decode(q, kc, vc, bt, lens, 0.25, "bf16", "bf16")
    perm = np.random.default_rng(5).permutation(kc.shape[0])      # new home of block b
    kc2 = np.empty_like(kc)
    vc2 = np.empty_like(vc)
    kc2[perm] = kc
    vc2[perm] = vc
    bt2 = np.where(bt >= 0, perm[np.maximum(bt, 0)], -1)
    got = A.paged_attention_decode(q, kc2, vc2, bt2, lens, 0.25, "bf16", "bf16")
    assert (got.view(np.uint64) == base.view(np.uint64)).all()


def test_context_one_returns_v_row_exactly():
    q, kc, vc, bt, lens, K, V = _random_paged(22, lens=(1, 1, 1))
    got = A.paged_attention_decode(q, kc, vc, bt, lens, 0.25, "bf16", "bf16")
    G = 8 // 2
    for s in range(3):
        for h in range(8):
            assert (got[s, h] == A.to_f64(V[s][0, h // G], "bf16")).all()


def test_constant_v_rows():
    q, kc, vc, bt, lens, _, _ = _random_paged(23, lens=(7, 30, 2))
    row = W.store(np.random.default_rng(1).standard_normal((2, 16), dtype=np.float32), "bf16")
    vc[:] = row[None, None]
    got = A.paged_attention_decode(q, kc, vc, bt, lens, 0.25, "bf16", "bf16")
    want = A.to_f64(row, "bf16")
    for s in range(3):
        for h in range(8):
            np.testing.assert_allclose(got[s, h], want[h // 4], rtol=4e-16, atol=0)


def test_empty_context_gives_zero():
    q, kc, vc, bt, lens, _, _ = _random_paged(24, lens=(0, 5, 0))
    got = A.paged_attention_decode(q, kc, vc, bt, lens, 0.25, "bf16", "bf16")
    assert (got[0] == 0).all() and (got[2] == 0).all() and np.abs(got[1]).sum() > 0


def test_brute_force_loops_tiny_workload():
    """The tiny fp32 workload against explicit loops with math.exp."""
    w = W.TINY
    r = np.random.default_rng(0)
    lens = W.context_lens(w).tolist()
    K = [r.standard_normal((L, w.num_kv_heads, w.head_dim), dtype=np.float32) for L in lens]
    V = [r.standard_normal((L, w.num_kv_heads, w.head_dim), dtype=np.float32) for L in lens]
    q = r.standard_normal((w.num_seqs, w.num_q_heads, w.head_dim), dtype=np.float32)
    kc, vc, bt = paged_from_contiguous(K, V, lens, w.block_size, 16,
                                       W.free_order(w, 16).tolist())
    got = A.paged_attention_decode(q, kc, vc, bt, lens, w.scale, "f32", "f32")
    for s, L in enumerate(lens):
        for h in range(w.num_q_heads):
            z = []
            for t in range(L):
                acc = 0.0
                for i in range(w.head_dim):
                    acc += float(q[s, h, i]) * float(K[s][t, h, i])
                z.append(acc * w.scale)
            m = max(z)
            e = [math.exp(v - m) for v in z]
            tot = sum(e)
            for i in range(w.head_dim):
                o = sum(e[t] * float(V[s][t, h, i]) for t in range(L)) / tot
                assert abs(got[s, h, i] - o) < 1e-13


def test_append_copy_and_fp8_against_torch():
    r = np.random.default_rng(31)
    nb, bs, hkv, d = 6, 4, 2, 16
    kc = np.full((nb, bs, hkv, d), 0x7FC0, np.uint16)
    vc = kc.copy()
    kn = W.store(r.standard_normal((3, hkv, d), dtype=np.float32), "bf16")
    vn = W.store(r.standard_normal((3, hkv, d), dtype=np.float32), "bf16")
    slots = np.array([9, -1, 22])
    A.reshape_and_cache(kn, vn, slots, kc, vc, "bf16", "bf16")
    assert (kc[2, 1] == kn[0]).all() and (vc[5, 2] == vn[2]).all()
    assert (kc[0] == 0x7FC0).all()                       # skipped token wrote nothing
    # FP8: code = E4M3(f32(x) / f32(scale)); torch's cast is an independent encoder
    k8 = np.zeros((nb, bs, hkv, d), np.uint8)
    v8 = k8.copy()
    ks = np.array([0.004, 0.02], np.float32)
    A.reshape_and_cache(kn, vn, slots, k8, v8, "bf16", "fp8_e4m3", ks, ks)
    x = A.to_f64(kn[2], "bf16").astype(np.float32) / ks[:, None]
    x = np.clip(x, -448, 448).astype(np.float32)
    ref = torch.from_numpy(x).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert (k8[5, 2] == ref).all()


# -- planted mistakes: a wrong oracle must fail the pins above ------------------
def _wrong_gqa_attend(q_heads, K, V, scale):
    hq, d = q_heads.shape
    hkv = K.shape[1]
    out = np.zeros((hq, d))
    if K.shape[0] == 0:
        return out
    for h in range(hq):
        g = h % hkv                                       # planted: wrong head map
        z = scale * (K[:, g, :] @ q_heads[h])
        p = np.exp(z - z.max())
        out[h] = (p / p.sum()) @ V[:, g, :]
    return out


def _wrong_gather(cache, table, seq_len):
    bs = cache.shape[1]
    nb = seq_len // bs                                    # planted: drops the ragged tail
    parts = [cache[int(table[j])] for j in range(nb)]
    return np.concatenate(parts, 0) if parts else cache[:0, 0]


@pytest.mark.parametrize("planted", ["gqa", "gather"])
def test_planted_mistakes_are_caught(monkeypatch, planted):
    if planted == "gqa":
        monkeypatch.setattr(A, "attend_one", _wrong_gqa_attend)
    else:
        monkeypatch.setattr(A, "gather_sequence", _wrong_gather)
    with pytest.raises(AssertionError):
        test_equals_unpaged_sdpa(*CASES[1])
