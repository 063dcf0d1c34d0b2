"""Pins for the paged prefill oracle.

What pins it (none of these re-types the oracle's formula):
* with no cached prefix (ctx == n) the causal result equals torch's
  scaled_dot_product_attention(is_causal=True) in float64 on unpaged K/V, a
  library routine;
* with a cached prefix it equals SDPA with an explicit boolean mask that lets
  query i see keys 0 .. ctx-n+i; without the causal mask, SDPA with no mask
  (the tutorial's section 4.4 forward over the whole cache);
* a chunk of one token equals the decode oracle, a separate function;
* chunked prefill: running a chunk as two consecutive chunks gives the same
  rows as one chunk;
* bit-identical output under a permutation of the physical blocks;
* brute force with explicit loops and math.exp on tiny inputs;
* planted mistakes (an off-by-one causal limit, query positions counted from
  0 instead of ctx - n) are caught by the pins above.
"""
import math

import numpy as np
import pytest
import torch

import workloads as W
from oracle import attention as A
from oracle import prefill as PF
from tests.test_oracle_attention import paged_from_contiguous


def make_case(seed, lens, nq, hq, hkv, d, bs, dt):
    """Contexts ``lens`` whose last ``nq[s]`` tokens are this call's queries."""
    r = np.random.default_rng(seed)
    K = [W.store(r.standard_normal((L, hkv, d), dtype=np.float32), dt) for L in lens]
    V = [W.store(r.standard_normal((L, hkv, d), dtype=np.float32), dt) for L in lens]
    qs = np.concatenate([[0], np.cumsum(nq)]).astype(np.int64)
    q = W.store(r.standard_normal((int(qs[-1]), hq, d), dtype=np.float32), dt)
    nb = sum(-(-L // bs) for L in lens) + 3
    kc, vc, bt = paged_from_contiguous(K, V, lens, bs, nb, r.permutation(nb).tolist(),
                                       fill=0)
    return q, qs, K, V, kc, vc, bt


def sdpa_rows(q64, K64, V64, n, causal, scale):
    """SDPA on one sequence: ``q64 [n, Hq, D]``, ``K64/V64 [L, Hkv, D]``."""
    L = K64.shape[0]
    qt = torch.from_numpy(q64).permute(1, 0, 2)[None]
    kt = torch.from_numpy(K64).permute(1, 0, 2)[None]
    vt = torch.from_numpy(V64).permute(1, 0, 2)[None]
    if causal and n == L:
        o = torch.nn.functional.scaled_dot_product_attention(qt, kt, vt, is_causal=True,
                                                             scale=scale, enable_gqa=True)
    else:
        mask = None
        if causal:
            i = torch.arange(n)[:, None]
            j = torch.arange(L)[None, :]
            mask = j <= (L - n + i)
        o = torch.nn.functional.scaled_dot_product_attention(qt, kt, vt, attn_mask=mask,
                                                             scale=scale, enable_gqa=True)
    return o[0].permute(1, 0, 2).numpy()


CASES = [  # (lens, nq, Hq, Hkv, D, bs, dtype)
    ([9, 16, 5], [9, 16, 5], 4, 4, 16, 4, "f32"),         # no prefix: SDPA is_causal
    ([23, 40], [7, 40], 8, 2, 32, 8, "bf16"),              # prefix + whole prompt
    ([33, 17, 1, 64], [16, 1, 1, 30], 8, 1, 16, 16, "bf16"),   # MQA, decode-like rows
    ([12, 7], [5, 7], 6, 3, 8, 2, "f32"),
]


@pytest.mark.parametrize("causal", [True, False])
@pytest.mark.parametrize("lens,nq,hq,hkv,d,bs,dt", CASES)
def test_equals_unpaged_sdpa(lens, nq, hq, hkv, d, bs, dt, causal):
    q, qs, K, V, kc, vc, bt = make_case(21, lens, nq, hq, hkv, d, bs, dt)
    scale = 1.0 / math.sqrt(d)
    got = PF.paged_attention_prefill(q, qs, kc, vc, bt, lens, scale, dt, dt, causal=causal)
    sc = float(np.float32(scale))
    for s, L in enumerate(lens):
        a, b = int(qs[s]), int(qs[s + 1])
        ref = sdpa_rows(A.to_f64(q[a:b], dt), A.to_f64(K[s], dt), A.to_f64(V[s], dt),
                        b - a, causal, sc)
        np.testing.assert_allclose(got[a:b], ref, rtol=0, atol=1e-12)


def test_single_token_chunks_equal_decode_oracle():
    lens = [1, 17, 40, 5]
    q, qs, K, V, kc, vc, bt = make_case(3, lens, [1, 1, 1, 1], 8, 2, 16, 8, "bf16")
    pre = PF.paged_attention_prefill(q, qs, kc, vc, bt, lens, 0.25, "bf16", "bf16")
    dec = A.paged_attention_decode(q, kc, vc, bt, lens, 0.25, "bf16", "bf16")
    np.testing.assert_array_equal(pre, dec)


@pytest.mark.parametrize("split", [1, 5, 11])
def test_two_chunks_equal_one_chunk(split):
    """The section 6.2 scheduler's chunking does not change a row's result."""
    L, n = 40, 16
    q, qs, K, V, kc, vc, bt = make_case(5, [L], [n], 4, 2, 16, 8, "bf16")
    whole = PF.paged_attention_prefill(q, qs, kc, vc, bt, [L], 0.3, "bf16", "bf16")
    first = PF.paged_attention_prefill(q[:split], [0, split], kc, vc, bt, [L - n + split],
                                       0.3, "bf16", "bf16")
    second = PF.paged_attention_prefill(q[split:], [0, n - split], kc, vc, bt, [L], 0.3,
                                        "bf16", "bf16")
    np.testing.assert_allclose(np.concatenate([first, second]), whole, rtol=0, atol=1e-14)


def test_block_permutation_is_bit_identical():
    lens, nq = [30, 19], [12, 19]
    q, qs, K, V, kc, vc, bt = make_case(8, lens, nq, 4, 4, 8, 4, "f32")
    base = PF.paged_attention_prefill(q, qs, kc, vc, bt, lens, 0.5, "f32", "f32")
    r = np.random.default_rng(9)
    perm = r.permutation(kc.shape[0])
    inv = np.argsort(perm)
    kc2, vc2 = kc[perm], vc[perm]                 # new block i holds old block perm[i]
    bt2 = np.where(bt >= 0, inv[np.maximum(bt, 0)], -1)
    got = PF.paged_attention_prefill(q, qs, kc2, vc2, bt2, lens, 0.5, "f32", "f32")
    np.testing.assert_array_equal(got, base)


def test_brute_force_loops():
    lens, nq, hq, hkv, d = [6, 4], [3, 4], 4, 2, 3
    q, qs, K, V, kc, vc, bt = make_case(13, lens, nq, hq, hkv, d, 2, "f32")
    got = PF.paged_attention_prefill(q, qs, kc, vc, bt, lens, 0.7, "f32", "f32")
    sc = float(np.float32(0.7))
    for s, L in enumerate(lens):
        n = nq[s]
        Ks, Vs = K[s].astype(float).tolist(), V[s].astype(float).tolist()
        for i in range(n):
            row = int(qs[s]) + i
            for h in range(hq):
                g = h // (hq // hkv)
                qv = q[row, h].astype(float).tolist()
                zs = [sc * sum(qv[e] * Ks[t][g][e] for e in range(d))
                      for t in range(L - n + i + 1)]
                mx = max(zs)
                ws = [math.exp(z - mx) for z in zs]
                tot = sum(ws)
                for e in range(d):
                    ref = sum(w * Vs[t][g][e] for t, w in enumerate(ws)) / tot
                    assert abs(got[row, h, e] - ref) < 1e-12


def test_first_row_without_prefix_is_its_own_v():
    """Causal, no prefix: token 0 sees only itself, so its output is V[0]."""
    q, qs, K, V, kc, vc, bt = make_case(4, [10], [10], 4, 2, 8, 4, "bf16")
    got = PF.paged_attention_prefill(q, qs, kc, vc, bt, [10], 0.4, "bf16", "bf16")
    v0 = A.to_f64(V[0][0], "bf16")
    for h in range(4):
        np.testing.assert_array_equal(got[0, h], v0[h // 2])


def test_planted_mistakes_are_caught(monkeypatch):
    lens, nq = [23, 40], [7, 40]
    q, qs, K, V, kc, vc, bt = make_case(21, lens, nq, 8, 2, 32, 8, "bf16")
    sc = float(np.float32(0.2))

    def max_err():
        got = PF.paged_attention_prefill(q, qs, kc, vc, bt, lens, 0.2, "bf16", "bf16")
        e = 0.0
        for s, L in enumerate(lens):
            a, b = int(qs[s]), int(qs[s + 1])
            ref = sdpa_rows(A.to_f64(q[a:b], "bf16"), A.to_f64(K[s], "bf16"),
                            A.to_f64(V[s], "bf16"), b - a, True, sc)
            e = max(e, float(np.abs(got[a:b] - ref).max()))
        return e

    assert max_err() < 1e-12
    real = PF.attend_rows
    monkeypatch.setattr(PF, "attend_rows",
                        lambda qr, K_, V_, s_, lim: real(qr, K_, V_, s_, [x - 1 for x in lim]))
    assert max_err() > 1e-3          # a row that misses its own key
    monkeypatch.setattr(PF, "attend_rows",
                        lambda qr, K_, V_, s_, lim: real(qr, K_, V_, s_, list(range(len(lim)))))
    assert max_err() > 1e-3          # positions counted from 0, prefix ignored
