"""Pins for the INT8 KV codec of the oracle ("LLM inference tutorial" section
3.1 symmetric quantisation with bits = 8).

What pins it: torch's own round / clamp / int8 cast on float32 tensors (a
library routine, independent of the numpy code), the exact round trip of every
code, the round-half-to-even cases, saturation, and attention over an INT8
cache equal to torch SDPA over the dequantised rows (different K and V scales,
so swapping them fails).
"""
import math

import numpy as np
import pytest
import torch

import workloads as W
from oracle import attention as A
from tests.test_oracle_attention import paged_from_contiguous


def test_encode_matches_torch_round_clamp():
    r = np.random.default_rng(0)
    x = (r.standard_normal((4000, 4, 16)) * 60).astype(np.float32)
    x[::7] = np.float32(3.5)                    # halfway after dividing by 1
    scale = np.array([1.0, 0.37, 2.5, 1e-3], dtype=np.float32)
    got = A.int8_encode(x, scale)
    q = torch.from_numpy(x) / torch.from_numpy(scale)[:, None]
    ref = torch.round(q).clamp(-128, 127).to(torch.int8).numpy()
    assert np.array_equal(got, ref)


def test_every_code_round_trips():
    codes = np.arange(-128, 128, dtype=np.int8).reshape(-1, 1, 1).repeat(3, axis=1)
    for s in (1.0, 0.0123, 7.5):
        scale = np.full(3, s, dtype=np.float32)
        x = codes.astype(np.float32) * scale[None, :, None]
        assert np.array_equal(A.int8_encode(x, scale), codes)
        assert np.array_equal(A.int8_dequant(codes, scale), x.astype(np.float64))


def test_halfway_saturation_and_nan():
    one = np.ones(1, dtype=np.float32)
    x = np.array([0.5, 1.5, 2.5, -0.5, -1.5, 126.5, 127.5, 300.0, -128.5, -1e9, np.nan,
                  np.inf, -np.inf], dtype=np.float32).reshape(-1, 1, 1)
    got = A.int8_encode(x, one)[:, 0, 0].tolist()
    assert got == [0, 2, 2, 0, -2, 126, 127, 127, -128, -128, 0, 127, -128]


@pytest.mark.parametrize("hq,hkv", [(4, 4), (8, 2)])
def test_int8_attention_equals_sdpa_on_dequantised_rows(hq, hkv):
    r = np.random.default_rng(hq)
    d, bs, lens = 16, 4, [9, 17]
    ks = np.linspace(0.01, 0.05, hkv).astype(np.float32)
    vs = np.linspace(0.03, 0.02, hkv).astype(np.float32)
    K = [A.int8_encode(r.standard_normal((L, hkv, d)).astype(np.float32), ks) for L in lens]
    V = [A.int8_encode(r.standard_normal((L, hkv, d)).astype(np.float32), vs) for L in lens]
    q = r.standard_normal((2, hq, d)).astype(np.float32)
    nb = 12
    kc, vc, bt = paged_from_contiguous(K, V, lens, bs, nb, r.permutation(nb).tolist(), fill=0)
    got = A.paged_attention_decode(q, kc, vc, bt, lens, 0.25, "f32", "int8", ks, vs)
    for s, L in enumerate(lens):
        kd = torch.from_numpy(K[s].astype(np.float32) * ks[None, :, None]).double()
        vd = torch.from_numpy(V[s].astype(np.float32) * vs[None, :, None]).double()
        o = torch.nn.functional.scaled_dot_product_attention(
            torch.from_numpy(q[s]).double()[None, :, None, :], kd.permute(1, 0, 2)[None],
            vd.permute(1, 0, 2)[None], scale=float(np.float32(0.25)), enable_gqa=True)
        np.testing.assert_allclose(got[s], o[0, :, 0, :].numpy(), rtol=0, atol=1e-12)


def test_scale_rule():
    assert W.int8_scale_from_absmax(np.array([127.0, 0.0]))[0] == np.float32(1.0)
    assert W.int8_scale_from_absmax(np.array([127.0, 0.0]))[1] == np.float32(1.0)
    assert math.isclose(float(W.int8_scale_from_absmax(np.array([2.54]))[0]), 0.02, rel_tol=1e-6)
