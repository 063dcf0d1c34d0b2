"""GPU parity: the C-ABI library against the oracle on seeded small decode steps.

Slots, tables and cache bytes must be bit-exact; attention outputs within the
stated max-abs tolerances (2e-3 for bf16/f32 KV, 1e-2 for FP8 and INT8 KV: the
8-bit paths carry q * k_scale and P as fp16, like the FP8 bound).
"""
import dataclasses

import numpy as np
import pytest

import workloads as W
from oracle import attention as OA
from tests import gpu_cases as GC

pytestmark = pytest.mark.gpu

TOL = {"f32": 2e-3, "bf16": 2e-3, "fp8_e4m3": 1e-2, "int8": 1e-2}


@pytest.fixture(scope="module")
def torch_cuda(lib):
    import torch
    if not torch.cuda.is_available():
        pytest.fail("CUDA device required for -m gpu tests")
    return torch


def _check_layer(case, eng, outs, layer, tol=None):
    kc, vc = GC.oracle_caches(case, layer)
    w = case.w
    gk = GC.from_torch(eng.k_cache(layer), w.kv_dtype)
    gv = GC.from_torch(eng.v_cache(layer), w.kv_dtype)
    assert gk.tobytes() == kc.tobytes(), "K cache bytes differ from the oracle append"
    assert gv.tobytes() == vc.tobytes(), "V cache bytes differ from the oracle append"
    ref = GC.oracle_out(case, layer, kc, vc)
    got = outs[layer]
    assert np.isfinite(got).all()
    err = np.abs(got.astype(np.float64) - ref).max()
    assert err <= (TOL[w.kv_dtype] if tol is None else tol), f"max abs err {err}"
    return err


def test_tiny_fp32_workload(torch_cuda):
    case, _ = GC.make_small(W.TINY)
    eng, outs, st = GC.run_gpu(case)
    assert st == 0
    err = _check_layer(case, eng, outs, 0, tol=1e-5)
    assert err < 1e-5


SMALL = {
    "llama7b_mha_bf16": (dataclasses.replace(W.LLAMA7B_LAYER, num_seqs=6),
                         [1, 16, 17, 255, 256, 700]),
    "llama70b_gqa8_bf16": (dataclasses.replace(W.LLAMA70B_GQA, num_seqs=4), [1, 128, 129, 1500]),
    "long_ctx_gqa4_bf16": (dataclasses.replace(W.LONG_CTX, num_seqs=2), [5000, 9000]),
    "ragged_fp8_prefix": (dataclasses.replace(W.RAGGED_FP8, num_seqs=10, num_layers=2,
                                              prefix_tokens=64, prefix_seqs=5),
                          [65, 66, 100, 300, 64 + 17, 1, 2, 33, 250, 400]),
    "d64_bf16_g2_bs1": (W.DecodeWorkload("d64g2", 3, 8, 4, 64, 1, "bf16", "bf16", seed=9,
                                         ctx_law="fixed"), [1, 7, 300]),
    "d256_bf16_mha_bs32": (W.DecodeWorkload("d256", 3, 2, 2, 256, 32, "bf16", "f32", seed=10,
                                            ctx_law="fixed"), [31, 32, 333]),
    "d64_fp8_g4_bs8": (W.DecodeWorkload("d64fp8", 3, 8, 2, 64, 8, "fp8_e4m3", "bf16", seed=11,
                                        ctx_law="fixed"), [3, 64, 513]),
    "d128_f32_g8_bs64": (W.DecodeWorkload("f32g8", 2, 16, 2, 128, 64, "f32", "f32", seed=12,
                                          ctx_law="fixed"), [64, 777]),
    "d64_bf16_g16_bs8_qf32": (W.DecodeWorkload("g16", 3, 32, 2, 64, 8, "bf16", "f32", seed=14,
                                               ctx_law="fixed"), [8, 9, 700]),
    "d128_bf16_g1_bs32_qf32": (W.DecodeWorkload("qf32", 3, 4, 4, 128, 32, "bf16", "f32",
                                                seed=15, ctx_law="fixed"), [1, 33, 1000]),
    "d128_bf16_g16_bs16": (W.DecodeWorkload("g16b", 2, 16, 1, 128, 16, "bf16", "bf16",
                                            seed=16, ctx_law="fixed"), [15, 1200]),
    "d256_bf16_g2_bs16": (W.DecodeWorkload("d256g2", 3, 8, 4, 256, 16, "bf16", "bf16",
                                           seed=24, ctx_law="fixed"), [1, 17, 700]),
    "d256_bf16_g16_bs64": (W.DecodeWorkload("d256g16", 2, 32, 2, 256, 64, "bf16", "bf16",
                                            seed=25, ctx_law="fixed"), [65, 1100]),
    "d128_fp8_g8_bs32_qf32": (W.DecodeWorkload("fp8g8", 3, 16, 2, 128, 32, "fp8_e4m3", "f32",
                                               seed=17, ctx_law="fixed"), [2, 31, 900]),
    "d128_fp8_g16_bs8": (W.DecodeWorkload("fp8g16", 2, 32, 2, 128, 8, "fp8_e4m3", "bf16",
                                          seed=18, ctx_law="fixed"), [9, 1300]),
    "d128_fp8_mha_bs16_qf32": (W.DecodeWorkload("fp8g1", 4, 4, 4, 128, 16, "fp8_e4m3", "f32",
                                                seed=23, ctx_law="fixed"), [1, 32, 33, 700]),
    "d128_int8_mha_bs16": (W.DecodeWorkload("i8g1", 4, 4, 4, 128, 16, "int8", "bf16", seed=19,
                                            ctx_law="fixed"), [1, 17, 300, 1000]),
    "d128_int8_g8_bs32_qf32": (W.DecodeWorkload("i8g8", 3, 16, 2, 128, 32, "int8", "f32",
                                                seed=20, ctx_law="fixed"), [2, 31, 900]),
    "d64_int8_g4_bs8": (W.DecodeWorkload("i8d64", 3, 8, 2, 64, 8, "int8", "bf16", seed=21,
                                         ctx_law="fixed"), [3, 64, 513]),
    # the largest block size: contexts inside, at and across 4096-token blocks
    "d128_bf16_g4_bs4096": (W.DecodeWorkload("bs4096", 4, 8, 2, 128, 4096, "bf16", "bf16",
                                             seed=22, ctx_law="fixed"), [1, 4096, 4097, 9000]),
}


@pytest.fixture(params=["auto", "mma", "simt"])
def decode_path(request, decode_kernel):
    """'auto' = the library's own kernel choice (transposed mma.sync kernel for
    groups up to 8); 'mma' skips it for the heads-as-rows mma.sync kernel;
    'simt' forces the CUDA-core kernel everywhere."""
    decode_kernel(request.param)
    return request.param


@pytest.mark.parametrize("name", sorted(SMALL))
@pytest.mark.parametrize("partition", [0, 64])
def test_small_parity(torch_cuda, name, partition, decode_path):
    w, lens = SMALL[name]
    if decode_path == "simt" and w.group > 8:
        pytest.skip("the CUDA-core kernel is built for groups of 1, 2, 4 and 8")
    if decode_path == "mma" and w.group > 8 and w.head_dim > 128:
        pytest.skip("head_dim 256 with 16 heads per KV head runs only on the transposed kernel")
    case, _ = GC.make_small(w, lens=lens)
    eng, outs, st = GC.run_gpu(case, partition=partition)
    assert st == 0
    for layer in range(len(outs)):
        _check_layer(case, eng, outs, layer)


@pytest.mark.parametrize("name", ["ragged_fp8_prefix", "d128_int8_mha_bs16",
                                  "d128_fp8_g8_bs32_qf32", "llama70b_gqa8_bf16"])
def test_q_far_outside_fp16_range(torch_cuda, name, decode_path):
    """Sequences whose q is scaled by 3e5 (past fp16's 65504), 1e-5 (fp16
    subnormal) or 1.  The 8-bit paths carry q in fp16, scaled by a power of two
    into its range; every path must match the oracle on the same q."""
    w, lens = SMALL[name]
    if decode_path == "simt" and w.group > 8:
        pytest.skip("the CUDA-core kernel is built for groups of 1, 2, 4 and 8")
    case, _ = GC.make_small(w, lens=lens)
    mul = np.resize(np.array([3e5, 1e-5, 1.0]), len(case.lens))[:, None, None]
    for layer in range(len(case.q)):
        q = OA.to_f64(case.q[layer], w.q_dtype) * mul
        case.q[layer] = W.store(q.astype(np.float32), w.q_dtype)
    assert np.abs(OA.to_f64(case.q[0], w.q_dtype)).max() > 65504.0
    eng, outs, st = GC.run_gpu(case)
    assert st == 0
    for layer in range(len(outs)):
        _check_layer(case, eng, outs, layer)


def split_invariance_bound(case, kc, vc, path, min_partition=64):
    """How far two split-KV partitionings of one decode step may differ, per
    output element, from the arithmetic of the kernels.

    The logits are the same bits in every partitioning (the same QK products
    on the same 16-token chunks).  What changes is the running max m each
    partition subtracts and the order of the float32 sums.  Against the exact
    result, one partitioning's output out = sum_t p_t v_t / sum_t p_t is then
    off by at most (e_p + e_acc) * (A + |out|) <= 2 (e_p + e_acc) A, where
    A = sum_t p_t |v_t| / sum_t p_t and
      e_p   = 2^-17 >= 2^-22 (ex2.approx) + 2^-19 (rounding of the exponent
              argument s*c - m, |s*c - m| <= 32 where p matters) + 2^-18 (P
              as bf16 hi + lo in the product, against float32 P in the sum);
      e_acc = n * 2^-24 for the n float32 additions on the longest chain:
              one per 16-token chunk on the tensor-core kernels (one per
              token on the CUDA-core kernel), at most 8 for combining the
              warps and the final scaling, and one per partition in the
              reduce (at most ceil(ctx / min_partition)).
    Two partitionings differ by at most twice that: 4 (e_p + e_acc) A."""
    w = case.w
    if w.kv_dtype == "bf16":
        vabs = vc & np.uint16(0x7FFF)
    else:
        vabs = np.abs(vc)
    A = GC.OA.paged_attention_decode(case.q[0], kc, vabs, case.tables, case.lens, w.scale,
                                     w.q_dtype, w.kv_dtype)
    ctx = case.lens.astype(np.float64)
    per_tok = 1.0 if path == "simt" else 1.0 / 16
    n = np.ceil(ctx * per_tok) + 8 + np.ceil(ctx / min_partition)
    eps = 2.0 ** -17 + n * 2.0 ** -24
    return 4 * eps[:, None, None] * A


@pytest.mark.parametrize("name", ["llama7b_mha_bf16", "long_ctx_gqa4_bf16", "d64_bf16_g16_bs8_qf32"])
def test_split_count_invariance(torch_cuda, name, decode_path):
    """The output with one partition per sequence (4096 tokens) and with 64-,
    192-token and automatic partitions differ element by element by no more
    than split_invariance_bound derives from the kernels' arithmetic."""
    w, lens = SMALL[name]
    if decode_path == "simt" and w.group > 8:
        pytest.skip("the CUDA-core kernel is built for groups of 1, 2, 4 and 8")
    case, _ = GC.make_small(w, lens=lens)
    kc, vc = GC.oracle_caches(case, 0)
    bound = split_invariance_bound(case, kc, vc, decode_path)
    _, outs, st = GC.run_gpu(case, partition=4096)
    assert st == 0
    ref = outs[0].astype(np.float64)
    worst = []
    for part in (0, 64, 192):
        _, outs, st = GC.run_gpu(case, partition=part)
        assert st == 0
        err = np.abs(outs[0].astype(np.float64) - ref)
        worst.append((part, float(err.max()), float((err / bound).max())))
        assert (err <= bound).all(), (part, float(err.max()), float((err / bound).max()))
    print(f"split invariance {name} {decode_path}: (partition, max |diff|, max diff/bound) {worst}")


def _decode_sink(k0):
    """Position 0 of every sequence far above the rest (as in the prefill
    test): q is 3 on dimension 0, that key k0 there and 0 elsewhere, the other
    keys (the step's new ones too) scaled by 1/4."""
    def shape(k, v, kn, vn, q, starts):
        q[:, :, 0] = 3.0
        k *= 0.25
        kn *= 0.25
        for s0 in starts:
            k[s0] = 0.0
            k[s0, :, 0] = k0
    return shape


@pytest.mark.parametrize("k0", [67, 49])
@pytest.mark.parametrize("kv", ["int8", "fp8_e4m3", "bf16"])
def test_long_context_with_an_attention_sink(torch_cuda, decode_path, kv, k0):
    """32K tokens and one key far above the rest: the other keys' P lie where
    fp16 (the 8-bit paths' P) keeps few bits or none; the INT8 path's +1152 V
    offset must still come off exactly once."""
    w = W.DecodeWorkload(f"sink_{kv}", 2, 8, 2, 128, 16, kv, "bf16", seed=81, ctx_law="fixed")
    case, _ = GC.make_small(w, lens=[32768, 30001], shape_rows=_decode_sink(k0))
    eng, outs, st = GC.run_gpu(case)
    assert st == 0
    err = _check_layer(case, eng, outs, 0)
    print(f"decode sink {kv} k0={k0} {decode_path}: max abs err {err}")


def test_block_permutation_bit_identical(torch_cuda, decode_path):
    torch = torch_cuda
    w, lens = SMALL["llama7b_mha_bf16"]
    case, _ = GC.make_small(w, lens=lens)
    eng, outs, _ = GC.run_gpu(case)
    perm = np.random.default_rng(3).permutation(case.nb)
    st2 = torch.empty_like(eng.storage)
    st2[:, :, torch.from_numpy(perm).cuda()] = eng.storage
    t2 = np.where(case.tables >= 0, perm[np.maximum(case.tables, 0)], -1).astype(np.int32)
    q = GC.to_torch(case.q[0], w.q_dtype)
    import paged_kv_cache_295_gb300 as pkv
    out2 = pkv.paged_attention_decode(q, st2[0, 0], st2[0, 1], torch.from_numpy(t2).cuda(),
                                      torch.from_numpy(case.lens.astype(np.int32)).cuda(),
                                      w.scale, int(case.lens.max()))
    assert out2.cpu().numpy().tobytes() == outs[0].tobytes()


@pytest.mark.parametrize("partition", [0, 64])
def test_table_entries_past_the_context_are_never_used(torch_cuda, decode_path, partition):
    """Entries at or beyond ceil(ctx / bs) may hold anything: out-of-range ids
    there (the kernels may load them before they know the context) raise no
    flag and change no output bit."""
    torch = torch_cuda
    w, lens = SMALL["llama7b_mha_bf16"]
    case, _ = GC.make_small(w, lens=lens)
    eng, outs, st = GC.run_gpu(case, partition=partition)
    assert st == 0
    t2 = case.tables.copy()
    for s, L in enumerate(case.lens):
        nb = -(-int(L) // w.block_size)
        t2[s, nb:] = np.where(np.arange(t2.shape[1] - nb) % 2 == 0, case.nb + 12345, -77)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    out2 = eng.attend(0, GC.to_torch(case.q[0], w.q_dtype), torch.from_numpy(t2).cuda(),
                      torch.from_numpy(case.lens.astype(np.int32)).cuda(), int(case.lens.max()),
                      partition=partition, device_status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    assert out2.cpu().numpy().tobytes() == outs[0].tobytes()


def test_context_one_and_constant_v(torch_cuda, decode_path):
    torch = torch_cuda
    w = W.DecodeWorkload("c1", 4, 8, 2, 128, 16, "bf16", "bf16", seed=13, ctx_law="fixed")
    case, _ = GC.make_small(w, lens=[1, 1, 40, 90])
    eng, outs, _ = GC.run_gpu(case)
    G = 4
    for s in (0, 1):
        row = GC.OA.to_f64(case.k_new[0][s], "bf16")  # ctx 1: the step's own token
        vrow = GC.OA.to_f64(case.v_new[0][s], "bf16")
        for h in range(8):
            assert np.array_equal(outs[0][s, h].astype(np.float64), vrow[h // G])
        del row
    # constant V rows: overwrite every V slot of the layer with one row per head
    const = GC.W.store(np.random.default_rng(2).standard_normal((2, 128), dtype=np.float32), "bf16")
    eng.v_cache(0)[:] = GC.to_torch(const, "bf16")[None, None]
    import paged_kv_cache_295_gb300 as pkv
    out = eng.attend(0, GC.to_torch(case.q[0], "bf16"),
                     torch.from_numpy(case.tables).cuda(),
                     torch.from_numpy(case.lens.astype(np.int32)).cuda(), 90).cpu().numpy()
    want = GC.OA.to_f64(const, "bf16")
    for s in range(4):
        for h in range(8):
            np.testing.assert_allclose(out[s, h], want[h // G], rtol=1e-5, atol=0)


def test_empty_context_and_status_flags(torch_cuda, decode_path):
    torch = torch_cuda
    w, lens = SMALL["llama7b_mha_bf16"]
    case, _ = GC.make_small(w, lens=lens)
    eng, outs, _ = GC.run_gpu(case)
    import paged_kv_cache_295_gb300 as pkv
    q = GC.to_torch(case.q[0], w.q_dtype)
    lens0 = case.lens.astype(np.int32).copy()
    lens0[2] = 0
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    out = eng.attend(0, q, torch.from_numpy(case.tables).cuda(), torch.from_numpy(lens0).cuda(),
                     int(case.lens.max()), device_status=status).cpu().numpy()
    assert (out[2] == 0).all() and status.item() == 0
    assert out[1].tobytes() == outs[0][1].tobytes()
    # an out-of-range block id is skipped (never read) and flagged
    bad = case.tables.copy()
    bad[5, 3] = case.nb + 7
    out = eng.attend(0, q, torch.from_numpy(bad).cuda(),
                     torch.from_numpy(case.lens.astype(np.int32)).cuda(), int(case.lens.max()),
                     device_status=status).cpu().numpy()
    torch.cuda.synchronize()
    assert status.item() & pkv.DEV_BAD_BLOCK
    assert out[:5].tobytes() == outs[0][:5].tobytes()
    # a context longer than the launch covers is clamped and flagged
    status.zero_()
    lens2 = case.lens.astype(np.int32).copy()
    lens2[0] = 700
    eng.attend(0, q, torch.from_numpy(case.tables).cuda(), torch.from_numpy(lens2).cuda(), 256,
               device_status=status)
    torch.cuda.synchronize()
    assert status.item() & pkv.DEV_BAD_CONTEXT
    # negative slots skip, slots beyond the pool are flagged and skipped
    status.zero_()
    before = eng.storage.clone()
    k1 = GC.to_torch(case.k_new[0][:2], "bf16")
    eng.append(0, k1, k1, torch.tensor([-1, case.nb * 16 + 3], dtype=torch.int64, device="cuda"),
               device_status=status)
    torch.cuda.synchronize()
    assert status.item() & pkv.DEV_BAD_SLOT
    assert torch.equal(before.view(torch.int16), eng.storage.view(torch.int16))


def _halfway_f32():
    from oracle import fp8 as OF8
    vals = sorted(set(OF8.decode_code(c) for c in range(0x00, 0x7F)))
    mids = [(a + b) / 2 for a, b in zip(vals, vals[1:])]
    out = []
    for m in mids:
        m32 = np.float32(m)
        out += [m32, np.nextafter(m32, np.float32(0)), np.nextafter(m32, np.float32(1e9))]
    out += [448.0, 449.0, 464.0, 465.0, 1e6, 2.0 ** -10, 2.0 ** -11, 0.0]
    out = np.array(out, dtype=np.float32)
    return np.concatenate([out, -out])


@pytest.mark.parametrize("scale", [1.0, 0.37])
def test_fp8_append_rounding_bit_exact(torch_cuda, scale):
    """Every E4M3 halfway case (and its neighbours) through the quantising append."""
    torch = torch_cuda
    import paged_kv_cache_295_gb300 as pkv
    from oracle import attention as OA
    x = _halfway_f32() * np.float32(scale)
    hkv, d = 2, 16
    n = -(-x.size // (hkv * d))
    pad = np.zeros(n * hkv * d, np.float32)
    pad[: x.size] = x
    k = pad.reshape(n, hkv, d)
    v = -k
    nb, bs = n, 1
    slots = np.random.default_rng(0).permutation(nb).astype(np.int64)
    sc = np.array([scale, scale], np.float32)
    kc = torch.zeros((nb, bs, hkv, d), dtype=torch.uint8, device="cuda")
    vc = torch.zeros_like(kc)
    pkv.reshape_and_cache(torch.from_numpy(k).cuda(), torch.from_numpy(v).cuda(),
                          torch.from_numpy(slots).cuda(), kc, vc, torch.from_numpy(sc).cuda(),
                          torch.from_numpy(sc).cuda())
    okc = np.zeros((nb, bs, hkv, d), np.uint8)
    ovc = okc.copy()
    OA.reshape_and_cache(k, v, slots, okc, ovc, "f32", "fp8_e4m3", sc, sc)
    assert np.array_equal(kc.cpu().numpy(), okc)
    assert np.array_equal(vc.cpu().numpy(), ovc)


@pytest.mark.parametrize("scale", [1.0, 0.37])
def test_int8_append_rounding_bit_exact(torch_cuda, scale):
    """Every half-integer quotient in and beyond [-128, 127] (and its float32
    neighbours), infinities and NaN through the INT8 quantising append."""
    torch = torch_cuda
    import paged_kv_cache_295_gb300 as pkv
    from oracle import attention as OA
    base = np.arange(-140, 141, dtype=np.float32) + np.float32(0.5)
    x = np.concatenate([base, np.nextafter(base, np.float32(-1e9)),
                        np.nextafter(base, np.float32(1e9)),
                        np.array([0, 127, -128, 1e30, -1e30, np.inf, -np.inf, np.nan],
                                 dtype=np.float32)]) * np.float32(scale)
    hkv, d = 2, 16
    n = -(-x.size // (hkv * d))
    pad = np.zeros(n * hkv * d, np.float32)
    pad[: x.size] = x
    k = pad.reshape(n, hkv, d)
    v = -k
    slots = np.random.default_rng(1).permutation(n).astype(np.int64)
    sc = np.array([scale, scale], np.float32)
    kc = torch.zeros((n, 1, hkv, d), dtype=torch.int8, device="cuda")
    vc = torch.zeros_like(kc)
    pkv.reshape_and_cache(torch.from_numpy(k).cuda(), torch.from_numpy(v).cuda(),
                          torch.from_numpy(slots).cuda(), kc, vc, torch.from_numpy(sc).cuda(),
                          torch.from_numpy(sc).cuda())
    okc = np.zeros((n, 1, hkv, d), np.int8)
    ovc = okc.copy()
    OA.reshape_and_cache(k, v, slots, okc, ovc, "f32", "int8", sc, sc)
    assert np.array_equal(kc.cpu().numpy(), okc)
    assert np.array_equal(vc.cpu().numpy(), ovc)

