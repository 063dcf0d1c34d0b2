"""GPU parity of paged_attention_decode_append: the decode kernel writing each
sequence's new token itself gives the same cache bytes and the same output
bytes as reshape_and_cache followed by paged_attention_decode, and the oracle's
result; a slot that is not the last position's is flagged and not written."""
import numpy as np
import pytest

import workloads as W
from tests import gpu_cases as GC

pytestmark = pytest.mark.gpu

TOL = {"bf16": 2e-3, "fp8_e4m3": 1e-2, "int8": 1e-2}


def _prompted(case):
    """Engine with the case's prompts appended (not the step's token)."""
    import torch
    from paged_kv_cache_295_gb300.engine import PagedKVCache
    w = case.w
    eng = PagedKVCache(1, w.num_kv_heads, w.head_dim, w.block_size, case.nb, GC.CODE[w.kv_dtype],
                       initial_free_order=case.order)
    sd = GC.src_dtype(w)
    if eng.k_scale is not None:
        eng.k_scale[0] = torch.from_numpy(case.k_scale[0]).cuda()
        eng.v_scale[0] = torch.from_numpy(case.v_scale[0]).cuda()
    if case.prompt_slots.size:
        eng.append(0, GC.to_torch(case.prompt_k[0], sd), GC.to_torch(case.prompt_v[0], sd),
                   torch.from_numpy(case.prompt_slots).cuda())
    torch.cuda.synchronize()
    return eng


def _both(case, slots, partition, src_dtype=None):
    """(separate calls, fused call): outputs, cache bytes, status words."""
    import torch
    w = case.w
    sd = src_dtype or GC.src_dtype(w)
    kn = GC.to_torch(case.k_new[0], sd)
    vn = GC.to_torch(case.v_new[0], sd)
    q = GC.to_torch(case.q[0], w.q_dtype)
    bt = torch.from_numpy(case.tables).cuda()
    cl = torch.from_numpy(case.lens.astype(np.int32)).cuda()
    sl = torch.from_numpy(np.asarray(slots, dtype=np.int64)).cuda()
    mc = int(case.lens.max())
    res = []
    for fused in (False, True):
        eng = _prompted(case)
        status = torch.zeros(1, dtype=torch.int32, device="cuda")
        if fused:
            out = eng.append_attend(0, q, kn, vn, sl, bt, cl, mc, partition=partition,
                                    device_status=status)
        else:
            eng.append(0, kn, vn, sl, device_status=status)
            out = eng.attend(0, q, bt, cl, mc, partition=partition, device_status=status)
        torch.cuda.synchronize()
        res.append((out.cpu().numpy(), eng.storage.view(torch.uint8).cpu().numpy().reshape(-1),
                    int(status.item())))
    return res


CASES = {
    "bf16_g4": (W.DecodeWorkload("fa_bf16", 24, 16, 4, 128, 16, "bf16", "bf16", seed=31,
                                 ctx_law="fixed"), None),
    "bf16_mha_bs8": (W.DecodeWorkload("fa_mha", 9, 8, 8, 128, 8, "bf16", "bf16", seed=32,
                                      ctx_law="fixed"), None),
    "bf16_d64": (W.DecodeWorkload("fa_d64", 12, 16, 2, 64, 16, "bf16", "bf16", seed=33,
                                  ctx_law="fixed"), None),
    "fp8_g8": (W.DecodeWorkload("fa_fp8", 16, 16, 2, 128, 16, "fp8_e4m3", "bf16", seed=34,
                                ctx_law="fixed"), None),
    "int8_g2": (W.DecodeWorkload("fa_int8", 14, 8, 4, 128, 32, "int8", "bf16", seed=35,
                                 ctx_law="fixed"), None),
    # head_dim 256: the append's K and V rows take two passes of the warp
    "bf16_d256_g2": (W.DecodeWorkload("fa_d256", 10, 8, 4, 256, 16, "bf16", "bf16", seed=36,
                                      ctx_law="fixed"), None),
    # 16 heads per KV head: two CTAs per KV head both copy the new row
    "bf16_g16": (W.DecodeWorkload("fa_g16", 10, 32, 2, 128, 16, "bf16", "bf16", seed=37,
                                  ctx_law="fixed"), None),
}


def _lens(S, seed):
    r = np.random.default_rng(seed)
    lens = r.integers(1, 600, size=S)
    lens[:4] = [1, 2, 64, 65]
    return lens


@pytest.mark.parametrize("name", sorted(CASES))
@pytest.mark.parametrize("partition", [0, 64])
def test_fused_equals_separate_and_oracle(lib, name, partition):
    w, _ = CASES[name]
    case, _ = GC.make_small(w, lens=_lens(w.num_seqs, w.seed), layers=1)
    (o_sep, c_sep, s_sep), (o_fus, c_fus, s_fus) = _both(case, case.step_slots, partition)
    assert s_sep == 0 and s_fus == 0
    assert c_fus.tobytes() == c_sep.tobytes()
    assert o_fus.tobytes() == o_sep.tobytes()
    kc, vc = GC.oracle_caches(case, 0)
    ref = GC.oracle_out(case, 0, kc, vc)
    assert np.abs(o_fus.astype(np.float64) - ref).max() <= TOL[w.kv_dtype]


def test_fused_fp8_from_f32_rows(lib):
    """8-bit caches quantise f32 sources in the decode kernel exactly as the
    append kernel does."""
    import torch
    w = W.DecodeWorkload("fa_fp8_f32", 10, 8, 2, 128, 16, "fp8_e4m3", "bf16", seed=36,
                         ctx_law="fixed")
    case, _ = GC.make_small(w, lens=_lens(10, 36), layers=1)
    r = np.random.default_rng(7)
    k32 = (r.standard_normal((10, 2, 128)) * 3).astype(np.float32)
    v32 = (r.standard_normal((10, 2, 128)) * 3).astype(np.float32)
    q = GC.to_torch(case.q[0], "bf16")
    bt = torch.from_numpy(case.tables).cuda()
    cl = torch.from_numpy(case.lens.astype(np.int32)).cuda()
    sl = torch.from_numpy(case.step_slots).cuda()
    outs = []
    for fused in (False, True):
        eng = _prompted(case)
        kn, vn = torch.from_numpy(k32).cuda(), torch.from_numpy(v32).cuda()
        if fused:
            o = eng.append_attend(0, q, kn, vn, sl, bt, cl, int(case.lens.max()))
        else:
            eng.append(0, kn, vn, sl)
            o = eng.attend(0, q, bt, cl, int(case.lens.max()))
        torch.cuda.synchronize()
        outs.append((o.cpu().numpy().tobytes(), eng.storage.view(torch.uint8).cpu().numpy().tobytes()))
    assert outs[0] == outs[1]


@pytest.mark.parametrize("path", ["simt", "mma"])
def test_two_kernel_fallback_paths_agree(lib, decode_kernel, path):
    decode_kernel(path)
    w, _ = CASES["bf16_g4"]
    case, _ = GC.make_small(w, lens=_lens(w.num_seqs, 5), layers=1)
    (o_sep, c_sep, s_sep), (o_fus, c_fus, s_fus) = _both(case, case.step_slots, 0)
    assert s_sep == 0 and s_fus == 0
    assert c_fus.tobytes() == c_sep.tobytes()
    assert o_fus.tobytes() == o_sep.tobytes()


def test_wrong_slot_is_flagged_and_not_written(lib):
    """A slot other than the block table's slot of position ctx - 1 is not
    written (another partition could be reading it) and flags BAD_SLOT; a
    negative slot appends nothing and flags nothing."""
    import torch
    import paged_kv_cache_295_gb300 as pkv
    w, _ = CASES["bf16_g4"]
    case, _ = GC.make_small(w, lens=_lens(w.num_seqs, 9), layers=1)
    # a sequence whose new token is not the first of its block, so slot - 1 is
    # its own previous position
    wrong = next(i for i, n in enumerate(case.lens) if n >= 2 and (n - 1) % w.block_size != 0)
    skip = next(i for i in range(w.num_seqs) if i != wrong)
    slots = case.step_slots.copy()
    slots[wrong] -= 1
    slots[skip] = -1
    before = _prompted(case).storage.view(torch.uint8).cpu().numpy().reshape(-1)
    _, (o_fus, c_fus, s_fus) = _both(case, slots, 0)
    assert s_fus & pkv.DEV_BAD_SLOT
    row = w.num_kv_heads * w.head_dim * 2          # bytes per slot and plane (bf16)
    plane = case.nb * w.block_size * row
    assert c_fus.size == 2 * plane and before.size == 2 * plane
    for sl in (slots[wrong], case.step_slots[wrong], case.step_slots[skip]):
        for kv in (0, 1):
            a = kv * plane + int(sl) * row
            assert c_fus[a:a + row].tobytes() == before[a:a + row].tobytes()
    # the other sequences' tokens were appended as usual
    other = next(i for i in range(w.num_seqs) if i not in (wrong, skip))
    a = int(case.step_slots[other]) * row
    assert c_fus[a:a + row].tobytes() != before[a:a + row].tobytes()
