"""paged_attention_decode_noalloc: decode without any device allocation.

Some callers may not allocate device memory at all (a plug-in whose host
program owns every allocation, a runtime that fixes its memory plan at
start-up, code that cannot afford the synchronisation an allocation brings).
For them the library keeps its split-KV scratch in a fixed device array.  These
tests call that entry point through the C ABI and compare it with the regular
paged_attention_decode (caller-supplied workspace, NaN-filled) and with the
oracle on the same inputs, twice in a row and then a large call followed by a
smaller one, so that whatever one call left in the shared array cannot leak
into the next.  This file is collected last on purpose.
"""
import ctypes as C
import dataclasses

import numpy as np
import pytest

import workloads as W
from tests import gpu_cases as GC

pytestmark = pytest.mark.gpu

def _ptr(t):
    return C.c_void_p(t.data_ptr()) if t is not None else None


def _noalloc(lib, torch, q, eng, tables, lens, max_ctx, out, partition, status):
    so = lib.library()
    S, hq, d = q.shape
    kc, vc = eng.k_cache(0), eng.v_cache(0)
    nb, bs, hkv, _ = kc.shape
    ks = None if eng.k_scale is None else eng.k_scale[0]
    vs = None if eng.v_scale is None else eng.v_scale[0]
    return so.paged_attention_decode_noalloc(
        _ptr(q), _ptr(kc), _ptr(vc), _ptr(tables), _ptr(lens), S, hq, hkv, d, bs, nb,
        tables.shape[1], max_ctx, eng.scale, lib.BF16 if q.dtype == torch.bfloat16 else lib.F32,
        eng.kv_dtype, _ptr(ks), _ptr(vs), _ptr(out), partition, _ptr(status),
        C.c_void_p(torch.cuda.current_stream().cuda_stream))


def _workspace_call(lib, torch, q, eng, tables, ctx, max_ctx, partition):
    """The regular entry point with its own workspace, filled with NaN first: a
    partial it read without writing would make its output NaN."""
    S, hq, d = q.shape
    need = lib.workspace_bytes(S, hq, eng.num_kv_heads, d, max_ctx, partition)
    ws = torch.full((max(need, 4) // 4,), float("nan"), dtype=torch.float32, device="cuda")
    ks = None if eng.k_scale is None else eng.k_scale[0]
    vs = None if eng.v_scale is None else eng.v_scale[0]
    return lib.paged_attention_decode(q, eng.k_cache(0), eng.v_cache(0), tables, ctx, eng.scale,
                                      max_ctx, k_scale=ks, v_scale=vs, workspace=ws,
                                      partition=partition)


# (name, workload, contexts, tolerance against the oracle)
CASES = {
    "bf16_mha": (dataclasses.replace(W.LLAMA7B_LAYER, num_seqs=6), [1, 16, 17, 255, 256, 700],
                 2e-3),
    "fp8_gqa4": (W.DecodeWorkload("noalloc_fp8", 5, 16, 4, 128, 16, "fp8_e4m3", "bf16", seed=61,
                                  ctx_law="fixed"), [3, 64, 65, 500, 1030], 1e-2),
}


@pytest.mark.parametrize("name", sorted(CASES))
@pytest.mark.parametrize("partition", [64, 0])
def test_noalloc_matches_workspace_entry_point_and_oracle_twice(lib, name, partition):
    """Two calls in a row with different queries: each output is the same bits
    as paged_attention_decode's on the same inputs, and within the parity
    tolerance of the oracle."""
    import torch
    assert torch.cuda.is_available()
    w, lens, tol = CASES[name]
    case, _ = GC.make_small(w, lens=lens)
    eng, _, _ = GC.run_gpu(case)
    kc, vc = GC.oracle_caches(case, 0)
    tables = torch.from_numpy(case.tables).cuda()
    ctx = torch.from_numpy(case.lens.astype(np.int32)).cuda()
    max_ctx = int(case.lens.max())
    need = lib.workspace_bytes(w.num_seqs, w.num_q_heads, w.num_kv_heads, w.head_dim, max_ctx,
                               partition)
    if partition:
        assert need > 0, "the case must exercise the split-KV scratch"
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    rng = np.random.default_rng(77)
    for call in range(2):   # two calls in a row, different queries
        q32 = rng.standard_normal((w.num_seqs, w.num_q_heads, w.head_dim), dtype=np.float32)
        qh = W.store(q32, "bf16")
        q = GC.to_torch(qh, "bf16")
        ref = _workspace_call(lib, torch, q, eng, tables, ctx, max_ctx, partition)
        out = torch.full_like(ref, float("nan"))
        st = _noalloc(lib, torch, q, eng, tables, ctx, max_ctx, out, partition, status)
        torch.cuda.synchronize()
        assert st == 0, lib.STATUS.get(st, st)
        assert status.item() == 0
        got, want = out.cpu().numpy(), ref.cpu().numpy()
        assert np.isfinite(got).all()
        assert got.tobytes() == want.tobytes(), f"call {call}: same kernels, same bits"
        oracle = GC.OA.paged_attention_decode(qh, kc, vc, case.tables, case.lens, w.scale, "bf16",
                                              w.kv_dtype, case.k_scale[0], case.v_scale[0])
        assert np.abs(got.astype(np.float64) - oracle).max() <= tol, f"call {call}"


def test_noalloc_leaves_nothing_for_a_smaller_call(lib):
    """A large call fills much of the array; a smaller one after it, whose
    partials sit at other offsets (fewer sequences, fewer partitions per
    sequence), must equal the workspace entry point on a NaN-filled workspace
    bit for bit - a partial it read without writing would show as a mismatch."""
    import torch
    assert torch.cuda.is_available()
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    big = dataclasses.replace(W.LLAMA7B_LAYER, num_seqs=8)
    small = dataclasses.replace(W.LLAMA7B_LAYER, num_seqs=3, seed=5)
    outs = []
    for w, lens in ((big, [4000, 3000, 2000, 1000, 900, 800, 700, 600]), (small, [1500, 70, 900])):
        case, _ = GC.make_small(w, lens=lens)
        eng, _, _ = GC.run_gpu(case)
        tables = torch.from_numpy(case.tables).cuda()
        ctx = torch.from_numpy(case.lens.astype(np.int32)).cuda()
        max_ctx = int(case.lens.max())
        q = GC.to_torch(case.q[0], "bf16")
        out = torch.full((w.num_seqs, w.num_q_heads, w.head_dim), float("nan"), device="cuda")
        st = _noalloc(lib, torch, q, eng, tables, ctx, max_ctx, out, 64, status)
        ref = _workspace_call(lib, torch, q, eng, tables, ctx, max_ctx, 64)
        torch.cuda.synchronize()
        assert st == 0 and status.item() == 0
        assert out.cpu().numpy().tobytes() == ref.cpu().numpy().tobytes()
        outs.append(out)
    assert np.isfinite(outs[1].cpu().numpy()).all()


def test_noalloc_rejects_requests_beyond_its_scratch(lib):
    import torch
    assert torch.cuda.is_available()
    # 64 sequences x 64 query heads x 128 partitions x (128 + 2) floats > 16 MiB
    S, hq, hkv, d, bs, max_ctx, part = 64, 64, 8, 128, 16, 8192, 64
    need = lib.workspace_bytes(S, hq, hkv, d, max_ctx, part)
    assert need > lib.NOALLOC_SCRATCH_BYTES
    dummy = torch.zeros(1024, dtype=torch.uint8, device="cuda")
    so = lib.library()
    st = so.paged_attention_decode_noalloc(
        _ptr(dummy), _ptr(dummy), _ptr(dummy), _ptr(dummy), _ptr(dummy), S, hq, hkv, d, bs, 10,
        max_ctx // bs, max_ctx, 0.088, lib.BF16, lib.BF16, None, None, _ptr(dummy), part, None,
        None)
    assert lib.STATUS[st] == "scratch_limit"
    assert so.pkv_status_string(st) == b"request exceeds the library's built-in decode scratch"
