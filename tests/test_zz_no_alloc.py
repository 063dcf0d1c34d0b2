"""paged_attention_decode_noalloc: decode without any device allocation.

Some callers may not allocate device memory at all (a plug-in whose host
program owns every allocation, a runtime that fixes its memory plan at
start-up, code that cannot afford the synchronisation an allocation brings).
For them the library keeps its split-KV scratch in a fixed device array.  These
tests call that entry point through the C ABI and compare it with the regular
paged_attention_decode (caller-supplied workspace) on the same inputs, twice in
a row so that whatever the first call left in the shared array cannot leak into
the second.  This file is collected last on purpose.
"""
import ctypes as C
import dataclasses

import numpy as np
import pytest

import workloads as W
from tests import gpu_cases as GC

pytestmark = pytest.mark.gpu

TOL = 2e-3   # max-abs tolerance the parity tests use for bf16 / f32 caches


def _ptr(t):
    return C.c_void_p(t.data_ptr()) if t is not None else None


def _noalloc(lib, torch, q, eng, tables, lens, max_ctx, out, partition, status):
    so = lib.library()
    S, hq, d = q.shape
    kc, vc = eng.k_cache(0), eng.v_cache(0)
    nb, bs, hkv, _ = kc.shape
    return so.paged_attention_decode_noalloc(
        _ptr(q), _ptr(kc), _ptr(vc), _ptr(tables), _ptr(lens), S, hq, hkv, d, bs, nb,
        tables.shape[1], max_ctx, eng.scale, lib.BF16 if q.dtype == torch.bfloat16 else lib.F32,
        eng.kv_dtype, None, None, _ptr(out), partition, _ptr(status),
        C.c_void_p(torch.cuda.current_stream().cuda_stream))


@pytest.mark.parametrize("partition", [64, 0])
def test_noalloc_matches_workspace_entry_point_twice(lib, partition):
    import torch
    assert torch.cuda.is_available()
    w = dataclasses.replace(W.LLAMA7B_LAYER, num_seqs=6)
    lens = [1, 16, 17, 255, 256, 700]
    case, _ = GC.make_small(w, lens=lens)
    eng, _, _ = GC.run_gpu(case)
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
        q = GC.to_torch(W.store(q32, "bf16"), "bf16")
        ref = lib.paged_attention_decode(q, eng.k_cache(0), eng.v_cache(0), tables, ctx, eng.scale,
                                         max_ctx, partition=partition)
        out = torch.full_like(ref, float("nan"))
        st = _noalloc(lib, torch, q, eng, tables, ctx, max_ctx, out, partition, status)
        torch.cuda.synchronize()
        assert st == 0, lib.STATUS.get(st, st)
        assert status.item() == 0
        got, want = out.cpu().numpy(), ref.cpu().numpy()
        assert np.isfinite(got).all()
        assert np.abs(got - want).max() <= TOL, f"call {call}"
        assert got.tobytes() == want.tobytes(), f"call {call}: same kernels, same bits"


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
