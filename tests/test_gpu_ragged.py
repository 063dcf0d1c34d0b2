"""GPU parity of decode on ragged contexts with every work item accounted for.

The decode grid is (KV head, partition, sequence), KV head fastest, and CTAs
past a sequence's last partition exit at once.  The split-KV workspace and
the output are poisoned with NaN, so a partition that ran twice, never ran, or
wrote outside its slot shows up.  Contexts mix zero, one, whole partitions,
one past and one short of a partition, on every decode kernel.
"""
import numpy as np
import pytest

import workloads as W
from tests import gpu_cases as GC

pytestmark = pytest.mark.gpu

TOL = {"bf16": 2e-3, "fp8_e4m3": 1e-2, "int8": 1e-2}


def _lens(r, S, P, hi):
    lens = r.integers(1, hi, size=S)
    special = [1, P - 1, P, P + 1, 2 * P, 3 * P - 1, hi]
    lens[:len(special)] = special
    return r.permutation(lens)


@pytest.mark.parametrize("path", ["auto", "mma", "simt"])
@pytest.mark.parametrize("kv,S,hkv,G,partition", [
    ("bf16", 70, 2, 4, 64),
    ("bf16", 33, 4, 1, 128),
    ("fp8_e4m3", 40, 2, 8, 64),
    ("int8", 21, 2, 2, 192),
    ("bf16", 24, 2, 4, 4096),     # one partition per sequence
])
def test_ragged_contexts_poisoned_workspace(lib, decode_kernel, path, kv, S, hkv, G, partition):
    import torch
    import paged_kv_cache_295_gb300 as pkv
    decode_kernel(path)
    r = np.random.default_rng(S * 7 + hkv)
    lens = _lens(r, S, min(partition, 256), 700)
    w = W.DecodeWorkload(f"ragged_{kv}", S, hkv * G, hkv, 128, 16, kv, "bf16", seed=S,
                         ctx_law="fixed")
    case, _ = GC.make_small(w, lens=lens)
    eng, _, st = GC.run_gpu(case, partition=partition)
    assert st == 0
    attend = lens.copy()
    attend[[3, S - 2]] = 0                        # empty sequences inside the batch
    max_ctx = int(attend.max())
    need = pkv.workspace_bytes(S, w.num_q_heads, hkv, 128, max_ctx, partition)
    ws = torch.full((max(need, 16) // 4,), float("nan"), dtype=torch.float32, device="cuda")
    out = torch.full((S, w.num_q_heads, 128), float("nan"), dtype=torch.float32, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    eng.attend(0, GC.to_torch(case.q[0], "bf16"), torch.from_numpy(case.tables).cuda(),
               torch.from_numpy(attend.astype(np.int32)).cuda(), max_ctx, out=out,
               workspace=ws, partition=partition, device_status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    got = out.cpu().numpy()
    assert np.isfinite(got).all()
    assert (got[[3, S - 2]] == 0).all()
    kc, vc = GC.oracle_caches(case, 0)
    keep = attend > 0
    ref = GC.oracle_out(case, 0, kc, vc)
    err = np.abs(got[keep].astype(np.float64) - ref[keep]).max()
    assert err <= TOL[kv], f"max abs err {err}"
