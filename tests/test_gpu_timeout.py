"""The bounded device waits, made to run out without faulting anything.

Every mbarrier wait in the TMA decode kernels gives up after 2 s: the warp
flags PKV_DEV_TIMEOUT in the caller's status word, waits (again bounded) for
its other copies in flight, leaves its share out and returns, so the context
stays usable.  pkv_test_decode_stall arms one barrier phase of the transposed
kernel for 16 bytes more than its copies bring; the copies land, that phase
never completes and the wait runs out.  A normal call right after must match
the oracle again.
"""
import time

import numpy as np
import pytest

import workloads as W
from tests import gpu_cases as GC

pytestmark = pytest.mark.gpu


def test_decode_wait_runs_out_flags_timeout_and_the_next_call_is_clean(lib):
    import torch
    assert torch.cuda.is_available()
    w = W.DecodeWorkload("stall", 3, 8, 2, 128, 16, "bf16", "bf16", seed=71, ctx_law="fixed")
    case, _ = GC.make_small(w, lens=[700, 40, 300])
    eng, outs, st = GC.run_gpu(case, partition=64)
    assert st == 0
    kc, vc = GC.oracle_caches(case, 0)
    ref = GC.oracle_out(case, 0, kc, vc)
    assert np.abs(outs[0].astype(np.float64) - ref).max() <= 2e-3
    q = GC.to_torch(case.q[0], "bf16")
    tables = torch.from_numpy(case.tables).cuda()
    ctx = torch.from_numpy(case.lens.astype(np.int32)).cuda()
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    torch.cuda.synchronize()
    lib.stall_decode_for_test(16)
    try:
        t0 = time.monotonic()
        eng.attend(0, q, tables, ctx, int(case.lens.max()), partition=64, device_status=status)
        torch.cuda.synchronize()
        waited = time.monotonic() - t0
    finally:
        lib.stall_decode_for_test(0)
    assert int(status.item()) & lib.DEV_TIMEOUT, int(status.item())
    assert 1.5 <= waited < 30.0, waited    # the 2 s bound ran out, once
    # the context is still usable and the next call is exact again
    status.zero_()
    out = eng.attend(0, q, tables, ctx, int(case.lens.max()), partition=64,
                     device_status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    got = out.cpu().numpy()
    assert got.tobytes() == outs[0].tobytes()
    assert np.abs(got.astype(np.float64) - ref).max() <= 2e-3
