"""Full-size parity: every workload at its full size, in the launch configuration
bench.py times (automatic split-KV partition, the bench's workspace), checked
against the oracle on sampled sequences of sampled layers.

For a sampled sequence the oracle rebuilds that sequence's cache from the same
source rows with its own append (into a compact cache whose block j holds
logical block j; the result does not depend on where blocks live, a property the
oracle pins pin) and runs its own gather + float64 attention.  The step's
appended rows are also compared byte for byte with the oracle's append.
"""
import numpy as np
import pytest

import workloads as W
from oracle import attention as OA

pytestmark = pytest.mark.gpu

TOL = {"f32": 2e-3, "bf16": 2e-3, "fp8_e4m3": 1e-2, "int8": 1e-2}


def _bits(t, dtype):
    import torch
    t = t.contiguous().cpu()
    if dtype == "bf16":
        return t.view(torch.int16).numpy().view(np.uint16)
    if dtype == "f32":
        return t.numpy()
    if dtype == "int8":
        return t.numpy().astype(np.int8)
    return t.numpy().astype(np.uint8)


def _sample_seqs(w, lens):
    order = np.argsort(lens)
    pick = {int(order[0]), int(order[-1]), int(order[len(order) // 2])}
    if w.prefix_tokens:
        pick |= {0, w.prefix_seqs}      # a prefix sharer and a non-sharer
    pick.add(int(np.random.default_rng(w.seed).integers(0, w.num_seqs)))
    return sorted(pick)


@pytest.mark.parametrize("name", [w.name for w in W.ALL] + ["llama7b_layer_int8",
                                                             "llama7b_layer_fp8",
                                                             "gqa16_128q_8kv_bf16",
                                                             "d256_gqa2_bf16"])
def test_fullsize_sampled_parity(lib, name):
    import torch
    import bench
    w = bench.WORKLOADS[name]
    dev = torch.device("cuda", 0)
    layers = sorted({0, w.num_layers - 1})
    st = bench.DeviceStep(w, dev, keep_layers=layers)
    eng = st.eng
    seqs = _sample_seqs(w, st.lens)
    sd = "f32" if w.kv_dtype == "f32" else "bf16"
    bs = w.block_size
    checked = 0
    for layer in layers:
        # the bench's step for this layer: append the new token and attend, as
        # the bench times it (one paged_attention_decode_append call)
        out = eng.append_attend(layer, st.q[layer][0], st.kn[layer][0], st.vn[layer][0],
                                st.slots, st.tables, st.ctx, st.max_ctx, workspace=st.ws,
                                device_status=st.status)
        torch.cuda.synchronize()
        assert int(st.status.item()) == 0
        got = out.cpu().numpy()
        assert np.isfinite(got).all()
        ks_dev, vs_dev = st.src[layer]
        kscale = vscale = None
        if w.kv_dtype in ("fp8_e4m3", "int8"):
            kscale = eng.k_scale[layer].cpu().numpy()
            vscale = eng.v_scale[layer].cpu().numpy()
        qh = _bits(st.q[layer][0], w.q_dtype)
        kn, vn = _bits(st.kn[layer][0], sd), _bits(st.vn[layer][0], sd)
        for s in seqs:
            L = int(st.lens[s])
            rows = []
            if w.prefix_tokens and s < w.prefix_seqs:
                rows.append(np.arange(*st.owner_rows))
            rows.append(np.arange(*st.seq_rows[s]))
            idx = torch.from_numpy(np.concatenate(rows)).to(dev)
            ksrc = np.concatenate([_bits(ks_dev[idx], sd), kn[s:s + 1]])
            vsrc = np.concatenate([_bits(vs_dev[idx], sd), vn[s:s + 1]])
            assert ksrc.shape[0] == L
            nb = -(-L // bs)
            dt = {"f32": np.float32, "bf16": np.uint16, "fp8_e4m3": np.uint8,
                  "int8": np.int8}[w.kv_dtype]
            kc = np.zeros((nb, bs, w.num_kv_heads, w.head_dim), dtype=dt)
            vc = np.zeros_like(kc)
            OA.reshape_and_cache(ksrc, vsrc, np.arange(L), kc, vc, sd, w.kv_dtype, kscale, vscale)
            # the step's appended row, byte for byte
            slot = int(st.step_slots_h[s])
            g_k = _bits(eng.k_cache(layer)[slot // bs, slot % bs], w.kv_dtype)
            g_v = _bits(eng.v_cache(layer)[slot // bs, slot % bs], w.kv_dtype)
            assert g_k.tobytes() == kc[(L - 1) // bs, (L - 1) % bs].tobytes()
            assert g_v.tobytes() == vc[(L - 1) // bs, (L - 1) % bs].tobytes()
            ref = OA.paged_attention_decode(qh[s:s + 1], kc, vc, np.arange(nb)[None], [L], w.scale,
                                            w.q_dtype, w.kv_dtype, kscale, vscale)[0]
            err = np.abs(got[s].astype(np.float64) - ref).max()
            print(f"fullsize {name} layer {layer} seq {s} ctx {L} max_abs_err {err:.3e}")
            checked += 1
            assert err <= TOL[w.kv_dtype], f"{name} layer {layer} seq {s} ctx {L}: {err}"
    assert checked == len(layers) * len(seqs) >= min(3, w.num_seqs)
    del st
    torch.cuda.empty_cache()
