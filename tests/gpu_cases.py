"""Builders for GPU parity cases: the same seeded decode step run through the
C-ABI library (C++ pool + CUDA kernels) and through the oracle."""
from __future__ import annotations

import dataclasses

import numpy as np

import workloads as W
from oracle import attention as OA
from oracle import fp8 as OF8
from oracle import pool as OP

CODE = {"f32": 0, "bf16": 1, "fp8_e4m3": 2, "int8": 3}
POISON = {"f32": (np.float32, np.float32(np.nan)), "bf16": (np.uint16, 0x7FC0),
          "fp8_e4m3": (np.uint8, 0x7F), "int8": (np.int8, 127)}


class OraclePool:
    """The oracle pool behind the call names of the C pool wrapper."""

    def __init__(self, *a, **k):
        self.p = OP.Pool(*a, **k)

    def seq_create(self, s):
        self.p.seq_create(s)

    def seq_fork_prefix(self, d, s, n):
        self.p.seq_fork_prefix(d, s, n)

    def append_tokens(self, s, n):
        return np.asarray(self.p.seq_append_tokens(s, n), dtype=np.int64)

    def append_slots(self, sids):
        return np.asarray(self.p.seq_append_slots(list(sids)), dtype=np.int64)


def src_dtype(w):
    return "bf16" if w.kv_dtype in ("fp8_e4m3", "int8") else w.kv_dtype


def torch_dtype(code_name):
    import torch
    return {"f32": torch.float32, "bf16": torch.bfloat16, "fp8_e4m3": torch.uint8,
            "int8": torch.int8}[code_name]


def to_torch(a, name, device="cuda"):
    """numpy storage array -> torch tensor of the storage dtype on device."""
    import torch
    if name == "bf16":
        return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16).to(device)
    return torch.from_numpy(np.ascontiguousarray(a)).to(device)


def from_torch(t, name):
    import torch
    if name == "bf16":
        return t.cpu().view(torch.int16).numpy().view(np.uint16)
    return t.cpu().numpy()


@dataclasses.dataclass
class SmallCase:
    """Every input of one decode step, small enough for the oracle end to end."""
    w: W.DecodeWorkload
    lens: np.ndarray
    nb: int
    order: np.ndarray
    prompt_slots: list          # per layer-independent slot arrays (owner first if any)
    prompt_k: list              # per layer: [U, Hkv, D] storage arrays
    prompt_v: list
    step_slots: np.ndarray
    k_new: list                 # per layer [S, Hkv, D]
    v_new: list
    q: list                     # per layer [S, Hq, D]
    k_scale: list               # per layer [Hkv] float32 (fp8) or None
    v_scale: list
    tables: np.ndarray          # oracle pool's [S, MB] padded -1
    max_blocks: int


def make_small(w: W.DecodeWorkload, lens=None, nb=None, layers=None, shape_rows=None) -> tuple:
    """Build a small case; returns (case, c-pool) after checking both pools agree.
    ``shape_rows(k, v, k_new, v_new, q, starts)`` may change a layer's float32
    prompt K / V rows ([U, Hkv, D], sequence s's first prompt row at
    starts[s]), the step's new rows and q in place before they are stored."""
    import paged_kv_cache_295_gb300 as pkv
    from paged_kv_cache_295_gb300.engine import build_prompts
    lens = W.context_lens(w) if lens is None else np.asarray(lens, dtype=np.int64)
    nb = W.num_blocks(w, lens) if nb is None else nb
    order = W.free_order(w, nb)
    L = w.num_layers if layers is None else layers
    esz = W.ELEM_BYTES[w.kv_dtype]
    cpool = pkv.Pool(L, w.num_kv_heads, w.head_dim, w.block_size, CODE[w.kv_dtype],
                     num_blocks=nb, initial_free_order=order)
    opool = OraclePool(L, w.num_kv_heads, w.head_dim, w.block_size, esz, nb,
                       initial_free_order=order.tolist())
    c_owner, c_slots, c_oslots = build_prompts(cpool, lens, w.prefix_tokens, w.prefix_seqs)
    o_owner, o_slots, o_oslots = build_prompts(opool, lens, w.prefix_tokens, w.prefix_seqs)
    assert c_owner == o_owner
    for a, b in zip(c_slots, o_slots):
        assert np.array_equal(a, b)
    if c_oslots is not None:
        assert np.array_equal(c_oslots, o_oslots)
    step_c = cpool.append_slots(range(len(lens)))
    step_o = opool.append_slots(range(len(lens)))
    assert np.array_equal(step_c, step_o)
    mb = max(len(opool.p.tables[s]) for s in range(len(lens)))
    t_o, l_o = opool.p.padded_tables(list(range(len(lens))), mb)
    t_c, l_c = cpool.batch_tables(list(range(len(lens))), mb)
    assert np.array_equal(np.asarray(t_o), t_c) and np.array_equal(np.asarray(l_o), l_c)
    assert np.array_equal(l_c, lens)

    prompt_slots = ([o_oslots] if o_oslots is not None else []) + list(o_slots)
    prompt_slots = np.concatenate(prompt_slots) if prompt_slots else np.zeros(0, np.int64)
    U = prompt_slots.size
    S, hkv, hq, d = len(lens), w.num_kv_heads, w.num_q_heads, w.head_dim
    sd = src_dtype(w)
    kh = W.k_head_scales(w)[None, :, None]
    own = [len(x) for x in o_slots]
    starts = np.cumsum([0] + own[:-1]) + (len(o_oslots) if o_oslots is not None else 0)
    pk, pv, kn, vn, qq, ks_l, vs_l = [], [], [], [], [], [], []
    for layer in range(L):
        base = 100 * (layer + 1)
        k32 = W.normal_f32(w.seed, base + 0, (U, hkv, d)) * kh
        v32 = W.normal_f32(w.seed, base + 1, (U, hkv, d))
        kn32 = W.normal_f32(w.seed, base + 2, (S, hkv, d)) * kh
        vn32 = W.normal_f32(w.seed, base + 3, (S, hkv, d))
        q32 = W.normal_f32(w.seed, base + 4, (S, hq, d))
        if shape_rows is not None:
            shape_rows(k32, v32, kn32, vn32, q32, starts)
        pk.append(W.store(k32, sd))
        pv.append(W.store(v32, sd))
        kn.append(W.store(kn32, sd))
        vn.append(W.store(vn32, sd))
        qq.append(W.store(q32, w.q_dtype))
        if w.kv_dtype in ("fp8_e4m3", "int8"):
            ka = np.abs(np.concatenate([OA.to_f64(pk[-1], sd), OA.to_f64(kn[-1], sd)])).max((0, 2))
            va = np.abs(np.concatenate([OA.to_f64(pv[-1], sd), OA.to_f64(vn[-1], sd)])).max((0, 2))
            rule = W.fp8_scale_from_absmax if w.kv_dtype == "fp8_e4m3" else W.int8_scale_from_absmax
            ks_l.append(rule(ka))
            vs_l.append(rule(va))
        else:
            ks_l.append(None)
            vs_l.append(None)
    case = SmallCase(w, lens, nb, order, prompt_slots, pk, pv, step_c, kn, vn, qq, ks_l, vs_l,
                     np.asarray(t_o, dtype=np.int32), mb)
    return case, cpool


def oracle_caches(case: SmallCase, layer: int):
    """Oracle cache state after the prompts and the step's append (numpy)."""
    w = case.w
    dt, pz = POISON[w.kv_dtype]
    shape = (case.nb, w.block_size, w.num_kv_heads, w.head_dim)
    kc = np.full(shape, pz, dtype=dt)
    vc = np.full(shape, pz, dtype=dt)
    sd = src_dtype(w)
    OA.reshape_and_cache(case.prompt_k[layer], case.prompt_v[layer], case.prompt_slots, kc, vc,
                         sd, w.kv_dtype, case.k_scale[layer], case.v_scale[layer])
    OA.reshape_and_cache(case.k_new[layer], case.v_new[layer], case.step_slots, kc, vc, sd,
                         w.kv_dtype, case.k_scale[layer], case.v_scale[layer])
    return kc, vc


def oracle_out(case: SmallCase, layer: int, kc, vc, seqs=None):
    w = case.w
    return OA.paged_attention_decode(case.q[layer], kc, vc, case.tables, case.lens, w.scale,
                                     w.q_dtype, w.kv_dtype, case.k_scale[layer],
                                     case.v_scale[layer], seqs=seqs)


def run_gpu(case: SmallCase, partition=0, layers=None, tables=None):
    """Product path for every layer: append prompts, append the step, attend.

    Returns (engine, list of per-layer outputs as numpy float32, status word).
    """
    import torch
    from paged_kv_cache_295_gb300.engine import PagedKVCache
    w = case.w
    L = len(case.prompt_k) if layers is None else layers
    eng = PagedKVCache(L, w.num_kv_heads, w.head_dim, w.block_size, case.nb, CODE[w.kv_dtype],
                       initial_free_order=case.order)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    sd = src_dtype(w)
    slots_p = torch.from_numpy(case.prompt_slots).cuda()
    slots_s = torch.from_numpy(case.step_slots).cuda()
    bt = torch.from_numpy(case.tables if tables is None else tables).cuda()
    cl = torch.from_numpy(case.lens.astype(np.int32)).cuda()
    outs = []
    for layer in range(L):
        if eng.k_scale is not None:
            eng.k_scale[layer] = torch.from_numpy(case.k_scale[layer]).cuda()
            eng.v_scale[layer] = torch.from_numpy(case.v_scale[layer]).cuda()
        if case.prompt_slots.size:
            eng.append(layer, to_torch(case.prompt_k[layer], sd), to_torch(case.prompt_v[layer], sd),
                       slots_p, device_status=status)
        eng.append(layer, to_torch(case.k_new[layer], sd), to_torch(case.v_new[layer], sd),
                   slots_s, device_status=status)
        out = eng.attend(layer, to_torch(case.q[layer], w.q_dtype), bt, cl, int(case.lens.max()),
                         partition=partition, device_status=status)
        outs.append(out.cpu().numpy())
    torch.cuda.synchronize()
    return eng, outs, int(status.item())


def make_prefill(w, chunk, prefix, seed=0, bad_block=None, kv="bf16", q_mul=None,
                 shape_rows=None):
    """A seeded chunked-prefill step: the oracle pool and the C pool hand out the
    same slots; the cached prefix rows are placed by the oracle's append; the
    chunk's rows are left for the GPU append.  ``kv`` is the cache type (bf16,
    or fp8_e4m3 / int8 with per-head absmax / 448 or / 127 scales); ``q_mul`` cycles per-token
    multipliers over q before its bf16 rounding; ``shape_rows(k, v, q, starts)``
    may change the float32 K / V rows ([sum(ctx), Hkv, D], sequence s from row
    starts[s]) and q ([sum(chunk), Hq, D]) in place before they are stored.
    Returns (device tensors, the
    oracle's host arrays after the chunk's append, max chunk, max context)."""
    import torch
    import paged_kv_cache_295_gb300 as pkv
    n = np.asarray(chunk, dtype=np.int64)
    ctx = n + np.asarray(prefix, dtype=np.int64)
    S, hq, hkv, d, bs = len(n), w.num_q_heads, w.num_kv_heads, w.head_dim, w.block_size
    nb = W.prefill_num_blocks(w, ctx) + 2
    order = W.rng(w.seed + seed, 2).permutation(nb).astype(np.int32)
    op = OP.Pool(1, hkv, d, bs, W.ELEM_BYTES[kv], nb, initial_free_order=order.tolist())
    cp = pkv.Pool(1, hkv, d, bs, CODE[kv], num_blocks=nb, initial_free_order=order)
    pre_slots, chunk_slots = [], []
    for s in range(S):
        op.seq_create(s)
        cp.seq_create(s)
        a = np.asarray(op.seq_append_tokens(s, int(ctx[s] - n[s])), dtype=np.int64)
        b = np.asarray(op.seq_append_tokens(s, int(n[s])), dtype=np.int64)
        assert np.array_equal(cp.append_tokens(s, int(ctx[s] - n[s])), a)
        assert np.array_equal(cp.append_tokens(s, int(n[s])), b)
        pre_slots.append(a)
        chunk_slots.append(b)
    mb = max(len(op.tables[s]) for s in range(S)) + 1
    t_o, _ = op.padded_tables(list(range(S)), mb, pad=-1)
    t_c, _ = cp.batch_tables(list(range(S)), mb)
    tables = np.asarray(t_o, dtype=np.int32)
    assert np.array_equal(tables, t_c)
    if bad_block is not None:                  # (seq, logical block) -> out-of-range id
        tables[bad_block] = nb + 5
    r = W.rng(w.seed + seed, 3)
    U = int(ctx.sum())
    kf = r.standard_normal((U, hkv, d), dtype=np.float32)
    vf = r.standard_normal((U, hkv, d), dtype=np.float32)
    T = int(n.sum())
    qf = r.standard_normal((T, hq, d), dtype=np.float32)
    if q_mul is not None:
        qf *= np.resize(np.asarray(q_mul, dtype=np.float32), T)[:, None, None]
    off = np.concatenate([[0], np.cumsum(ctx)])
    if shape_rows is not None:
        shape_rows(kf, vf, qf, off[:-1])
    k_rows, v_rows, q = W.store(kf, "bf16"), W.store(vf, "bf16"), W.store(qf, "bf16")
    pre_idx = np.concatenate([np.arange(off[s], off[s] + ctx[s] - n[s]) for s in range(S)])
    chk_idx = np.concatenate([np.arange(off[s] + ctx[s] - n[s], off[s + 1]) for s in range(S)])
    ps = np.concatenate(pre_slots) if pre_slots else np.zeros(0, np.int64)
    cs = np.concatenate(chunk_slots)
    ks = vs = None
    if kv in ("fp8_e4m3", "int8"):
        rule = W.fp8_scale_from_absmax if kv == "fp8_e4m3" else W.int8_scale_from_absmax
        ks = rule(np.abs(OA.to_f64(k_rows, "bf16")).max((0, 2)))
        vs = rule(np.abs(OA.to_f64(v_rows, "bf16")).max((0, 2)))
    dt, pz = POISON[kv]
    kc = np.full((nb, bs, hkv, d), pz, dtype=dt)
    vc = kc.copy()
    OA.reshape_and_cache(k_rows[pre_idx], v_rows[pre_idx], ps, kc, vc, "bf16", kv, ks, vs)
    dev = {
        "kc": to_torch(kc, kv), "vc": to_torch(vc, kv),
        "ks": None if ks is None else torch.from_numpy(ks).cuda(),
        "vs": None if vs is None else torch.from_numpy(vs).cuda(),
        "kn": to_torch(k_rows[chk_idx], "bf16"), "vn": to_torch(v_rows[chk_idx], "bf16"),
        "slots": torch.from_numpy(cs).cuda(), "q": to_torch(q, "bf16"),
        "tables": torch.from_numpy(tables).cuda(),
        "ctx": torch.from_numpy(ctx.astype(np.int32)).cuda(),
        "qs": torch.from_numpy(np.concatenate([[0], np.cumsum(n)]).astype(np.int32)).cuda(),
    }
    OA.reshape_and_cache(k_rows[chk_idx], v_rows[chk_idx], cs, kc, vc, "bf16", kv, ks, vs)
    host = {"kc": kc, "vc": vc, "q": q, "tables": tables, "ctx": ctx,
            "qs": np.concatenate([[0], np.cumsum(n)]), "kv": kv, "ks": ks, "vs": vs}
    return dev, host, int(n.max()), int(ctx.max())


def run_prefill_gpu(w, dev, max_q, max_ctx, causal=True, status=None):
    """GPU append of the chunk rows, then paged_attention_prefill (float32 out)."""
    import torch
    import paged_kv_cache_295_gb300 as pkv
    pkv.reshape_and_cache(dev["kn"], dev["vn"], dev["slots"], dev["kc"], dev["vc"],
                          k_scale=dev.get("ks"), v_scale=dev.get("vs"), device_status=status)
    out = torch.full((dev["q"].shape[0], w.num_q_heads, w.head_dim), float("nan"),
                     dtype=torch.float32, device="cuda")
    pkv.paged_attention_prefill(dev["q"], dev["qs"], dev["kc"], dev["vc"], dev["tables"],
                                dev["ctx"], w.scale, max_q, max_ctx, causal=causal, out=out,
                                k_scale=dev.get("ks"), v_scale=dev.get("vs"),
                                device_status=status)
    torch.cuda.synchronize()
    return out.cpu().numpy()
