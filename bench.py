#!/usr/bin/env python3
"""Benchmark of the paged decode-attention hot path on one GB300 (or N replicas).

One step = one decode step of the workload: append the new token's K/V of every
sequence into the paged cache (reshape_and_cache) and attend with one query
token per sequence over its whole paged context (paged_attention_decode, with
its split-KV reduce when launched), for every layer of the workload.

Default workload: one LLaMA-7B-shaped layer (32 sequences, 32 query = 32 KV
heads, head_dim 128, bf16 KV, block_size 16, contexts uniform in [512, 4096],
shuffled physical blocks).  Metric: effective KV GB/s (K and V bytes the step
attends over / step time), plus decode tokens/s and attention us per layer.

Arms:
  (default)          the CUDA library through its C ABI, inputs resident in HBM;
  --impl reference   the plain CPU oracle on this host's cores, on a bounded
                     sample of the same workload.
With torchrun (N>1) every rank runs its own replica ("replicas only": the
decode step needs no exchange between GPUs) and the time is the max over ranks.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import time

if "--impl" in sys.argv and "reference" in sys.argv:
    for _v in ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS"):
        os.environ[_v] = "1"

import numpy as np  # noqa: E402

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import workloads as W  # noqa: E402

FALLBACK_HBM_GBS = 6800.0
METRIC = "paged decode attention: effective KV GB/s (% HBM peak), decode tokens/s"
PREFILL_METRIC = "paged prefill attention: TFLOP/s (% bf16 tensor peak), prefill tokens/s"
FORK_METRIC = "copy-on-write block copies of a beam fork: GB/s (distinct sources read + copies written; % HBM peak)"
SWAP_METRIC = "swap of whole sequences to host memory and back: GB/s over the host link"
WORKLOADS = {w.name: w for w in W.ALL + W.EXTRA + W.PREFILL + W.FORK + W.SWAP}
DEFAULT_WORKLOAD = W.LLAMA7B_LAYER.name

# DRAM bytes (read + write) per launch of the decode kernel from an ncu capture,
# valid only while the kernel sources hash to `sources_sha`.
NCU_TRAFFIC = {"sources_sha": "34bc4b5b2c71edc2", "workload": "llama7b_layer_bf16",
               # paged_decode_mma2_kernel (append fused in) 1.239778 GB read + 4.985 MB
               # written, plus the reduce kernel's 1.440 MB read
               "bytes_per_launch": 1239777792 + 4985344 + 1440000}


def parse_args(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.splitlines()[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=1000)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", choices=sorted(WORKLOADS), default=DEFAULT_WORKLOAD)
    ap.add_argument("--num-layers", type=int, default=0,
                    help="override the workload's layer count (small profiling captures)")
    ap.add_argument("--partition", type=int, default=0, help="split-KV tokens (0 = auto)")
    ap.add_argument("--e2e-steps", type=int, default=0, help="e2e steps (0 = min(steps, 200))")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-configs", action="store_true",
                    help="time the selected workload only (profiling runs)")
    ap.add_argument("--sustain-seconds", type=float, default=1.0,
                    help="after the timed steps, repeat the step this long for the clock record")
    ap.add_argument("--clock-period-ms", type=int, default=20)
    ap.add_argument("--cpu-cores", type=int, default=0,
                    help="reference arm: oracle worker processes (0 = every core this "
                         "process may run on)")
    ap.add_argument("--no-bandwidth-ref", action="store_true",
                    help="skip the in-run copy/read reference kernels (profiling runs)")
    ap.add_argument("--bandwidth-gb", type=float, default=4.0,
                    help="bytes the in-run copy and read kernels move (GB; smaller for captures)")
    ap.add_argument("--cpu-baseline-worker", action="store_true", help=argparse.SUPPRESS)
    ap.add_argument("--cpu-seconds", type=float, default=12.0, help=argparse.SUPPRESS)
    return ap.parse_args(argv)


def workload_of(args):
    """The selected workload, with --num-layers applied when given."""
    import dataclasses
    w = WORKLOADS[args.workload]
    if getattr(args, "num_layers", 0) and hasattr(w, "num_layers"):
        w = dataclasses.replace(w, num_layers=args.num_layers)
    return w


# The sources the decode kernels (and their launch) are built from.
DECODE_SOURCES = ("common.cuh", "decode_api.cu", "decode_kernel.cuh", "decode_launch.cuh",
                  "decode_mma.cuh", "decode_mma2.cuh", "decode_mma_fp8.cuh",
                  "decode_mma_launch.cu", "tmap.cuh")


def kernel_sources_sha() -> str:
    """Hash of the decode kernels' sources, to tie an ncu traffic figure to one
    kernel version (changes elsewhere in the library do not invalidate it)."""
    csrc = os.path.join(ROOT, "paged_kv_cache_295_gb300", "csrc")
    h = hashlib.sha256()
    for f in DECODE_SOURCES:
        h.update(f.encode())
        h.update(open(os.path.join(csrc, f), "rb").read())
    return h.hexdigest()[:16]


def measured_peaks(key="hbm_gbs", fallback=None):
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        try:
            d = json.load(open(p))
            return float(d[key]), "measured"
        except Exception:
            pass
    return (FALLBACK_HBM_GBS if fallback is None else fallback), "fallback"


# ---------------------------------------------------------------- clocks ---
CLOCK_FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
                "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
                "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")


class ClockSampler:
    """nvidia-smi sampling of SM clocks and throttle reasons during a region."""

    def __init__(self, gpu_index: int, period_ms: int = 50):
        import tempfile
        self.path = os.path.join(tempfile.gettempdir(), f"pagedkv_clocks_gpu{gpu_index}.csv")
        self.proc = None
        try:
            self.fh = open(self.path, "w")
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={gpu_index}", f"--query-gpu={CLOCK_FIELDS}",
                 "--format=csv,noheader,nounits", f"-lms={period_ms}"],
                stdout=self.fh, stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        self.fh.close()
        rows = []
        for ln in open(self.path):
            parts = [x.strip() for x in ln.split(",")]
            if len(parts) < 9:
                continue
            try:
                rows.append((float(parts[1]), float(parts[2]), float(parts[3]), parts[5:9]))
            except ValueError:
                continue
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"], "samples": 0}
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i, v in enumerate(r[3])
                          if v.lower() == "active"})
        return {"sm_mhz": statistics.median(r[0] for r in rows),
                "sm_max_mhz": max(r[1] for r in rows),
                "power_w_max": max(r[2] for r in rows),
                "reasons": reasons, "samples": len(rows)}


# ----------------------------------------------------------- distributed ---
def dist_env():
    return (int(os.environ.get("RANK", "0")), int(os.environ.get("WORLD_SIZE", "1")),
            int(os.environ.get("LOCAL_RANK", "0")))


def max_over_ranks(x: float, world: int, device=None) -> float:
    """Max of a per-rank scalar (the slowest rank sets the job time)."""
    if world <= 1:
        return x
    import torch
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def sum_over_ranks(x: float, world: int, device=None) -> float:
    if world <= 1:
        return x
    import torch
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.SUM)
    return float(t.item())


def barrier(world: int):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


# ------------------------------------------------------- byte accounting ---
def row_bytes(w) -> int:
    """K (or V) bytes of one token of one layer: num_kv_heads * head_dim * elem."""
    return w.num_kv_heads * w.head_dim * W.ELEM_BYTES[w.kv_dtype]


def kv_bytes_logical(w, lens) -> int:
    """K+V bytes every sequence attends over (a shared prefix counted per reader)."""
    return int(np.sum(lens)) * 2 * row_bytes(w)


def kv_bytes_unique(w, lens) -> int:
    """K+V bytes of distinct cache rows read (a shared prefix counted once)."""
    shared = max(0, w.prefix_seqs - 1) * w.prefix_tokens if w.prefix_tokens else 0
    return (int(np.sum(lens)) - shared) * 2 * row_bytes(w)


def attention_alg_bytes(w, lens) -> int:
    """Algorithmic bytes of one attention launch (one layer): unique K/V rows,
    q, the float32 output, the block-table entries read and the lengths."""
    S, hq, d = w.num_seqs, w.num_q_heads, w.head_dim
    qb = 4 if w.q_dtype == "f32" else 2
    tables = int(np.sum(-(-np.asarray(lens) // w.block_size))) * 4
    return kv_bytes_unique(w, lens) + S * hq * d * (qb + 4) + tables + S * 4


def append_alg_bytes(w) -> int:
    """Bytes of one append launch: the new rows read (source type) and written."""
    src = 2 if w.kv_dtype in ("bf16", "fp8_e4m3", "int8") else 4
    return w.num_seqs * 2 * w.num_kv_heads * w.head_dim * (src + W.ELEM_BYTES[w.kv_dtype]) + \
        w.num_seqs * 8


# layers of the model each single-layer workload is shaped after
MODEL_LAYERS = {"llama7b_layer_bf16": ("LLaMA-7B", 32), "llama7b_layer_int8": ("LLaMA-7B", 32),
                "llama7b_layer_fp8": ("LLaMA-7B", 32),
                "llama70b_gqa8_bf16": ("LLaMA-70B", 80)}


def model_tokens_per_s(w, step_s_per_layer):
    """Decode tokens/s of the whole model the layer is shaped after: the batch
    over (per-layer step time x the model's layers); attention and append only,
    extrapolated from one layer (None for workloads that are not one layer)."""
    if w.name not in MODEL_LAYERS:
        return None
    model, layers = MODEL_LAYERS[w.name]
    return {"value": round(w.num_seqs / (step_s_per_layer * layers), 1), "model": model,
            "layers": layers, "note": "extrapolated: one layer's append + attention x layers"}


def decode_kernel_name(w) -> str:
    """The decode kernel the library picks for this workload's shape."""
    if w.group > 16 or w.block_size < 8:
        return "paged_decode_kernel"
    if (w.group <= 8 or w.group == 16) and ((w.kv_dtype == "bf16" and w.head_dim in (64, 128, 256))
                         or (w.kv_dtype in ("fp8_e4m3", "int8") and w.head_dim == 128)):
        return "paged_decode_mma2_kernel"
    if w.kv_dtype == "bf16" and w.head_dim in (64, 128):
        return "paged_decode_mma_kernel"
    if w.kv_dtype == "fp8_e4m3" and w.head_dim == 128:
        return "paged_decode_mma_fp8_kernel"
    return "paged_decode_kernel"


# --------------------------------------------------- device-side workload ---
class DeviceStep:
    """A decode step of workload ``w`` resident on one GPU, run through the C ABI."""

    def __init__(self, w, device, partition=0, nsets=2, keep_layers=()):
        import torch
        import paged_kv_cache_295_gb300 as pkv
        from paged_kv_cache_295_gb300.engine import PagedKVCache, build_prompts
        self.w, self.device, self.partition = w, device, partition
        S, hq, hkv, d, bs = w.num_seqs, w.num_q_heads, w.num_kv_heads, w.head_dim, w.block_size
        code = {"f32": pkv.F32, "bf16": pkv.BF16, "fp8_e4m3": pkv.FP8_E4M3,
                "int8": pkv.INT8}[w.kv_dtype]
        self.lens = W.context_lens(w)
        nb = W.num_blocks(w, self.lens)
        self.eng = eng = PagedKVCache(w.num_layers, hkv, d, bs, nb, code, device=device,
                                      initial_free_order=W.free_order(w, nb))
        _, slots, oslots = build_prompts(eng.pool, self.lens, w.prefix_tokens, w.prefix_seqs)
        prompt = np.concatenate(([oslots] if oslots is not None else []) + list(slots))
        # rows of the prompt tensor: the prefix owner's first, then each sequence's own
        self.owner_rows = (0, len(oslots)) if oslots is not None else None
        starts = np.cumsum([0] + [len(x) for x in slots]) + (len(oslots) if oslots is not None else 0)
        self.seq_rows = [(int(starts[i]), int(starts[i + 1])) for i in range(S)]
        self.src = {}
        step_slots = eng.pool.append_slots(range(S))
        mb = int(max(len(eng.pool.block_table(s)) for s in range(S)))
        tables, lens_pool = eng.pool.batch_tables(list(range(S)), mb)
        assert np.array_equal(lens_pool, self.lens)
        self.max_ctx = int(self.lens.max())
        self.tables_h, self.step_slots_h = tables, step_slots
        self.tables = torch.from_numpy(tables).to(device)
        self.ctx = torch.from_numpy(self.lens.astype(np.int32)).to(device)
        self.slots = torch.from_numpy(step_slots).to(device)
        self.src_dt = torch.float32 if w.kv_dtype == "f32" else torch.bfloat16
        self.q_dt = torch.float32 if w.q_dtype == "f32" else torch.bfloat16
        kh = torch.from_numpy(W.k_head_scales(w)).to(device)[None, :, None]
        prompt_d = torch.from_numpy(prompt).to(device)
        gen = torch.Generator(device=device)
        self.q, self.kn, self.vn = [], [], []
        for layer in range(w.num_layers):
            gen.manual_seed(w.seed * 1000 + layer)
            ks, vs = self._randn_rows(gen, prompt.size, kh), self._randn_rows(gen, prompt.size, None)
            q = [torch.randn((S, hq, d), generator=gen, device=device).to(self.q_dt)
                 for _ in range(nsets)]
            kn = [(torch.randn((S, hkv, d), generator=gen, device=device) * kh).to(self.src_dt)
                  for _ in range(nsets)]
            vn = [torch.randn((S, hkv, d), generator=gen, device=device).to(self.src_dt)
                  for _ in range(nsets)]
            if code in (pkv.FP8_E4M3, pkv.INT8):
                # static per-head scale absmax / qmax over the layer's data (448 E4M3, 127 INT8)
                qmax = 448.0 if code == pkv.FP8_E4M3 else 127.0
                ka = torch.maximum(ks.float().abs().amax((0, 2)), torch.stack(kn).float().abs().amax((0, 1, 3)))
                va = torch.maximum(vs.float().abs().amax((0, 2)), torch.stack(vn).float().abs().amax((0, 1, 3)))
                eng.k_scale[layer] = torch.where(ka > 0, ka / qmax, torch.ones_like(ka))
                eng.v_scale[layer] = torch.where(va > 0, va / qmax, torch.ones_like(va))
            if prompt.size:
                eng.append(layer, ks, vs, prompt_d)
            if layer in keep_layers:   # kept for oracle checks of this layer
                self.src[layer] = (ks, vs)
            del ks, vs
            self.q.append(q)
            self.kn.append(kn)
            self.vn.append(vn)
        self.out = torch.empty((S, hq, d), dtype=torch.float32, device=device)
        self.ws = eng.workspace_for(S, hq, self.max_ctx, partition, device=device)
        self.P = pkv.partition_tokens(S, hq, hkv, self.max_ctx, partition)
        if partition == 0 and w.kv_dtype in ("fp8_e4m3", "int8"):   # 8-bit rows: twice
            self.P = min(4096, 2 * self.P)
        self.max_parts = max(1, -(-self.max_ctx // self.P))
        self.status = torch.zeros(1, dtype=torch.int32, device=device)
        torch.cuda.synchronize(device)

    def _randn_rows(self, gen, n, kh, chunk=1 << 18):
        import torch
        w = self.w
        out = torch.empty((n, w.num_kv_heads, w.head_dim), dtype=self.src_dt, device=self.device)
        for a in range(0, n, chunk):
            b = min(n, a + chunk)
            x = torch.randn((b - a, w.num_kv_heads, w.head_dim), generator=gen, device=self.device)
            out[a:b] = (x * kh if kh is not None else x).to(self.src_dt)
        return out

    def fused(self) -> bool:
        """The append runs inside the decode kernel (the transposed kernel, 16-bit
        caches); 8-bit caches run the append kernel first."""
        return decode_kernel_name(self.w) == "paged_decode_mma2_kernel" and self.w.kv_dtype == "bf16"

    def launches_per_step(self) -> int:
        """Our kernels per step: per layer one decode (with the append fused in,
        else an append kernel too) and one reduce if split."""
        return self.w.num_layers * ((1 if self.fused() else 2) + (1 if self.max_parts > 1 else 0))

    def run(self, i, ev=None):
        """One decode step (every layer) through paged_attention_decode_append;
        ``ev`` = (start, end) event lists per layer around that call."""
        eng, k = self.eng, i % len(self.q[0])
        self.runs = i + 1
        for layer in range(self.w.num_layers):
            if ev is not None:
                ev[0][layer].record()
            eng.append_attend(layer, self.q[layer][k], self.kn[layer][k], self.vn[layer][k],
                              self.slots, self.tables, self.ctx, self.max_ctx, out=self.out,
                              workspace=self.ws, partition=self.partition,
                              device_status=self.status)
            if ev is not None:
                ev[1][layer].record()


    def sample(self, s):
        """Host copies of what sequence ``s`` attended over in the last layer of
        the last step, for a check against the oracle: its q row, its blocks
        (in table order, so the table becomes 0 .. nb-1), the layer's scales and
        the output row the kernel wrote."""
        import torch
        w, layer = self.w, self.w.num_layers - 1
        L = int(self.lens[s])
        nb = -(-L // w.block_size)
        idx = torch.from_numpy(self.tables_h[s, :nb].astype(np.int64)).to(self.device)

        def host(t):
            t = t.contiguous().cpu()
            if t.dtype == torch.bfloat16:
                return t.view(torch.int16).numpy().view(np.uint16)
            return t.numpy()
        k_last = (self.runs - 1) % len(self.q[layer])
        ks = None if self.eng.k_scale is None else host(self.eng.k_scale[layer])
        vs = None if self.eng.v_scale is None else host(self.eng.v_scale[layer])
        return {"seq": int(s), "context": L, "layer": layer,
                "q": host(self.q[layer][k_last][s:s + 1]),
                "k": host(self.eng.k_cache(layer).index_select(0, idx)),
                "v": host(self.eng.v_cache(layer).index_select(0, idx)),
                "k_scale": ks, "v_scale": vs, "out": host(self.out[s:s + 1]),
                "scale": self.eng.scale, "q_dtype": w.q_dtype, "kv_dtype": w.kv_dtype}


# ------------------------------------------------- in-run HBM references ---
def in_run_bandwidth(device, nbytes=4 << 30, reps=10):
    """GB/s of the library's copy kernel (2N bytes) and read kernel (N bytes)."""
    import torch
    import paged_kv_cache_295_gb300 as pkv
    a = torch.empty(nbytes // 2, dtype=torch.uint8, device=device)
    b = torch.empty_like(a)
    a.fill_(1)
    r = torch.empty(nbytes, dtype=torch.uint8, device=device)
    r.fill_(2)
    sink = torch.empty(pkv.read_kernel_sink_floats(), dtype=torch.float32, device=device)
    res = {}
    for name, fn, moved in (("copy_gbs", lambda: pkv.copy_kernel(a, b), 2 * a.numel()),
                            ("read_gbs", lambda: pkv.read_kernel(r, sink), r.numel())):
        for _ in range(3):
            fn()
        ts = []
        for _ in range(reps):
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record()
            fn()
            e1.record()
            e1.synchronize()
            ts.append(e0.elapsed_time(e1) * 1e-3)
        res[name] = moved / min(ts) / 1e9
    del a, b, r
    torch.cuda.empty_cache()
    return res


# --------------------------------------------------------------- our arm ---
# The workloads every default run also times, each in this process after the
# headline one: the tiny fp32 case (parity only), the 70B-shaped GQA-8 layer,
# the 128K-context split-KV layer and the ragged 32-layer FP8 step.
CONFIG_SET = ("tiny_fp32_mha", "llama70b_gqa8_bf16", "long_ctx_splitkv_bf16",
              "ragged_32layer_fp8")
# max-abs tolerance against the oracle by cache type (f32 / bf16: 2e-3; 8-bit: 1e-2)
ORACLE_TOL = {"f32": 2e-3, "bf16": 2e-3, "fp8_e4m3": 1e-2, "int8": 1e-2}


def time_steps(st, n, first=0):
    """Runs ``n`` steps of ``st`` with CUDA events around the whole region and
    around every layer's call; returns (region seconds, per-call seconds)."""
    import torch
    L = st.w.num_layers
    ev = [[[torch.cuda.Event(enable_timing=True) for _ in range(L)] for _ in range(2)]
          for _ in range(n)]
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    t0.record()
    for i in range(n):
        st.run(first + i, ev[i])
    t1.record()
    torch.cuda.synchronize(st.device)
    calls = [ev[i][0][l].elapsed_time(ev[i][1][l]) * 1e-3 for i in range(n) for l in range(L)]
    return t0.elapsed_time(t1) * 1e-3, calls


def prime_queue(device):
    """A short device-side delay before a timed region, so the host enqueues
    the first timed launches while the GPU is still busy (the first interval
    then holds no launch latency).  It runs before the region's start event."""
    import torch
    torch.cuda._sleep(2_000_000)


def call_stats(w, lens, calls, peak):
    """Mean / median / p10 / p90 of one launch's time and the roofline
    fractions they give (algorithmic bytes: unique K/V rows read, q, out,
    tables, lengths, plus the appended rows)."""
    alg = attention_alg_bytes(w, lens) + append_alg_bytes(w)
    mean, med = statistics.fmean(calls), statistics.median(calls)
    p10, p90 = (float(np.percentile(calls, q)) for q in (10, 90))
    return {"us_per_layer_mean": round(mean * 1e6, 3), "us_per_layer_median": round(med * 1e6, 3),
            "us_per_layer_p10_p90": [round(p10 * 1e6, 3), round(p90 * 1e6, 3)],
            "alg_bytes_per_launch": alg,
            "achieved_gbs_mean": round(alg / mean / 1e9, 2),
            "achieved_gbs_median": round(alg / med / 1e9, 2),
            "frac_mean": round(alg / mean / 1e9 / peak, 4),
            "frac_median": round(alg / med / 1e9 / peak, 4)}


def run_config(name, args, dev, peak):
    """One more workload timed like the headline one (same steps and warm-up),
    plus the host copy of one sequence for the oracle check; frees its pool."""
    import torch
    w = WORKLOADS[name]
    st = DeviceStep(w, dev, partition=args.partition)
    for i in range(args.warmup):
        st.run(i)
    torch.cuda.synchronize(dev)
    prime_queue(dev)
    dt, calls = time_steps(st, args.steps, args.warmup)
    rec = {"kind": "parity only" if name == "tiny_fp32_mha" else "timed",
           "num_layers": w.num_layers, "num_seqs": w.num_seqs,
           "num_q_heads": w.num_q_heads, "num_kv_heads": w.num_kv_heads,
           "block_size": w.block_size, "kv_dtype": w.kv_dtype,
           "kernel": decode_kernel_name(w) + (" + paged_decode_reduce_kernel"
                                              if st.max_parts > 1 else ""),
           "partition_tokens": st.P, "max_partitions": st.max_parts,
           "append": "fused into the decode kernel" if st.fused() else "append kernel, then decode",
           "ms_per_step": round(dt / args.steps * 1e3, 5),
           "kv_gb_per_step_unique": round(kv_bytes_unique(w, st.lens) * w.num_layers / 1e9, 4),
           "value_logical_gbs": round(kv_bytes_logical(w, st.lens) * w.num_layers * args.steps
                                      / dt / 1e9, 2),
           "decode_tokens_per_s": round(w.num_seqs * args.steps / dt, 1),
           "device_status": int(st.status.item())}
    rec.update(call_stats(w, st.lens, calls, peak))
    seqs = range(w.num_seqs) if w.num_seqs <= 2 else [int(np.argmax(st.lens))]
    samples = [st.sample(s) for s in seqs]
    del st
    torch.cuda.empty_cache()
    return rec, samples


def run_ours(args):
    import torch
    rank, world, local = dist_env()
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", init_method="env://")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    w = workload_of(args)
    K, Wm = args.steps, args.warmup
    if Wm < 3:
        raise SystemExit("--warmup must be >= 3")
    bw = None if args.no_bandwidth_ref else in_run_bandwidth(
        dev, nbytes=int(args.bandwidth_gb * (1 << 30)) // 64 * 64)
    st = DeviceStep(w, dev, partition=args.partition)
    lens, nb = st.lens, st.eng.num_blocks
    L = w.num_layers
    peak, peak_src = measured_peaks()
    # nvidia-smi starts before the warm-up, so its start-up stays out of the region
    clocks = ClockSampler(local, period_ms=args.clock_period_ms)
    time.sleep(0.3)
    for i in range(Wm):
        st.run(i)
    torch.cuda.synchronize(dev)
    barrier(world)
    torch.cuda.synchronize(dev)
    prime_queue(dev)
    dt_local, attn_s = time_steps(st, K, Wm)
    barrier(world)
    # The same step again for at least --sustain-seconds while the sampler
    # runs, so the clock record covers a region long enough to sample; its
    # times are reported beside the K-step figures and never replace them.
    sustain = None
    if args.sustain_seconds > 0:
        n_ext = max(K, int(math.ceil(args.sustain_seconds / max(dt_local / K, 1e-6))))
        prime_queue(dev)
        dt_ext, ext_s = time_steps(st, n_ext, Wm + K)
        sustain = {"steps": n_ext, "seconds": round(dt_ext, 3),
                   "ms_per_step": round(dt_ext / n_ext * 1e3, 5)}
        sustain.update(call_stats(w, st.lens, ext_s, peak))
    clk = clocks.stop()
    dt = max_over_ranks(dt_local, world, dev)
    status = int(st.status.item())
    samples = {w.name: [st.sample(int(np.argmax(lens)))]} if rank == 0 else {}

    kv_log = kv_bytes_logical(w, lens) * L
    kv_uni = kv_bytes_unique(w, lens) * L
    total_kv = sum_over_ranks(kv_log * K, world, dev)
    value = total_kv / dt / 1e9
    # the timed call appends too: its rows count (0.04 % of the 7B layer's bytes)
    head = call_stats(w, lens, attn_s, peak)
    attn_bytes = head["alg_bytes_per_launch"]
    attn_avg = statistics.fmean(attn_s)
    achieved = attn_bytes / attn_avg / 1e9
    if clk.get("sm_mhz"):
        head["us_median_x_sm_mhz"] = round(head["us_per_layer_median"] * clk["sm_mhz"], 1)
    sha = kernel_sources_sha()
    traffic = (NCU_TRAFFIC.get("bytes_per_launch")
               if NCU_TRAFFIC.get("sources_sha") == sha and NCU_TRAFFIC.get("workload") == w.name
               else None)

    graph = None
    if w.graph:   # the same step replayed as one CUDA graph (buckets 1..S, padding)
        graph, dt, value, dt_local = run_graph(st, K, Wm, world, dev, dt, kv_log)
    e2e = run_e2e(st, args, dev, world)
    configs = None
    if world == 1 and not args.no_configs and w.name == DEFAULT_WORKLOAD:
        nsm = torch.cuda.get_device_properties(dev).multi_processor_count
        del st
        torch.cuda.empty_cache()
        configs = {w.name: dict(head, kind="timed (the headline line)", ms_per_step=round(
            dt / K * 1e3, 5), device_status=status, kernel=decode_kernel_name(w) + (
                " + paged_decode_reduce_kernel" if paged_parts(w, args.partition) > 1 else ""),
            partition_tokens=paged_partition(w, args.partition))}
        for name in CONFIG_SET:
            configs[name], samples[name] = run_config(name, args, dev, peak)
        configs["_note"] = (f"each workload timed in this process with the same steps / warm-up "
                            f"({K} / {Wm}); frac = algorithmic bytes per launch / launch time / "
                            f"{peak} GB/s; {nsm} SMs")
    cpu = None
    if rank == 0 and not args.no_cpu_baseline:
        cpu = cpu_baseline(args, samples=samples, configs=configs)
    if rank != 0:
        return
    line = {
        "metric": METRIC, "value": round(value, 2), "unit": "GB/s", "n_gpus": world,
        "steps": K, "warmup": Wm, "ms_per_step": round(dt / K * 1e3, 5),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32",
        "data": "synthetic",
        "config": workload_config(w, lens, nb),
        "launch": {"partition_tokens": paged_partition(w, args.partition),
                   "parallelism": f"replicas x{world}"},
        "kv_gb_per_step": {"logical": kv_log / 1e9, "unique": kv_uni / 1e9},
        "value_unique_gbs": round(sum_over_ranks(kv_uni * K, world, dev) / dt / 1e9, 2),
        "decode_tokens_per_s": round(world * w.num_seqs * K / dt, 1),
        "attention_us_per_layer": round(attn_avg * 1e6, 3),
        "attention_us_median": head["us_per_layer_median"],
        "attention_us_p10_median_p90": [head["us_per_layer_p10_p90"][0],
                                        head["us_per_layer_median"],
                                        head["us_per_layer_p10_p90"][1]],
        "attention_us_median_x_sm_mhz": head.get("us_median_x_sm_mhz"),
        "append_plus_attention_us_per_layer": round(dt_local / K / L * 1e6, 3),
        "decode_tokens_per_s_model": model_tokens_per_s(w, dt_local / K / L),
        "append": "fused into the decode kernel" if decode_kernel_name(w) ==
                  "paged_decode_mma2_kernel" and w.kv_dtype == "bf16"
                  else "append kernel, then decode",
        "roofline": {"bound": "hbm", "achieved": round(achieved, 2), "peak": peak, "unit": "GB/s",
                     "frac": round(achieved / peak, 4), "traffic": traffic,
                     "frac_median": head["frac_median"],
                     "peak_source": f"{peak_src} (MEASURED_PEAKS.json hbm_gbs, burst copy)"
                     if peak_src == "measured" else "fallback 6800 GB/s",
                     "kernel": decode_kernel_name(w) + (" + paged_decode_reduce_kernel"
                                                        if paged_parts(w, args.partition) > 1
                                                        else ""),
                     "alg_bytes_per_launch": attn_bytes,
                     "frac_of_in_run_copy": round(achieved / bw["copy_gbs"], 4) if bw else None,
                     "frac_of_in_run_read": round(achieved / bw["read_gbs"], 4) if bw else None},
        "sustained": sustain,
        "in_run_bandwidth_gbs": {k: round(v, 1) for k, v in bw.items()} if bw else None,
        "configs": configs,
        "graph": graph,
        "cpu_baseline": cpu,
        "e2e": e2e,
        "gpu_launches": K * launches_per_step(w, args.partition),
        "clocks": clk,
        "device_status": status,
        "kernel_sources_sha": sha,
    }
    print(json.dumps(line), flush=True)


def paged_partition(w, partition=0) -> int:
    """The partition the library picks (8-bit caches: twice the 16-bit one)."""
    import paged_kv_cache_295_gb300 as pkv
    lens = W.context_lens(w)
    P = pkv.partition_tokens(w.num_seqs, w.num_q_heads, w.num_kv_heads, int(lens.max()),
                             partition)
    if partition == 0 and w.kv_dtype in ("fp8_e4m3", "int8"):
        P = min(4096, 2 * P)
    return P


def paged_parts(w, partition=0) -> int:
    return max(1, -(-int(W.context_lens(w).max()) // paged_partition(w, partition)))


def launches_per_step(w, partition=0) -> int:
    """Our kernels per step: per layer one decode (with the append fused in,
    else an append kernel too) and one reduce if split."""
    fused = decode_kernel_name(w) == "paged_decode_mma2_kernel" and w.kv_dtype == "bf16"
    return w.num_layers * ((1 if fused else 2) + (1 if paged_parts(w, partition) > 1 else 0))


def run_graph(st, K, Wm, world, dev, dt_eager, kv_log):
    """Times the step as a replayed CUDA graph (decode_graph_*): returns the
    graph report and the (dt, value, dt_local) that replace the eager ones."""
    import torch
    import paged_kv_cache_295_gb300 as pkv
    w = st.w
    S = w.num_seqs
    buckets = sorted({1 << i for i in range(S.bit_length()) if (1 << i) < S} | {S})
    g = pkv.DecodeGraph(st.eng, w.num_q_heads, st.tables.shape[1], buckets,
                        device_status=st.status)
    L = w.num_layers
    for l in range(L):
        g.q[l, :S] = st.q[l][0]
        g.k_new[l, :S] = st.kn[l][0]
        g.v_new[l, :S] = st.vn[l][0]
    g.slots[:S] = st.slots
    g.tables[:S] = st.tables
    g.lens[:S] = st.ctx
    for _ in range(Wm):
        g.launch(S)
    torch.cuda.synchronize(dev)
    barrier(world)
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    t0.record()
    for _ in range(K):
        g.launch(S)
    t1.record()
    torch.cuda.synchronize(dev)
    barrier(world)
    dt_local = t0.elapsed_time(t1) * 1e-3
    dt = max_over_ranks(dt_local, world, dev)
    value = sum_over_ranks(kv_log * K, world, dev) / dt / 1e9
    rep = {"buckets": buckets, "bucket_used": S, "ms_per_step": round(dt / K * 1e3, 5),
           "eager_ms_per_step": round(dt_eager / K * 1e3, 5),
           "speedup_vs_eager": round(dt_eager / dt, 3),
           "partition_tokens": pkv.partition_tokens(S, w.num_q_heads, w.num_kv_heads,
                                                    st.tables.shape[1] * w.block_size),
           "note": "value, ms_per_step and decode_tokens_per_s are the graph replay's"}
    g.close()
    return rep, dt, value, dt_local


def run_e2e(st, args, dev, world):
    """The same step through the public API from pinned host buffers each step:
    host block tables from the pool, H2D of q / new K,V / slots / tables /
    lengths, append + attention for every layer, D2H of the output, sync."""
    import torch
    w = st.w
    n = args.e2e_steps or min(args.steps, 200)
    L, S = w.num_layers, w.num_seqs
    mb = st.tables_h.shape[1]
    pin = dict(pin_memory=True)
    q_h = [[x.cpu().pin_memory() for x in st.q[l]] for l in range(L)]
    kn_h = [[x.cpu().pin_memory() for x in st.kn[l]] for l in range(L)]
    vn_h = [[x.cpu().pin_memory() for x in st.vn[l]] for l in range(L)]
    slots_h = torch.from_numpy(st.step_slots_h.copy()).pin_memory()
    tables_h = torch.empty((S, mb), dtype=torch.int32, **pin)
    lens_h = torch.empty((S,), dtype=torch.int32, **pin)
    out_h = torch.empty((S, w.num_q_heads, w.head_dim), dtype=torch.float32, **pin)
    q_d = [torch.empty_like(st.q[l][0]) for l in range(L)]
    kn_d = [torch.empty_like(st.kn[l][0]) for l in range(L)]
    vn_d = [torch.empty_like(st.vn[l][0]) for l in range(L)]
    slots_d, tables_d, lens_d = (torch.empty_like(st.slots), torch.empty_like(st.tables),
                                 torch.empty_like(st.ctx))
    bi = (sum(x[0].numel() * x[0].element_size() for x in q_h + kn_h + vn_h)
          + slots_h.numel() * 8 + tables_h.numel() * 4 + lens_h.numel() * 4)
    bo = out_h.numel() * 4
    seqs = list(range(S))
    stream = torch.cuda.current_stream(dev)

    def one(i):
        k = i % len(q_h[0])
        st.eng.pool.batch_tables(seqs, mb, tables_h.numpy(), lens_h.numpy())
        slots_d.copy_(slots_h, non_blocking=True)
        tables_d.copy_(tables_h, non_blocking=True)
        lens_d.copy_(lens_h, non_blocking=True)
        for l in range(L):
            q_d[l].copy_(q_h[l][k], non_blocking=True)
            kn_d[l].copy_(kn_h[l][k], non_blocking=True)
            vn_d[l].copy_(vn_h[l][k], non_blocking=True)
            st.eng.append_attend(l, q_d[l], kn_d[l], vn_d[l], slots_d, tables_d, lens_d,
                                 st.max_ctx, out=st.out, workspace=st.ws,
                                 partition=st.partition)
        out_h.copy_(st.out, non_blocking=True)
        stream.synchronize()

    for i in range(3):
        one(i)
    barrier(world)
    torch.cuda.synchronize(dev)
    t = time.perf_counter()
    for i in range(n):
        one(i)
    dt = max_over_ranks(time.perf_counter() - t, world, dev)
    kv = sum_over_ranks(kv_bytes_logical(w, st.lens) * L * n, world, dev)
    eager = {"value": round(kv / dt / 1e9, 2), "ms_per_step": round(dt / n * 1e3, 5),
             "calls": "per step: pool tables, torch copies, paged_attention_decode_append "
                      "per layer, D2H, sync"}

    # the same step as one public call: decode_graph_step_host on a captured graph
    import paged_kv_cache_295_gb300 as pkv
    g = pkv.DecodeGraph(st.eng, w.num_q_heads, mb, [S], device_status=st.status)
    qg = torch.stack([q_h[l][0] for l in range(L)]).pin_memory()
    kg = torch.stack([kn_h[l][0] for l in range(L)]).pin_memory()
    vg = torch.stack([vn_h[l][0] for l in range(L)]).pin_memory()
    outg = torch.empty((L, S, w.num_q_heads, w.head_dim), dtype=torch.float32, pin_memory=True)
    for _ in range(3):
        g.step_host(st.eng.pool, seqs, qg, kg, vg, slots_h, outg, stream=stream)
    barrier(world)
    t = time.perf_counter()
    for _ in range(n):
        g.step_host(st.eng.pool, seqs, qg, kg, vg, slots_h, outg, stream=stream)
    dtg = max_over_ranks(time.perf_counter() - t, world, dev)
    g.close()
    bo_g = outg.numel() * 4
    return {"value": round(kv / dtg / 1e9, 2), "unit": "GB/s", "steps": n,
            "ms_per_step": round(dtg / n * 1e3, 5),
            "h2d_bytes_per_step": int(bi), "d2h_bytes_per_step": int(bo_g),
            "decode_tokens_per_s": round(world * S * n / dtg, 1),
            "call": "decode_graph_step_host: pool tables -> pinned staging, one copy per "
                    "input buffer, graph replay of every layer's append + decode, output "
                    "copy, one stream sync",
            "timer": "host wall clock around each call", "eager": eager}


# ---------------------------------------------------------- prefill arm ---
def prefill_alg_flops(n, ctx, num_q_heads, head_dim, causal=True) -> int:
    """Flops of the two contractions of one prefill launch: 4 * head_dim per
    (query token, query head, visible key) - 2 D for q.k and 2 D for p.v."""
    n = np.asarray(n, dtype=np.int64)
    ctx = np.asarray(ctx, dtype=np.int64)
    keys = (n * (ctx - n) + n * (n + 1) // 2) if causal else n * ctx
    return int(keys.sum()) * num_q_heads * 4 * head_dim


class PrefillStep:
    """A chunked-prefill step of ``w`` resident on one GPU: append the chunk's
    K/V rows, then prefill attention over each sequence's paged context."""

    def __init__(self, w, device, keep_src=False):
        import torch
        import paged_kv_cache_295_gb300 as pkv
        from paged_kv_cache_295_gb300.engine import PagedKVCache
        self.w, self.device = w, device
        self.n, self.lens = W.prefill_lens(w)
        S, hq, hkv, d, bs = len(self.n), w.num_q_heads, w.num_kv_heads, w.head_dim, w.block_size
        nb = W.prefill_num_blocks(w, self.lens)
        code = {"bf16": pkv.BF16, "fp8_e4m3": pkv.FP8_E4M3, "int8": pkv.INT8}[w.kv_dtype]
        self.eng = eng = PagedKVCache(1, hkv, d, bs, nb, code, device=device,
                                      initial_free_order=W.free_order(w, nb))
        pre, chk = [], []
        for s in range(S):
            eng.pool.seq_create(s)
            pre.append(eng.pool.append_tokens(s, int(self.lens[s] - self.n[s])))
            chk.append(eng.pool.append_tokens(s, int(self.n[s])))
        mb = int(max(len(eng.pool.block_table(s)) for s in range(S)))
        tables, lens_pool = eng.pool.batch_tables(list(range(S)), mb)
        assert np.array_equal(lens_pool, self.lens)
        self.tables_h = tables
        self.max_q, self.max_ctx = int(self.n.max()), int(self.lens.max())
        off = np.concatenate([[0], np.cumsum(self.lens)])
        pre_idx = np.concatenate([np.arange(off[s], off[s + 1] - self.n[s]) for s in range(S)])
        chk_idx = np.concatenate([np.arange(off[s + 1] - self.n[s], off[s + 1])
                                  for s in range(S)])
        gen = torch.Generator(device=device)
        gen.manual_seed(w.seed * 1000)
        U, T = int(self.lens.sum()), int(self.n.sum())
        k_src = torch.randn((U, hkv, d), generator=gen, device=device).to(torch.bfloat16)
        v_src = torch.randn((U, hkv, d), generator=gen, device=device).to(torch.bfloat16)
        self.q = torch.randn((T, hq, d), generator=gen, device=device).to(torch.bfloat16)
        if w.kv_dtype in ("fp8_e4m3", "int8"):   # static per-head scales: absmax / 448 or / 127
            qmax = 448.0 if w.kv_dtype == "fp8_e4m3" else 127.0
            eng.k_scale[0] = k_src.float().abs().amax(dim=(0, 2)) / qmax
            eng.v_scale[0] = v_src.float().abs().amax(dim=(0, 2)) / qmax
        pre_i = torch.from_numpy(pre_idx).to(device)
        if pre_idx.size:
            eng.append(0, k_src[pre_i], v_src[pre_i],
                       torch.from_numpy(np.concatenate(pre)).to(device))
        chk_i = torch.from_numpy(chk_idx).to(device)
        self.kn, self.vn = k_src[chk_i].contiguous(), v_src[chk_i].contiguous()
        self.slots = torch.from_numpy(np.concatenate(chk)).to(device)
        self.src = (k_src, v_src, off) if keep_src else None
        del k_src, v_src
        self.qs_h = np.concatenate([[0], np.cumsum(self.n)]).astype(np.int32)
        self.qs = torch.from_numpy(self.qs_h).to(device)
        self.tables = torch.from_numpy(tables).to(device)
        self.ctx = torch.from_numpy(self.lens.astype(np.int32)).to(device)
        self.out = torch.empty((T, hq, d), dtype=torch.float32, device=device)
        self.status = torch.zeros(1, dtype=torch.int32, device=device)
        torch.cuda.synchronize(device)

    def run(self, ev=None):
        self.eng.append(0, self.kn, self.vn, self.slots, device_status=self.status)
        if ev is not None:
            ev[0].record()
        self.eng.prefill(0, self.q, self.qs, self.tables, self.ctx, self.max_q, self.max_ctx,
                         out=self.out, device_status=self.status)
        if ev is not None:
            ev[1].record()


def prefill_config(w, n, lens, nb):
    return {"workload": w.name, "num_layers": w.num_layers, "num_seqs": int(len(n)),
            "num_q_heads": w.num_q_heads, "num_kv_heads": w.num_kv_heads,
            "head_dim": w.head_dim, "block_size": w.block_size, "kv_dtype": w.kv_dtype,
            "q_dtype": w.q_dtype, "out_dtype": "f32", "causal": True,
            "chunk_tokens": int(n.max()), "query_tokens": int(n.sum()),
            "cached_prefix": f"{w.chunk_tokens} x U{{0..{w.max_prefix_chunks}}} seed {w.seed}",
            "sum_ctx": int(lens.sum()), "max_ctx": int(lens.max()), "num_blocks": int(nb),
            "l2": f"inputs larger than L2: {int(lens.sum()) * 2 * w.num_kv_heads * w.head_dim * 2 / 1e9:.3f}"
                  " GB of K/V per step vs 129 MB L2"}


def run_prefill_e2e(st, args, dev, world):
    """The prefill step through the public API from pinned host buffers: H2D of
    q, the chunk's K/V rows, slots, query_start, tables and lengths; append +
    prefill; D2H of the output; one stream sync."""
    import torch
    n = args.e2e_steps or min(args.steps, 50)
    pin = dict(pin_memory=True)
    host = {k: v.cpu().pin_memory() for k, v in (("q", st.q), ("kn", st.kn), ("vn", st.vn),
                                                  ("slots", st.slots), ("qs", st.qs),
                                                  ("tables", st.tables), ("ctx", st.ctx))}
    devb = {k: torch.empty_like(getattr(st, k)) for k in host}
    out_h = torch.empty(st.out.shape, dtype=torch.float32, **pin)
    bi = sum(t.numel() * t.element_size() for t in host.values())
    bo = out_h.numel() * 4
    stream = torch.cuda.current_stream(dev)

    def one():
        for k in host:
            devb[k].copy_(host[k], non_blocking=True)
        st.eng.append(0, devb["kn"], devb["vn"], devb["slots"])
        st.eng.prefill(0, devb["q"], devb["qs"], devb["tables"], devb["ctx"], st.max_q,
                       st.max_ctx, out=st.out)
        out_h.copy_(st.out, non_blocking=True)
        stream.synchronize()

    for _ in range(3):
        one()
    barrier(world)
    torch.cuda.synchronize(dev)
    t = time.perf_counter()
    for _ in range(n):
        one()
    dt = max_over_ranks(time.perf_counter() - t, world, dev)
    flops = sum_over_ranks(prefill_alg_flops(st.n, st.lens, st.w.num_q_heads, st.w.head_dim) * n,
                           world, dev)
    return {"value": round(flops / dt / 1e12, 2), "unit": "TFLOP/s", "steps": n,
            "ms_per_step": round(dt / n * 1e3, 5), "h2d_bytes_per_step": int(bi),
            "d2h_bytes_per_step": int(bo),
            "prefill_tokens_per_s": round(world * int(st.n.sum()) * n / dt, 1),
            "timer": "host wall clock, one stream sync per step"}


def run_prefill(args):
    import torch
    rank, world, local = dist_env()
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", init_method="env://")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    w = workload_of(args)
    K, Wm = args.steps, args.warmup
    if Wm < 3:
        raise SystemExit("--warmup must be >= 3")
    st = PrefillStep(w, dev)
    for _ in range(Wm):
        st.run()
    torch.cuda.synchronize(dev)
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(K)]
    clocks = ClockSampler(local)
    barrier(world)
    torch.cuda.synchronize(dev)
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    t0.record()
    for i in range(K):
        st.run(ev[i])
    t1.record()
    torch.cuda.synchronize(dev)
    barrier(world)
    clk = clocks.stop()
    dt = max_over_ranks(t0.elapsed_time(t1) * 1e-3, world, dev)
    attn = [e[0].elapsed_time(e[1]) * 1e-3 for e in ev]
    flops = prefill_alg_flops(st.n, st.lens, w.num_q_heads, w.head_dim)
    value = sum_over_ranks(flops * K, world, dev) / dt / 1e12
    attn_avg = statistics.fmean(attn)
    peak, peak_src = measured_peaks("bf16_tflops", 1900.0)
    achieved = flops / attn_avg / 1e12
    e2e = run_prefill_e2e(st, args, dev, world)
    cpu = None
    if rank == 0 and not args.no_cpu_baseline:
        cpu = cpu_baseline(args)
    if rank != 0:
        return
    line = {
        "metric": PREFILL_METRIC, "value": round(value, 2), "unit": "TFLOP/s", "n_gpus": world,
        "steps": K, "warmup": Wm, "ms_per_step": round(dt / K * 1e3, 5),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic",
        "config": prefill_config(w, st.n, st.lens, st.eng.num_blocks),
        "launch": {"parallelism": f"replicas x{world}", "query_rows_per_cta": 128,
                   "keys_per_tile": 64},
        "prefill_tokens_per_s": round(world * int(st.n.sum()) * K / dt, 1),
        "attention_us": round(attn_avg * 1e6, 3),
        "attention_us_median": round(statistics.median(attn) * 1e6, 3),
        "append_plus_attention_us": round(dt / K * 1e6, 3),
        "roofline": {"bound": "tensor", "achieved": round(achieved, 2), "peak": peak,
                     "unit": "TFLOP/s", "frac": round(achieved / peak, 4), "traffic": None,
                     "peak_source": f"{peak_src} (MEASURED_PEAKS.json bf16_tflops, burst)"
                     if peak_src == "measured" else "fallback 1900 TFLOP/s",
                     "kernel": "paged_prefill_tc_kernel", "alg_flops_per_launch": flops},
        "cpu_baseline": cpu,
        "e2e": e2e,
        "gpu_launches": 2 * K,
        "clocks": clk,
        "device_status": int(st.status.item()),
        "kernel_sources_sha": kernel_sources_sha(),
    }
    print(json.dumps(line), flush=True)


class OraclePrefillStep:
    """One sequence of the prefill workload on the host for the oracle; a step
    is one query row (every head) against its visible keys."""

    def __init__(self, w):
        from oracle import attention as OA
        self.w = w
        self.n, self.lens = W.prefill_lens(w)
        s = int(np.argmax(self.lens))
        self.s, L, hkv, d = s, int(self.lens[s]), w.num_kv_heads, w.head_dim
        r = W.rng(w.seed, 900)
        self.K = OA.to_f64(W.store(r.standard_normal((L, hkv, d), dtype=np.float32), "bf16"),
                           "bf16")
        self.V = OA.to_f64(W.store(r.standard_normal((L, hkv, d), dtype=np.float32), "bf16"),
                           "bf16")
        self.q = OA.to_f64(W.store(r.standard_normal((int(self.n[s]), w.num_q_heads, d),
                                                     dtype=np.float32), "bf16"), "bf16")
        if w.kv_dtype == "fp8_e4m3":   # the cache holds E4M3 codes: their dequantised values
            from oracle import fp8
            for name in ("K", "V"):
                x = getattr(self, name).astype(np.float32)
                sc = (np.abs(x).max(axis=(0, 2)) / np.float32(448.0)).astype(np.float32)
                codes = fp8.encode_f32(x / sc[None, :, None])
                setattr(self, name, OA.fp8_dequant(codes, sc))
        elif w.kv_dtype == "int8":   # INT8 codes: their dequantised values
            for name in ("K", "V"):
                x = getattr(self, name).astype(np.float32)
                sc = (np.abs(x).max(axis=(0, 2)) / np.float32(127.0)).astype(np.float32)
                setattr(self, name, OA.int8_dequant(OA.int8_encode(x, sc), sc))

    def run(self, i):
        from oracle import prefill as OPF
        n, L = int(self.n[self.s]), int(self.lens[self.s])
        row = i % n
        OPF.attend_rows(self.q[row:row + 1], self.K, self.V, self.w.scale, [L - n + row])
        return (L - n + row + 1) * self.w.num_q_heads * 4 * self.w.head_dim


def run_prefill_reference(args):
    rank, world, _ = dist_env()
    if rank != 0:
        return
    w = workload_of(args)
    K, Wm = args.steps, args.warmup
    st = OraclePrefillStep(w)
    for i in range(Wm):
        st.run(i)
    fl, t = 0, time.perf_counter()
    for i in range(K):
        fl += st.run(Wm + i)
    dt = time.perf_counter() - t
    value = fl / dt / 1e12
    nb = W.prefill_num_blocks(w, st.lens)
    sample = (f"sequence {st.s} (context {int(st.lens[st.s])}), one query row (all heads) per "
              f"step, {K} steps, numpy float64 oracle, 1 thread")
    print(json.dumps({
        "impl": "reference", "metric": PREFILL_METRIC, "value": round(value, 8),
        "unit": "TFLOP/s", "n_gpus": world, "steps": K, "warmup": Wm,
        "ms_per_step": round(dt / K * 1e3, 4), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": prefill_config(w, st.n, st.lens, nb),
        "cpu_baseline": {"value": round(value, 8), "unit": "TFLOP/s", "cores": 1,
                         "kind": "oracle", "sample": sample},
        "e2e": {"value": round(value, 8), "unit": "TFLOP/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }), flush=True)


# ------------------------------------------------------- beam-fork arm ---
class ForkStep:
    """Beam forks over a resident pool: prompts appended, each forked into
    beams, one decode token per beam appended through the pool - the
    copy-on-write pairs that produces are this step's copy_blocks work."""

    def __init__(self, w, device):
        import torch
        import paged_kv_cache_295_gb300 as pkv
        from paged_kv_cache_295_gb300.engine import PagedKVCache
        self.w = w
        lens = W.fork_prompt_lens(w)
        bs = w.block_size
        nb = int(math.ceil(w.pool_slack * (int((-(-lens // bs)).sum()) + w.num_prompts * w.beams)))
        self.eng = eng = PagedKVCache(w.num_layers, w.num_kv_heads, w.head_dim, bs, nb, pkv.BF16,
                                      device=device, initial_free_order=W.free_order(w, nb),
                                      poison=False)
        gen = torch.Generator(device=device)
        gen.manual_seed(w.seed * 1000)
        for layer in range(w.num_layers):   # every block gets data (whole pool, one layer at a time)
            eng.storage[layer].copy_(torch.randn(eng.storage[layer].shape, generator=gen,
                                                 device=device).to(torch.bfloat16))
        beams = []
        for s, n in enumerate(lens):
            eng.pool.seq_create(s)
            eng.pool.append_tokens(s, int(n), want_slots=False)
            beams.append(s)
        nid = len(lens)
        for s, n in enumerate(lens):
            for _ in range(w.beams - 1):
                eng.pool.seq_fork_prefix(nid, s, int(n))
                beams.append(nid)
                nid += 1
        eng.pool.append_slots(beams)
        pairs = eng.pool.take_copies()
        # the engine's order: pairs of one source side by side (re-reads hit L2)
        self.pairs_h = np.ascontiguousarray(pairs[np.argsort(pairs[:, 0], kind="stable")])
        self.pairs = torch.from_numpy(self.pairs_h).to(device)
        self.lens = lens
        plane = eng.storage[0, 0]
        self.block_bytes = plane[0].numel() * plane.element_size()
        self.planes = 2 * w.num_layers
        self.nb = nb
        self.status = torch.zeros(1, dtype=torch.int32, device=device)
        torch.cuda.synchronize(device)

    def moved_bytes(self) -> int:
        """Algorithmic bytes of one copy_blocks launch: every distinct source
        block read once, every destination written (a prompt's partly filled
        block is the source of beams - 1 copies)."""
        srcs = len(set(self.pairs_h[:, 0].tolist()))
        return (srcs + int(self.pairs_h.shape[0])) * self.planes * self.block_bytes

    def run(self):
        import paged_kv_cache_295_gb300 as pkv
        pkv.copy_blocks(self.eng.storage, self.pairs, device_status=self.status)


def fork_config(w, lens, npairs, nb):
    return {"workload": w.name, "num_layers": w.num_layers, "num_prompts": w.num_prompts,
            "beams": w.beams, "num_kv_heads": w.num_kv_heads, "head_dim": w.head_dim,
            "block_size": w.block_size, "kv_dtype": w.kv_dtype,
            "prompt_lens": f"uniform[{w.ctx_lo},{w.ctx_hi}] seed {w.seed}, no multiple of the "
                           "block size", "copy_pairs": int(npairs), "planes": 2 * w.num_layers,
            "num_blocks": int(nb),
            "l2": "inputs larger than L2: each launch copies "
                  f"{npairs * 2 * w.num_layers * w.block_size * w.num_kv_heads * w.head_dim * 2 / 1e9:.2f}"
                  " GB vs 129 MB L2"}


def run_fork(args):
    import torch
    rank, world, local = dist_env()
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", init_method="env://")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    w = workload_of(args)
    K, Wm = args.steps, args.warmup
    if Wm < 3:
        raise SystemExit("--warmup must be >= 3")
    st = ForkStep(w, dev)
    for _ in range(Wm):
        st.run()
    torch.cuda.synchronize(dev)
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(K)]
    clocks = ClockSampler(local)
    barrier(world)
    torch.cuda.synchronize(dev)
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    t0.record()
    for i in range(K):
        ev[i][0].record()
        st.run()
        ev[i][1].record()
    t1.record()
    torch.cuda.synchronize(dev)
    barrier(world)
    clk = clocks.stop()
    dt = max_over_ranks(t0.elapsed_time(t1) * 1e-3, world, dev)
    ker = [e[0].elapsed_time(e[1]) * 1e-3 for e in ev]
    moved = st.moved_bytes()
    value = sum_over_ranks(moved * K, world, dev) / dt / 1e9
    peak, peak_src = measured_peaks()
    achieved = moved / statistics.fmean(ker) / 1e9
    # e2e: the pairs from pinned host memory, the copies, the status word back
    pairs_h = torch.from_numpy(st.pairs_h).pin_memory()
    pairs_d = torch.empty_like(st.pairs)
    stat_h = torch.empty(1, dtype=torch.int32, pin_memory=True)
    import paged_kv_cache_295_gb300 as pkv
    stream = torch.cuda.current_stream(dev)
    n_e2e = args.e2e_steps or min(K, 200)

    def one():
        pairs_d.copy_(pairs_h, non_blocking=True)
        pkv.copy_blocks(st.eng.storage, pairs_d, device_status=st.status)
        stat_h.copy_(st.status, non_blocking=True)
        stream.synchronize()

    for _ in range(3):
        one()
    barrier(world)
    t = time.perf_counter()
    for _ in range(n_e2e):
        one()
    dte = max_over_ranks(time.perf_counter() - t, world, dev)
    e2e = {"value": round(sum_over_ranks(moved * n_e2e, world, dev) / dte / 1e9, 2),
           "unit": "GB/s", "steps": n_e2e, "ms_per_step": round(dte / n_e2e * 1e3, 5),
           "h2d_bytes_per_step": int(pairs_h.numel() * 4), "d2h_bytes_per_step": 4,
           "timer": "host wall clock, one stream sync per step"}
    cpu = None
    if rank == 0 and not args.no_cpu_baseline:
        cpu = cpu_baseline(args)
    if rank != 0:
        return
    print(json.dumps({
        "metric": FORK_METRIC, "value": round(value, 2), "unit": "GB/s", "n_gpus": world,
        "steps": K, "warmup": Wm, "ms_per_step": round(dt / K * 1e3, 5),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic", "config": fork_config(w, st.lens, st.pairs_h.shape[0], st.nb),
        "launch": {"parallelism": f"replicas x{world}", "ctas": int(st.pairs_h.shape[0]) * st.planes},
        "copy_us": round(statistics.fmean(ker) * 1e6, 3),
        "roofline": {"bound": "hbm", "achieved": round(achieved, 2), "peak": peak, "unit": "GB/s",
                     "frac": round(achieved / peak, 4), "traffic": None,
                     "peak_source": f"{peak_src} (MEASURED_PEAKS.json hbm_gbs)",
                     "kernel": "copy_blocks_kernel", "alg_bytes_per_launch": moved},
        "cpu_baseline": cpu, "e2e": e2e, "gpu_launches": K, "clocks": clk,
        "device_status": int(st.status.item()), "kernel_sources_sha": kernel_sources_sha(),
    }), flush=True)


def run_fork_reference(args):
    """The oracle's copy_blocks on a host pool of the workload's plane shape:
    each step copies the pairs of one prompt's beams (beams - 1 blocks)."""
    from oracle import attention as OA
    rank, world, _ = dist_env()
    if rank != 0:
        return
    w = workload_of(args)
    K, Wm = args.steps, args.warmup
    nb = 2 * w.beams
    pool = W.store(W.rng(w.seed, 900).standard_normal(
        (w.num_layers, 2, nb, w.block_size, w.num_kv_heads, w.head_dim), dtype=np.float32),
        "bf16")
    pairs = [(0, 1 + i) for i in range(w.beams - 1)]
    for _ in range(Wm):
        OA.copy_blocks(pool, pairs)
    t = time.perf_counter()
    for _ in range(K):
        OA.copy_blocks(pool, pairs)
    dt = time.perf_counter() - t
    moved = (1 + len(pairs)) * 2 * w.num_layers * pool[0, 0, 0].nbytes * K   # one source
    value = moved / dt / 1e9
    sample = (f"{len(pairs)} block copies (one prompt's beams) x {2 * w.num_layers} planes per "
              f"step, {K} steps, numpy, 1 thread")
    print(json.dumps({
        "impl": "reference", "metric": FORK_METRIC, "value": round(value, 4), "unit": "GB/s",
        "n_gpus": world, "steps": K, "warmup": Wm, "ms_per_step": round(dt / K * 1e3, 4),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic",
        "config": fork_config(w, W.fork_prompt_lens(w), w.num_prompts * (w.beams - 1), 0),
        "cpu_baseline": {"value": round(value, 4), "unit": "GB/s", "cores": 1, "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": round(value, 4), "unit": "GB/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }), flush=True)


# ------------------------------------------------------------- swap arm ---
class SwapStep:
    """Every sequence swapped out (device -> host) and back in, through the
    pool and swap_blocks; the host area is page-locked memory."""

    def __init__(self, w, device):
        import torch
        import paged_kv_cache_295_gb300 as pkv
        from paged_kv_cache_295_gb300.engine import PagedKVCache
        self.w = w
        self.lens = W.swap_lens(w)
        bs = w.block_size
        blocks = int((-(-self.lens // bs)).sum())
        nb = blocks + 16
        self.eng = eng = PagedKVCache(w.num_layers, w.num_kv_heads, w.head_dim, bs, nb, pkv.BF16,
                                      device=device, initial_free_order=W.free_order(w, nb),
                                      poison=False)
        gen = torch.Generator(device=device)
        gen.manual_seed(w.seed * 1000)
        for layer in range(w.num_layers):
            eng.storage[layer].copy_(torch.randn(eng.storage[layer].shape, generator=gen,
                                                 device=device).to(torch.bfloat16))
        eng.host_area(blocks)
        for s, n in enumerate(self.lens):
            eng.pool.seq_create(s)
            eng.pool.append_tokens(s, int(n), want_slots=False)
        plane = eng.storage[0, 0]
        self.block_bytes = plane[0].numel() * plane.element_size()
        self.moved = blocks * 2 * w.num_layers * self.block_bytes   # each way
        self.nb = nb
        self.status = torch.zeros(1, dtype=torch.int32, device=device)
        torch.cuda.synchronize(device)

    def run(self, ev=None):
        seqs = range(len(self.lens))
        if ev is not None:
            ev[0].record()
        for s in seqs:
            self.eng.swap_out(s, device_status=self.status)
        if ev is not None:
            ev[1].record()
        for s in seqs:
            self.eng.swap_in(s, device_status=self.status)
        if ev is not None:
            ev[2].record()


def link_reference(device, nbytes=1 << 30, reps=5):
    """GB/s of cudaMemcpyAsync between page-locked host memory and the device."""
    import torch
    h = torch.empty(nbytes, dtype=torch.uint8, pin_memory=True)
    d = torch.empty(nbytes, dtype=torch.uint8, device=device)
    res = {}
    for name, fn in (("d2h_gbs", lambda: h.copy_(d, non_blocking=True)),
                     ("h2d_gbs", lambda: d.copy_(h, non_blocking=True))):
        fn()
        ts = []
        for _ in range(reps):
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record()
            fn()
            e1.record()
            e1.synchronize()
            ts.append(e0.elapsed_time(e1) * 1e-3)
        res[name] = nbytes / min(ts) / 1e9
    del h, d
    return res


def run_swap(args):
    import torch
    rank, world, local = dist_env()
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", init_method="env://")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    w = workload_of(args)
    K, Wm = args.steps, args.warmup
    if Wm < 3:
        raise SystemExit("--warmup must be >= 3")
    link = link_reference(dev)
    st = SwapStep(w, dev)
    for _ in range(Wm):
        st.run()
    torch.cuda.synchronize(dev)
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(K)]
    clocks = ClockSampler(local)
    barrier(world)
    torch.cuda.synchronize(dev)
    t = time.perf_counter()
    for i in range(K):
        st.run(ev[i])
    torch.cuda.synchronize(dev)
    dt = max_over_ranks(time.perf_counter() - t, world, dev)
    barrier(world)
    clk = clocks.stop()
    out_s = statistics.fmean(e[0].elapsed_time(e[1]) * 1e-3 for e in ev)
    in_s = statistics.fmean(e[1].elapsed_time(e[2]) * 1e-3 for e in ev)
    value = sum_over_ranks(2 * st.moved * K, world, dev) / dt / 1e9
    out_gbs, in_gbs = st.moved / out_s / 1e9, st.moved / in_s / 1e9
    cpu = None
    if rank == 0 and not args.no_cpu_baseline:
        cpu = cpu_baseline(args)
    if rank != 0:
        return
    print(json.dumps({
        "metric": SWAP_METRIC, "value": round(value, 2), "unit": "GB/s", "n_gpus": world,
        "steps": K, "warmup": Wm, "ms_per_step": round(dt / K * 1e3, 5),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic",
        "config": {"workload": w.name, "num_seqs": w.num_seqs, "num_layers": w.num_layers,
                   "num_kv_heads": w.num_kv_heads, "head_dim": w.head_dim,
                   "block_size": w.block_size, "kv_dtype": w.kv_dtype,
                   "context_lens": f"uniform[{w.ctx_lo},{w.ctx_hi}] seed {w.seed}",
                   "bytes_each_way": st.moved, "num_blocks": st.nb,
                   "l2": f"inputs larger than L2: {st.moved / 1e9:.2f} GB each way vs 129 MB L2"},
        "swap_out_gbs": round(out_gbs, 2), "swap_in_gbs": round(in_gbs, 2),
        "roofline": {"bound": "host_link", "achieved": round(min(out_gbs, in_gbs), 2),
                     "peak": round(min(link["d2h_gbs"], link["h2d_gbs"]), 2), "unit": "GB/s",
                     "frac": round(min(out_gbs / link["d2h_gbs"], in_gbs / link["h2d_gbs"]), 4),
                     "traffic": None,
                     "peak_source": "in-run cudaMemcpyAsync of 1 GiB between page-locked host "
                                    "memory and the device (the slower direction)",
                     "kernel": "swap_blocks_kernel (timed by direction, host pool calls and "
                               "pair uploads inside)",
                     "alg_bytes_per_direction": st.moved},
        "in_run_link_gbs": {k: round(v, 1) for k, v in link.items()},
        "cpu_baseline": cpu,
        "e2e": {"value": round(value, 2), "unit": "GB/s", "steps": K,
                "ms_per_step": round(dt / K * 1e3, 5),
                "h2d_bytes_per_step": int(st.moved), "d2h_bytes_per_step": int(st.moved),
                "timer": "host wall clock over the whole step (pool calls, pair uploads, "
                         "both directions)"},
        "gpu_launches": 2 * w.num_seqs * K, "clocks": clk,
        "device_status": int(st.status.item()), "kernel_sources_sha": kernel_sources_sha(),
    }), flush=True)


def run_swap_reference(args):
    """The oracle pool's swap out and in plus its host copies for one sequence
    per step, on a host pool of the workload's plane shape."""
    from oracle import attention as OA
    from oracle import pool as OP
    rank, world, _ = dist_env()
    if rank != 0:
        return
    w = workload_of(args)
    K, Wm = args.steps, args.warmup
    lens = W.swap_lens(w)
    n = int(lens[0])
    nb = -(-n // w.block_size) + 2
    pool = W.store(W.rng(w.seed, 900).standard_normal(
        (w.num_layers, 2, nb, w.block_size, w.num_kv_heads, w.head_dim), dtype=np.float32), "bf16")
    host = np.zeros((nb,) + pool.shape[:2] + pool.shape[3:], dtype=pool.dtype)
    op = OP.Pool(w.num_layers, w.num_kv_heads, w.head_dim, w.block_size, 2, nb)
    op.host_init(nb)
    op.seq_create(0)
    op.seq_append_tokens(0, n)
    moved = 0

    def step():
        OA.swap_blocks(pool, host, op.seq_swap_out(0), True)
        pairs = op.seq_swap_in(0)
        OA.swap_blocks(pool, host, pairs, False)
        return 2 * len(pairs) * pool[:, :, 0].nbytes

    for _ in range(Wm):
        step()
    t = time.perf_counter()
    for _ in range(K):
        moved += step()
    dt = time.perf_counter() - t
    value = moved / dt / 1e9
    sample = f"sequence 0 ({n} tokens) out and back in per step, {K} steps, numpy, 1 thread"
    print(json.dumps({
        "impl": "reference", "metric": SWAP_METRIC, "value": round(value, 4), "unit": "GB/s",
        "n_gpus": world, "steps": K, "warmup": Wm, "ms_per_step": round(dt / K * 1e3, 4),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic", "config": {"workload": w.name},
        "cpu_baseline": {"value": round(value, 4), "unit": "GB/s", "cores": 1, "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": round(value, 4), "unit": "GB/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }), flush=True)


# ------------------------------------------------- reference arm (oracle) ---
def workload_config(w, lens, nb):
    """The workload description both arms report (no launch details)."""
    return {
        "workload": w.name, "num_layers": w.num_layers, "num_seqs": w.num_seqs,
        "num_q_heads": w.num_q_heads, "num_kv_heads": w.num_kv_heads,
        "head_dim": w.head_dim, "block_size": w.block_size, "kv_dtype": w.kv_dtype,
        "q_dtype": w.q_dtype, "out_dtype": "f32",
        "context_lens": (f"{w.ctx_law}[{w.ctx_lo},{w.ctx_hi}] seed {w.seed}"
                         if w.ctx_law != "fixed" else str(list(w.ctx_fixed))),
        "prefix": (f"{w.prefix_tokens} tokens shared by {w.prefix_seqs} sequences"
                   if w.prefix_tokens else None),
        "sum_ctx": int(np.sum(lens)), "max_ctx": int(np.max(lens)), "num_blocks": int(nb),
        "l2": f"inputs larger than L2: {kv_bytes_unique(w, lens) * w.num_layers / 1e9:.3f} GB "
              "of K/V read per step vs 129 MB L2",
    }


class OracleStep:
    """Layer 0 of the workload on the host for the oracle: one sequence per step."""

    def __init__(self, w, seqs):
        import torch
        from oracle import pool as OP
        from paged_kv_cache_295_gb300.engine import build_prompts

        class OraclePool:   # the oracle pool behind the C pool wrapper's call names
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

        self.w = w
        S, hkv, d, bs = w.num_seqs, w.num_kv_heads, w.head_dim, w.block_size
        self.lens = W.context_lens(w)
        self.nb = W.num_blocks(w, self.lens)
        op = OraclePool(w.num_layers, hkv, d, bs, W.ELEM_BYTES[w.kv_dtype], self.nb,
                        initial_free_order=W.free_order(w, self.nb).tolist())
        build_prompts(op, self.lens, w.prefix_tokens, w.prefix_seqs)
        op.append_slots(range(S))
        mb = max(len(op.p.tables[s]) for s in range(S))
        self.tables = np.asarray(op.p.padded_tables(list(range(S)), mb)[0], dtype=np.int64)
        dt = {"f32": np.float32, "bf16": np.uint16, "fp8_e4m3": np.uint8,
              "int8": np.int8}[w.kv_dtype]
        self.kc = np.zeros((self.nb, bs, hkv, d), dtype=dt)
        self.vc = np.zeros_like(self.kc)
        r = W.rng(w.seed, 900)
        self.k_scale = np.full(hkv, 4.5 / 448, np.float32)
        self.v_scale = np.full(hkv, 4.5 / 448, np.float32)
        kh = W.k_head_scales(w)[None, None, :, None]
        done = set()
        for s in seqs:
            for b in self.tables[s][: -(-int(self.lens[s]) // bs)]:
                if b in done:
                    continue
                done.add(int(b))
                for cache, sc in ((self.kc, self.k_scale), (self.vc, self.v_scale)):
                    x = r.standard_normal((1, bs, hkv, d), dtype=np.float32)
                    if cache is self.kc:
                        x = x * kh
                    if w.kv_dtype == "fp8_e4m3":   # input generation via torch's float8 cast
                        y = np.clip(x / sc[None, None, :, None], -448, 448).astype(np.float32)
                        cache[b] = torch.from_numpy(y[0]).to(torch.float8_e4m3fn).view(
                            torch.uint8).numpy()
                    elif w.kv_dtype == "int8":     # codes drawn directly
                        cache[b] = r.integers(-127, 128, size=(bs, hkv, d)).astype(np.int8)
                    else:
                        cache[b] = W.store(x[0], w.kv_dtype)
        self.q = W.store(r.standard_normal((S, w.num_q_heads, d), dtype=np.float32), w.q_dtype)

    def run(self, s):
        from oracle import attention as OA
        w = self.w
        OA.paged_attention_decode(self.q, self.kc, self.vc, self.tables, self.lens, w.scale,
                                  w.q_dtype, w.kv_dtype, self.k_scale, self.v_scale, seqs=[s])
        return int(self.lens[s]) * 2 * row_bytes(w)


def _affinity_cores() -> int:
    try:
        return len(os.sched_getaffinity(0))
    except Exception:
        return os.cpu_count() or 1


def _oracle_worker(wname, seqs, steps, warm, ready, go, results):
    """One reference worker process: the oracle on its own sequences of layer 0,
    one sequence per step, after every worker has built its inputs."""
    w = WORKLOADS[wname]
    st = OracleStep(w, sorted(set(seqs)))
    order = [seqs[i % len(seqs)] for i in range(warm + steps)]
    for i in range(warm):
        st.run(order[i])
    ready.release()
    go.wait()
    t0, byts = time.monotonic(), 0
    for i in range(steps):
        byts += st.run(order[warm + i])
    results.put((byts, t0, time.monotonic()))


def run_reference(args):
    """The oracle on this host's cores: ``--cpu-cores`` worker processes (all
    the cores this process may run on by default), one NumPy thread each; a
    step is one sequence of layer 0 per worker, worker i taking sequences i,
    i + N, ... in turn."""
    rank, world, _ = dist_env()
    if rank != 0:
        return
    w = workload_of(args)
    K, Wm = args.steps, args.warmup
    cores = args.cpu_cores or _affinity_cores()
    cores = max(1, min(cores, w.num_seqs))
    if cores == 1:
        order = [i % w.num_seqs for i in range(Wm + K)]
        st = OracleStep(w, sorted(set(order)))
        for i in range(Wm):
            st.run(order[i])
        byts, t = 0, time.perf_counter()
        for i in range(K):
            byts += st.run(order[Wm + i])
        dt = time.perf_counter() - t
        nb = st.nb
    else:
        import multiprocessing as mp
        ctx = mp.get_context("spawn")
        ready, go, results = ctx.Semaphore(0), ctx.Event(), ctx.Queue()
        procs = [ctx.Process(target=_oracle_worker,
                             args=(w.name, list(range(i, w.num_seqs, cores)), K, Wm, ready, go,
                                   results)) for i in range(cores)]
        for pr in procs:
            pr.start()
        for _ in procs:
            ready.acquire()
        go.set()
        res = [results.get() for _ in procs]
        for pr in procs:
            pr.join()
        byts = sum(r[0] for r in res)
        dt = max(r[2] for r in res) - min(r[1] for r in res)
        nb = W.num_blocks(w, W.context_lens(w))
    value = byts / dt / 1e9
    sample = (f"layer 0, one sequence per step per worker ({cores} worker process"
              f"{'es' if cores > 1 else ''}, sequences dealt round-robin), {K} steps each, "
              "numpy float64 oracle, 1 thread per process")
    line = {
        "impl": "reference", "metric": METRIC, "value": round(value, 4), "unit": "GB/s",
        "n_gpus": world, "steps": K, "warmup": Wm, "ms_per_step": round(dt / K * 1e3, 4),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic", "config": workload_config(w, W.context_lens(w), nb),
        "cpu_baseline": {"value": round(value, 4), "unit": "GB/s", "cores": cores,
                         "kind": "oracle", "sample": sample, "cpu_model": _cpu_model()},
        "e2e": {"value": round(value, 4), "unit": "GB/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def oracle_check(samples, configs):
    """The oracle on each sampled sequence (the host copies of what the kernel
    read), against the output row the kernel wrote: max-abs error per workload,
    added to its ``configs`` record."""
    from oracle import attention as OA
    out = {}
    for name, rows in samples.items():
        errs, ctxs = [], []
        for smp in rows:
            nb = smp["k"].shape[0]
            ref = OA.paged_attention_decode(
                smp["q"], smp["k"], smp["v"], np.arange(nb, dtype=np.int64)[None, :],
                np.array([smp["context"]]), smp["scale"], smp["q_dtype"], smp["kv_dtype"],
                smp["k_scale"], smp["v_scale"])
            errs.append(float(np.abs(smp["out"].astype(np.float64) - ref).max()))
            ctxs.append(smp["context"])
        tol = ORACLE_TOL[rows[0]["kv_dtype"]]
        rec = {"seqs": [r["seq"] for r in rows], "contexts": ctxs, "layer": rows[0]["layer"],
               "max_abs_err": max(errs), "tol": tol, "ok": bool(max(errs) <= tol)}
        out[name] = rec
        if configs is not None and name in configs:
            configs[name]["oracle"] = rec
    return out


def cpu_baseline(args, samples=None, configs=None):
    """The oracle timed on this host on a bounded sample of the workload, in
    fresh processes: one worker with one thread, and (decode workloads) one
    worker per core this process may run on.  With ``samples`` it first checks
    the kernel's output rows against the oracle."""
    w = workload_of(args)
    prefill = isinstance(w, W.PrefillWorkload)
    parity = oracle_check(samples, configs) if samples else None
    if isinstance(w, (W.ForkWorkload, W.SwapWorkload)):
        steps = 100
    else:
        lens = W.prefill_lens(w)[1] if prefill else W.context_lens(w)
        per_step = float(np.mean(lens)) * w.num_q_heads * 1.2e-6     # ~1.2 us per token-head
        steps = int(max(2, min(10 * w.num_seqs, args.cpu_seconds / per_step)))
    env = dict(os.environ, OMP_NUM_THREADS="1", OPENBLAS_NUM_THREADS="1", MKL_NUM_THREADS="1",
               RANK="0", WORLD_SIZE="1", LOCAL_RANK="0", CUDA_VISIBLE_DEVICES="")
    unit = "TFLOP/s" if prefill else "GB/s"

    def one(cores, nsteps):
        cmd = [sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
               "--workload", w.name, "--steps", str(nsteps), "--warmup", "1",
               "--cpu-cores", str(cores)]
        try:
            r = subprocess.run(cmd, env=env, capture_output=True, text=True, timeout=600)
            line = json.loads([x for x in r.stdout.splitlines() if x.startswith("{")][-1])
            cb = line["cpu_baseline"]
            cb["cpu_model"] = _cpu_model()
            return cb
        except Exception as e:   # the baseline is reported, never the target
            return {"value": None, "unit": unit, "cores": cores, "kind": "oracle",
                    "sample": f"failed: {type(e).__name__}: {e}"[:200]}

    single = one(1, steps)
    decode = isinstance(w, W.DecodeWorkload)
    cores = min(_affinity_cores(), w.num_seqs) if decode else 1
    if cores > 1:
        cb = one(cores, steps)
        cb["single_core"] = single
    else:
        cb = single
    cb["threads_per_process"] = 1
    if parity is not None:
        cb["oracle_check"] = parity
    return cb


# Arm (implementer 0x41) CPU part numbers -> core names, for hosts whose
# /proc/cpuinfo gives only the part number.
_ARM_PARTS = {"0xd0c": "Arm Neoverse-N1", "0xd40": "Arm Neoverse-V1",
              "0xd49": "Arm Neoverse-N2", "0xd4f": "Arm Neoverse-V2"}


def _cpu_model():
    try:
        r = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10)
        for ln in r.stdout.splitlines():
            if ln.lower().startswith("model name"):
                name = ln.split(":", 1)[1].strip()
                if name and name != "-":
                    return name
    except Exception:
        pass
    try:
        part = None
        for ln in open("/proc/cpuinfo"):
            key = ln.lower()
            if key.startswith("model name"):
                return ln.split(":", 1)[1].strip()
            if key.startswith("cpu part") and part is None:
                part = ln.split(":", 1)[1].strip().lower()
        if part is not None:
            return _ARM_PARTS.get(part, f"Arm part {part}")
    except Exception:
        pass
    import platform
    return platform.machine()


def main(argv=None):
    args = parse_args(argv)
    w = workload_of(args)
    if isinstance(w, W.PrefillWorkload):
        arms = (run_prefill_reference, run_prefill)
    elif isinstance(w, W.ForkWorkload):
        arms = (run_fork_reference, run_fork)
    elif isinstance(w, W.SwapWorkload):
        arms = (run_swap_reference, run_swap)
    else:
        arms = (run_reference, run_ours)
    arms[0 if args.impl == "reference" else 1](args)


if __name__ == "__main__":
    main()
