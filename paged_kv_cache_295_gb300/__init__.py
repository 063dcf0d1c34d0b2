"""Python binding of libpagedkv (paged KV cache + PagedAttention decode, sm_103a).

Argument marshalling only: every step of the path runs in the C++ pool and the
CUDA kernels of ``libpagedkv.so``; torch provides device memory and the
current stream.  There is no CPU fallback: if the library is missing or the
device is not a CUDA GPU, the calls raise.

Names follow the C ABI in ``include/pagedkv.h``.
"""
from __future__ import annotations

import ctypes as C
import os

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libpagedkv.so")

F32, BF16, FP8_E4M3, INT8 = 0, 1, 2, 3
DTYPE_NAMES = {F32: "f32", BF16: "bf16", FP8_E4M3: "fp8_e4m3", INT8: "int8"}
DEV_BAD_BLOCK, DEV_BAD_SLOT, DEV_BAD_CONTEXT, DEV_TIMEOUT = 0x1, 0x2, 0x4, 0x8

STATUS = {0: "ok", 1: "invalid_arg", 2: "no_free_block", 3: "bad_block", 4: "refcount",
          5: "unsupported", 6: "cuda", 7: "host_memory", 8: "scratch_limit"}
NOALLOC_SCRATCH_BYTES = 16 * 1024 * 1024


class PagedKVError(RuntimeError):
    def __init__(self, code: int, where: str):
        super().__init__(f"{where}: {STATUS.get(code, code)}")
        self.code = code
        self.status = STATUS.get(code, str(code))


class _PoolConfig(C.Structure):
    _fields_ = [("num_layers", C.c_int32), ("num_kv_heads", C.c_int32),
                ("head_dim", C.c_int32), ("block_size", C.c_int32),
                ("kv_dtype", C.c_int32), ("num_blocks", C.c_int64),
                ("free_bytes", C.c_int64), ("initial_free_order", C.POINTER(C.c_int32))]


class _PoolStats(C.Structure):
    _fields_ = [("total_blocks", C.c_int64), ("used_blocks", C.c_int64),
                ("free_blocks", C.c_int64), ("utilization", C.c_double),
                ("block_bytes", C.c_int64), ("total_bytes", C.c_int64),
                ("used_bytes", C.c_int64)]


class _GraphConfig(C.Structure):
    _fields_ = [("num_layers", C.c_int32), ("num_q_heads", C.c_int32),
                ("num_kv_heads", C.c_int32), ("head_dim", C.c_int32),
                ("block_size", C.c_int32), ("num_blocks", C.c_int64),
                ("max_blocks_per_seq", C.c_int32), ("q_dtype", C.c_int32),
                ("kv_dtype", C.c_int32), ("src_dtype", C.c_int32), ("scale", C.c_float),
                ("k_caches", C.POINTER(C.c_void_p)), ("v_caches", C.POINTER(C.c_void_p)),
                ("k_scales", C.POINTER(C.c_void_p)), ("v_scales", C.POINTER(C.c_void_p)),
                ("q", C.c_void_p), ("k_new", C.c_void_p), ("v_new", C.c_void_p),
                ("slot_mapping", C.c_void_p), ("block_tables", C.c_void_p),
                ("context_lens", C.c_void_p), ("out", C.c_void_p), ("workspace", C.c_void_p),
                ("workspace_bytes", C.c_size_t), ("device_status", C.c_void_p),
                ("buckets", C.POINTER(C.c_int32)), ("num_buckets", C.c_int32)]


_lib = None
P, I32, I64, SZ, FL = C.c_void_p, C.c_int32, C.c_int64, C.c_size_t, C.c_float
_SIGS = {
    "pkv_status_string": (C.c_char_p, [I32]),
    "pkv_block_bytes": (I64, [C.POINTER(_PoolConfig)]),
    "kv_pool_init": (I32, [C.POINTER(_PoolConfig), C.POINTER(P)]),
    "kv_pool_destroy": (None, [P]),
    "block_alloc": (I32, [P, C.POINTER(I32)]),
    "block_ref": (I32, [P, I32]),
    "block_free": (I32, [P, I32]),
    "block_refcount": (I32, [P, I32, C.POINTER(I32)]),
    "kv_pool_stats": (I32, [P, C.POINTER(_PoolStats)]),
    "kv_pool_free_list": (I32, [P, P, I64, C.POINTER(I64)]),
    "seq_create": (I32, [P, I64]),
    "seq_fork_prefix": (I32, [P, I64, I64, I32]),
    "seq_append_slots": (I32, [P, P, I32, P]),
    "seq_append_tokens": (I32, [P, I64, I32, P]),
    "seq_length": (I32, [P, I64, C.POINTER(I32)]),
    "seq_block_table": (I32, [P, I64, P, I32, C.POINTER(I32)]),
    "seq_batch_tables": (I32, [P, P, I32, I32, P, P]),
    "seq_free": (I32, [P, I64]),
    "pool_take_copies": (I32, [P, P, I32, C.POINTER(I32)]),
    "prefix_cache_insert": (I32, [P, P, I32, I64]),
    "prefix_cache_lookup": (I32, [P, P, I32, C.POINTER(I32), P, I32, C.POINTER(I32)]),
    "seq_create_from_prefix": (I32, [P, I64, P, I32, C.POINTER(I32)]),
    "prefix_cache_release": (I32, [P, P, I32]),
    "prefix_cache_count": (I32, [P, P, I32, C.POINTER(I32)]),
    "copy_blocks": (I32, [P, I32, I64, I64, I64, P, I32, P, P]),
    "kv_pool_host_init": (I32, [P, I64]),
    "pool_lru_order": (I32, [P, P, I64, C.POINTER(I64)]),
    "seq_swap_out": (I32, [P, I64, P, I32, C.POINTER(I32)]),
    "seq_swap_in": (I32, [P, I64, P, I32, C.POINTER(I32)]),
    "seq_is_swapped": (I32, [P, I64, C.POINTER(I32)]),
    "swap_blocks": (I32, [P, I32, I64, I64, I64, P, I64, P, I32, I32, P, P]),
    "decode_graph_create": (I32, [C.POINTER(_GraphConfig), C.POINTER(P)]),
    "decode_graph_launch": (I32, [P, I32, C.POINTER(I32), P]),
    "decode_graph_destroy": (None, [P]),
    "decode_graph_step_host": (I32, [P, P, P, I32, P, P, P, P, P, P]),
    "reshape_and_cache": (I32, [P, P, P, P, P, I32, I32, I32, I32, I64, I32, I32, P, P, P, P]),
    "paged_attention_partition_tokens": (I32, [I32, I32, I32, I32, I32]),
    "paged_attention_workspace_bytes": (SZ, [I32, I32, I32, I32, I32, I32]),
    "paged_attention_decode": (I32, [P, P, P, P, P, I32, I32, I32, I32, I32, I64, I32, I32, FL,
                                     I32, I32, P, P, P, P, SZ, I32, P, P]),
    "paged_attention_decode_append": (I32, [P, P, P, P, I32, P, P, P, P, I32, I32, I32, I32, I32,
                                            I64, I32, I32, FL, I32, I32, P, P, P, P, SZ, I32, P,
                                            P]),
    "paged_attention_decode_noalloc": (I32, [P, P, P, P, P, I32, I32, I32, I32, I32, I64, I32,
                                             I32, FL, I32, I32, P, P, P, I32, P, P]),
    "paged_attention_prefill": (I32, [P, P, P, P, P, P, I32, I32, I32, I32, I32, I32, I32, I64,
                                      I32, I32, FL, I32, I32, I32, P, P, P, P, P]),
    "pkv_test_force_decode_kernel": (I32, [I32]),
    "pkv_test_decode_stall": (I32, [C.c_uint32]),
    "pkv_copy_kernel": (I32, [P, P, SZ, P]),
    "pkv_read_kernel": (I32, [P, SZ, P, P]),
    "pkv_read_kernel_sink_floats": (I32, []),
}


def library():
    """Load ``libpagedkv.so`` (raises if it has not been built)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"libpagedkv.so not built at {LIB_PATH}: run "
                               "paged_kv_cache_295_gb300._build.build_library()")
        lib = C.CDLL(LIB_PATH)
        for name, (res, args) in _SIGS.items():
            fn = getattr(lib, name)
            fn.restype = res
            fn.argtypes = args
        _lib = lib
    return _lib


def _check(code: int, where: str):
    if code != 0:
        raise PagedKVError(code, where)


def _np_ptr(a: np.ndarray):
    return a.ctypes.data_as(C.c_void_p)


def block_bytes(num_layers, block_size, num_kv_heads, head_dim, kv_dtype=BF16) -> int:
    cfg = _PoolConfig(num_layers, num_kv_heads, head_dim, block_size, kv_dtype, 0, 0, None)
    return int(library().pkv_block_bytes(C.byref(cfg)))


class Pool:
    """Host block pool (C++): FIFO free list, refcounts, tables and slots."""

    def __init__(self, num_layers, num_kv_heads, head_dim, block_size, kv_dtype=BF16,
                 num_blocks=0, free_bytes=0, initial_free_order=None):
        lib = library()
        order = None
        if initial_free_order is not None:
            self._order = np.ascontiguousarray(initial_free_order, dtype=np.int32)
            order = self._order.ctypes.data_as(C.POINTER(C.c_int32))
        cfg = _PoolConfig(num_layers, num_kv_heads, head_dim, block_size, kv_dtype,
                          num_blocks, free_bytes, order)
        h = C.c_void_p()
        _check(lib.kv_pool_init(C.byref(cfg), C.byref(h)), "kv_pool_init")
        self._h = h
        self.block_size = block_size
        self.num_blocks = self.stats()["total_blocks"]

    def close(self):
        if getattr(self, "_h", None):
            library().kv_pool_destroy(self._h)
            self._h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def block_alloc(self) -> int:
        b = C.c_int32()
        _check(library().block_alloc(self._h, C.byref(b)), "block_alloc")
        return b.value

    def block_ref(self, b: int):
        _check(library().block_ref(self._h, b), "block_ref")

    def block_free(self, b: int):
        _check(library().block_free(self._h, b), "block_free")

    def refcount(self, b: int) -> int:
        c = C.c_int32()
        _check(library().block_refcount(self._h, b, C.byref(c)), "block_refcount")
        return c.value

    def stats(self) -> dict:
        s = _PoolStats()
        _check(library().kv_pool_stats(self._h, C.byref(s)), "kv_pool_stats")
        return {f: getattr(s, f) for f, _ in _PoolStats._fields_}

    def free_list(self) -> list:
        n = C.c_int64()
        buf = np.empty(self.num_blocks, dtype=np.int32)
        _check(library().kv_pool_free_list(self._h, _np_ptr(buf), buf.size, C.byref(n)),
               "kv_pool_free_list")
        return buf[: n.value].tolist()

    def seq_create(self, sid: int):
        _check(library().seq_create(self._h, sid), "seq_create")

    def seq_fork_prefix(self, dst: int, src: int, ntok: int):
        _check(library().seq_fork_prefix(self._h, dst, src, ntok), "seq_fork_prefix")

    def append_slots(self, sids) -> np.ndarray:
        ids = np.ascontiguousarray(sids, dtype=np.int64)
        out = np.empty(ids.size, dtype=np.int64)
        _check(library().seq_append_slots(self._h, _np_ptr(ids), ids.size, _np_ptr(out)),
               "seq_append_slots")
        return out

    def append_tokens(self, sid: int, n: int, want_slots: bool = True):
        out = np.empty(n, dtype=np.int64) if want_slots else None
        _check(library().seq_append_tokens(self._h, sid, n,
                                           _np_ptr(out) if want_slots else None),
               "seq_append_tokens")
        return out

    def seq_length(self, sid: int) -> int:
        n = C.c_int32()
        _check(library().seq_length(self._h, sid, C.byref(n)), "seq_length")
        return n.value

    def block_table(self, sid: int) -> list:
        n = C.c_int32()
        st = library().seq_block_table(self._h, sid, None, 0, C.byref(n))
        if st not in (0, 1):
            _check(st, "seq_block_table")
        buf = np.empty(max(n.value, 1), dtype=np.int32)
        _check(library().seq_block_table(self._h, sid, _np_ptr(buf), buf.size, C.byref(n)),
               "seq_block_table")
        return buf[: n.value].tolist()

    def batch_tables(self, sids, max_blocks: int, tables=None, lens=None):
        """``[n, max_blocks]`` int32 tables (pad -1) and ``[n]`` int32 lengths.

        ``tables`` / ``lens`` may be caller-owned contiguous int32 arrays (for
        example views of pinned host tensors) to write into.
        """
        ids = np.ascontiguousarray(sids, dtype=np.int64)
        if tables is None:
            tables = np.empty((ids.size, max_blocks), dtype=np.int32)
        if lens is None:
            lens = np.empty(ids.size, dtype=np.int32)
        if (tables.dtype != np.int32 or lens.dtype != np.int32 or tables.size < ids.size * max_blocks
                or lens.size < ids.size or not tables.flags.c_contiguous
                or not lens.flags.c_contiguous):
            raise ValueError("tables/lens must be contiguous int32 arrays of the batch's size")
        _check(library().seq_batch_tables(self._h, _np_ptr(ids), ids.size, max_blocks,
                                          _np_ptr(tables), _np_ptr(lens)), "seq_batch_tables")
        return tables, lens

    def seq_free(self, sid: int):
        _check(library().seq_free(self._h, sid), "seq_free")

    def take_copies(self) -> np.ndarray:
        """Pending copy-on-write pairs ``[k, 2]`` int32 (source, new block); clears them."""
        n = C.c_int32()
        st = library().pool_take_copies(self._h, None, 0, C.byref(n))
        if st != 0 and n.value == 0:
            _check(st, "pool_take_copies")
        buf = np.empty((max(n.value, 1), 2), dtype=np.int32)
        _check(library().pool_take_copies(self._h, _np_ptr(buf), buf.shape[0], C.byref(n)),
               "pool_take_copies")
        return buf[: n.value]

    def host_init(self, num_host_blocks: int):
        _check(library().kv_pool_host_init(self._h, int(num_host_blocks)), "kv_pool_host_init")

    def lru_order(self) -> list:
        n = C.c_int64()
        st = library().pool_lru_order(self._h, None, 0, C.byref(n))
        if st != 0 and n.value == 0:
            _check(st, "pool_lru_order")
        buf = np.empty(max(n.value, 1), dtype=np.int64)
        _check(library().pool_lru_order(self._h, _np_ptr(buf), buf.size, C.byref(n)),
               "pool_lru_order")
        return buf[: n.value].tolist()

    def _swap(self, fn, sid, where):
        n = C.c_int32()
        cap = max(len(self.block_table(sid)), 1)   # at most one pair per table entry
        buf = np.empty((cap, 2), dtype=np.int32)
        _check(fn(self._h, sid, _np_ptr(buf), cap, C.byref(n)), where)
        return buf[: n.value]

    def swap_out(self, sid: int) -> np.ndarray:
        """(device block, host slot) pairs ``[k, 2]`` of the sequence's private blocks."""
        return self._swap(library().seq_swap_out, sid, "seq_swap_out")

    def swap_in(self, sid: int) -> np.ndarray:
        """(host slot, device block) pairs ``[k, 2]``."""
        return self._swap(library().seq_swap_in, sid, "seq_swap_in")

    def is_swapped(self, sid: int) -> bool:
        v = C.c_int32()
        _check(library().seq_is_swapped(self._h, sid, C.byref(v)), "seq_is_swapped")
        return bool(v.value)

    @staticmethod
    def _tokens(tokens):
        t = np.ascontiguousarray(tokens, dtype=np.int32)
        return t, (_np_ptr(t) if t.size else None)

    def prefix_insert(self, tokens, sid: int):
        t, ptr = self._tokens(tokens)
        _check(library().prefix_cache_insert(self._h, ptr, t.size, sid), "prefix_cache_insert")

    def prefix_lookup(self, tokens):
        """(matched length, blocks) of the longest cached prefix; a hit counts."""
        t, ptr = self._tokens(tokens)
        m, nb = C.c_int32(), C.c_int32()
        buf = np.empty(max(1, -(-t.size // self.block_size)), dtype=np.int32)
        _check(library().prefix_cache_lookup(self._h, ptr, t.size, C.byref(m), _np_ptr(buf),
                                             buf.size, C.byref(nb)), "prefix_cache_lookup")
        return m.value, buf[: nb.value].tolist()

    def seq_create_from_prefix(self, sid: int, tokens) -> int:
        t, ptr = self._tokens(tokens)
        m = C.c_int32()
        _check(library().seq_create_from_prefix(self._h, sid, ptr, t.size, C.byref(m)),
               "seq_create_from_prefix")
        return m.value

    def prefix_release(self, tokens):
        t, ptr = self._tokens(tokens)
        _check(library().prefix_cache_release(self._h, ptr, t.size), "prefix_cache_release")

    def prefix_count(self, tokens) -> int:
        t, ptr = self._tokens(tokens)
        c = C.c_int32()
        _check(library().prefix_cache_count(self._h, ptr, t.size, C.byref(c)),
               "prefix_cache_count")
        return c.value


# ---------------------------------------------------------------------------
# Device calls (torch tensors in, async on the current stream).
# ---------------------------------------------------------------------------
def _torch():
    import torch
    return torch


def _dtype_code(t) -> int:
    torch = _torch()
    if t.dtype == torch.float32:
        return F32
    if t.dtype == torch.bfloat16:
        return BF16
    if t.dtype in (torch.uint8, torch.float8_e4m3fn):
        return FP8_E4M3
    if t.dtype == torch.int8:
        return INT8
    raise TypeError(f"unsupported dtype {t.dtype}")


def _dev(t, name):
    if t is None:
        return None
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor (no CPU path)")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    return C.c_void_p(t.data_ptr())


def _stream(stream):
    torch = _torch()
    s = stream if stream is not None else torch.cuda.current_stream()
    return C.c_void_p(s.cuda_stream)


def reshape_and_cache(k_new, v_new, slot_mapping, k_cache, v_cache, k_scale=None,
                      v_scale=None, device_status=None, stream=None):
    """Append token rows ``[T, Hkv, D]`` into one layer's ``[NB, bs, Hkv, D]`` cache."""
    T, hkv, d = k_new.shape
    nb, bs = k_cache.shape[0], k_cache.shape[1]
    st = library().reshape_and_cache(
        _dev(k_new, "k_new"), _dev(v_new, "v_new"), _dev(slot_mapping, "slot_mapping"),
        _dev(k_cache, "k_cache"), _dev(v_cache, "v_cache"), T, hkv, d, bs, nb,
        _dtype_code(k_new), _dtype_code(k_cache), _dev(k_scale, "k_scale"),
        _dev(v_scale, "v_scale"), _dev(device_status, "device_status"), _stream(stream))
    _check(st, "reshape_and_cache")


def partition_tokens(num_seqs, num_q_heads, num_kv_heads, max_context_len, requested=0) -> int:
    return int(library().paged_attention_partition_tokens(num_seqs, num_q_heads, num_kv_heads,
                                                           max_context_len, requested))


def workspace_bytes(num_seqs, num_q_heads, num_kv_heads, head_dim, max_context_len,
                    partition=0) -> int:
    return int(library().paged_attention_workspace_bytes(num_seqs, num_q_heads, num_kv_heads,
                                                         head_dim, max_context_len, partition))


DECODE_KERNELS = {"auto": 0, "mma": 1, "simt": 2}


def force_decode_kernel(name: str = "auto"):
    """Tests and profiles: make later decode calls skip to the heads-as-rows
    mma.sync kernel ("mma") or the CUDA-core kernel ("simt") where it supports
    the shape; "auto" restores the choice by shape (pkv_test_force_decode_kernel)."""
    _check(library().pkv_test_force_decode_kernel(DECODE_KERNELS[name]),
           "pkv_test_force_decode_kernel")


def stall_decode_for_test(nbytes: int = 0):
    """Tests of the bounded waits: later launches of the transposed decode
    kernel wait in vain for ``nbytes`` on one barrier phase (0 = normal)."""
    _check(library().pkv_test_decode_stall(int(nbytes)), "pkv_test_decode_stall")


def paged_attention_decode(q, k_cache, v_cache, block_tables, context_lens, scale,
                           max_context_len, out=None, k_scale=None, v_scale=None,
                           workspace=None, partition=0, device_status=None, stream=None):
    """Decode attention; returns ``out [S, Hq, D]`` float32 (allocated if None).

    ``max_context_len`` is a host int (an upper bound of ``context_lens``).
    The split-KV workspace is allocated with torch when not given.
    """
    torch = _torch()
    S, hq, d = q.shape
    nb, bs, hkv, _ = k_cache.shape
    mb = block_tables.shape[1]
    if out is None:
        out = torch.empty((S, hq, d), dtype=torch.float32, device=q.device)
    need = workspace_bytes(S, hq, hkv, d, max_context_len, partition)
    if need and (workspace is None or workspace.numel() * workspace.element_size() < need):
        workspace = torch.empty(need, dtype=torch.uint8, device=q.device)
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    st = library().paged_attention_decode(
        _dev(q, "q"), _dev(k_cache, "k_cache"), _dev(v_cache, "v_cache"),
        _dev(block_tables, "block_tables"), _dev(context_lens, "context_lens"), S, hq, hkv, d,
        bs, nb, mb, int(max_context_len), float(scale), _dtype_code(q), _dtype_code(k_cache),
        _dev(k_scale, "k_scale"), _dev(v_scale, "v_scale"), _dev(out, "out"),
        _dev(workspace, "workspace") if workspace is not None else None, ws_bytes,
        int(partition), _dev(device_status, "device_status"), _stream(stream))
    _check(st, "paged_attention_decode")
    return out


def paged_attention_decode_append(q, k_new, v_new, slot_mapping, k_cache, v_cache, block_tables,
                                  context_lens, scale, max_context_len, out=None, k_scale=None,
                                  v_scale=None, workspace=None, partition=0, device_status=None,
                                  stream=None):
    """``reshape_and_cache`` of one new token per sequence (``k_new`` / ``v_new``
    ``[S, Hkv, D]``, ``slot_mapping`` int64 ``[S]``, each the slot of position
    ``context_lens[s] - 1``) and ``paged_attention_decode``, as one call."""
    torch = _torch()
    S, hq, d = q.shape
    nb, bs, hkv, _ = k_cache.shape
    mb = block_tables.shape[1]
    if out is None:
        out = torch.empty((S, hq, d), dtype=torch.float32, device=q.device)
    need = workspace_bytes(S, hq, hkv, d, max_context_len, partition)
    if need and (workspace is None or workspace.numel() * workspace.element_size() < need):
        workspace = torch.empty(need, dtype=torch.uint8, device=q.device)
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    st = library().paged_attention_decode_append(
        _dev(q, "q"), _dev(k_new, "k_new"), _dev(v_new, "v_new"),
        _dev(slot_mapping, "slot_mapping"), _dtype_code(k_new), _dev(k_cache, "k_cache"),
        _dev(v_cache, "v_cache"), _dev(block_tables, "block_tables"),
        _dev(context_lens, "context_lens"), S, hq, hkv, d, bs, nb, mb, int(max_context_len),
        float(scale), _dtype_code(q), _dtype_code(k_cache), _dev(k_scale, "k_scale"),
        _dev(v_scale, "v_scale"), _dev(out, "out"),
        _dev(workspace, "workspace") if workspace is not None else None, ws_bytes,
        int(partition), _dev(device_status, "device_status"), _stream(stream))
    _check(st, "paged_attention_decode_append")
    return out


def paged_attention_decode_noalloc(q, k_cache, v_cache, block_tables, context_lens, scale,
                                   max_context_len, out, k_scale=None, v_scale=None, partition=0,
                                   device_status=None, stream=None):
    """``paged_attention_decode`` into a caller-owned ``out`` with the library's
    built-in split-KV scratch (no device allocation by the library or here)."""
    S, hq, d = q.shape
    nb, bs, hkv, _ = k_cache.shape
    st = library().paged_attention_decode_noalloc(
        _dev(q, "q"), _dev(k_cache, "k_cache"), _dev(v_cache, "v_cache"),
        _dev(block_tables, "block_tables"), _dev(context_lens, "context_lens"), S, hq, hkv, d,
        bs, nb, block_tables.shape[1], int(max_context_len), float(scale), _dtype_code(q),
        _dtype_code(k_cache), _dev(k_scale, "k_scale"), _dev(v_scale, "v_scale"),
        _dev(out, "out"), int(partition), _dev(device_status, "device_status"), _stream(stream))
    _check(st, "paged_attention_decode_noalloc")
    return out


def paged_attention_prefill(q, query_start, k_cache, v_cache, block_tables, context_lens,
                            scale, max_query_len, max_context_len, causal=True, out=None,
                            k_scale=None, v_scale=None, device_status=None, stream=None):
    """Chunked prefill attention; returns ``out [T, Hq, D]`` float32 (allocated
    if None).  ``query_start`` is int32 ``[S + 1]`` on the device;
    ``max_query_len`` and ``max_context_len`` are host ints (upper bounds);
    ``k_scale`` / ``v_scale`` (``[Hkv]`` float32) for an FP8 cache."""
    torch = _torch()
    T, hq, d = q.shape
    nb, bs, hkv, _ = k_cache.shape
    S = query_start.shape[0] - 1
    if out is None:
        out = torch.empty((T, hq, d), dtype=torch.float32, device=q.device)
    st = library().paged_attention_prefill(
        _dev(q, "q"), _dev(query_start, "query_start"), _dev(k_cache, "k_cache"),
        _dev(v_cache, "v_cache"), _dev(block_tables, "block_tables"),
        _dev(context_lens, "context_lens"), S, T, int(max_query_len), hq, hkv, d, bs, nb,
        block_tables.shape[1], int(max_context_len), float(scale), 1 if causal else 0,
        _dtype_code(q), _dtype_code(k_cache), _dev(k_scale, "k_scale"), _dev(v_scale, "v_scale"),
        _dev(out, "out"), _dev(device_status, "device_status"), _stream(stream))
    _check(st, "paged_attention_prefill")
    return out


def copy_blocks(pool_tensor, pairs, device_status=None, stream=None):
    """Copy-on-write copies on the pool tensor ``[L, 2, NB, bs, Hkv, D]``:
    ``pairs`` is a device int32 ``[k, 2]`` of (source, destination) blocks."""
    L, two, nb = pool_tensor.shape[:3]
    plane = pool_tensor[0, 0]
    bb = plane[0].numel() * plane.element_size()
    k = pairs.shape[0] if pairs.dim() else 0
    st = library().copy_blocks(_dev(pool_tensor, "pool"), L * two, nb * bb, bb, nb,
                               _dev(pairs, "pairs") if k else None, k,
                               _dev(device_status, "device_status"), _stream(stream))
    _check(st, "copy_blocks")


class DecodeGraph:
    """A decode step (every layer: append + attention) captured as one CUDA
    graph per batch-size bucket over fixed device buffers, replayed with the
    batch padded to the nearest larger bucket.

    ``engine`` is a ``PagedKVCache``; the buffers are allocated here for the
    largest bucket: ``q [L, Bmax, Hq, D]``, ``k_new``/``v_new [L, Bmax, Hkv,
    D]``, ``slots [Bmax]``, ``tables [Bmax, max_blocks]``, ``lens [Bmax]``,
    ``out [L, Bmax, Hq, D]``.  Fill the first ``batch`` rows, call
    ``launch(batch)``, read ``out[:, :batch]``.
    """

    def __init__(self, engine, num_q_heads, max_blocks, buckets, q_dtype=None, src_dtype=None,
                 device_status=None):
        torch = _torch()
        e = engine
        dev = e.storage.device
        self.buckets = sorted(int(b) for b in buckets)
        B, L = self.buckets[-1], e.num_layers
        hq, hkv, d = num_q_heads, e.num_kv_heads, e.head_dim
        q_dtype = torch.bfloat16 if q_dtype is None else q_dtype
        if src_dtype is None:
            src_dtype = torch.float32 if e.kv_dtype == F32 else torch.bfloat16
        self.q = torch.zeros((L, B, hq, d), dtype=q_dtype, device=dev)
        self.k_new = torch.zeros((L, B, hkv, d), dtype=src_dtype, device=dev)
        self.v_new = torch.zeros_like(self.k_new)
        self.slots = torch.full((B,), -1, dtype=torch.int64, device=dev)
        self.tables = torch.full((B, max_blocks), -1, dtype=torch.int32, device=dev)
        self.lens = torch.zeros((B,), dtype=torch.int32, device=dev)
        self.out = torch.zeros((L, B, hq, d), dtype=torch.float32, device=dev)
        max_ctx = max_blocks * e.block_size
        need = workspace_bytes(B, hq, hkv, d, max_ctx, 0)
        self.ws = torch.empty(max(need, 16), dtype=torch.uint8, device=dev)
        self.status = device_status
        kp = (C.c_void_p * L)(*[e.k_cache(l).data_ptr() for l in range(L)])
        vp = (C.c_void_p * L)(*[e.v_cache(l).data_ptr() for l in range(L)])
        ksp = vsp = None
        if e.k_scale is not None:
            ksp = (C.c_void_p * L)(*[e.k_scale[l].data_ptr() for l in range(L)])
            vsp = (C.c_void_p * L)(*[e.v_scale[l].data_ptr() for l in range(L)])
        bk = (C.c_int32 * len(self.buckets))(*self.buckets)
        self._keep = (kp, vp, ksp, vsp, bk, e)
        cfg = _GraphConfig(
            L, hq, hkv, d, e.block_size, e.num_blocks, max_blocks,
            _dtype_code(self.q), e.kv_dtype, _dtype_code(self.k_new), float(e.scale),
            C.cast(kp, C.POINTER(C.c_void_p)), C.cast(vp, C.POINTER(C.c_void_p)),
            C.cast(ksp, C.POINTER(C.c_void_p)) if ksp else None,
            C.cast(vsp, C.POINTER(C.c_void_p)) if vsp else None,
            self.q.data_ptr(), self.k_new.data_ptr(), self.v_new.data_ptr(),
            self.slots.data_ptr(), self.tables.data_ptr(), self.lens.data_ptr(),
            self.out.data_ptr(), self.ws.data_ptr(), self.ws.numel(),
            device_status.data_ptr() if device_status is not None else None,
            C.cast(bk, C.POINTER(C.c_int32)), len(self.buckets))
        h = C.c_void_p()
        _check(library().decode_graph_create(C.byref(cfg), C.byref(h)), "decode_graph_create")
        self._h = h

    def launch(self, batch, stream=None) -> int:
        """Replay the step for ``batch`` rows; returns the bucket used."""
        b = C.c_int32()
        _check(library().decode_graph_launch(self._h, int(batch), C.byref(b), _stream(stream)),
               "decode_graph_launch")
        return b.value

    def step_host(self, pool, seq_ids, q_host, k_new_host, v_new_host, slots_host, out_host,
                  stream=None):
        """The whole step from host memory (``decode_graph_step_host``): tables
        from ``pool``, host inputs ``q [L, B, Hq, D]``, ``k/v [L, B, Hkv, D]``,
        ``slots [B]`` copied in, the replay, ``out [L, B, Hq, D]`` copied back.
        Host tensors should be pinned; returns when the output is in host memory."""
        ids = np.ascontiguousarray(seq_ids, dtype=np.int64)
        for t, name in ((q_host, "q"), (k_new_host, "k_new"), (v_new_host, "v_new"),
                        (slots_host, "slots"), (out_host, "out")):
            if t.is_cuda or not t.is_contiguous():
                raise ValueError(f"{name} must be a contiguous host tensor")
        st = library().decode_graph_step_host(
            self._h, pool._h, _np_ptr(ids), ids.size, C.c_void_p(q_host.data_ptr()),
            C.c_void_p(k_new_host.data_ptr()), C.c_void_p(v_new_host.data_ptr()),
            C.c_void_p(slots_host.data_ptr()), C.c_void_p(out_host.data_ptr()), _stream(stream))
        _check(st, "decode_graph_step_host")

    def close(self):
        if getattr(self, "_h", None):
            library().decode_graph_destroy(self._h)
            self._h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


def swap_blocks(pool_tensor, host_tensor, pairs, to_host, device_status=None, stream=None):
    """Block copies between the pool tensor ``[L, 2, NB, bs, Hkv, D]`` and a
    pinned host tensor ``[H, L, 2, bs, Hkv, D]``; ``pairs`` device int32
    ``[k, 2]`` ((device, host) to host, (host, device) back)."""
    L, two, nb = pool_tensor.shape[:3]
    plane = pool_tensor[0, 0]
    bb = plane[0].numel() * plane.element_size()
    if not host_tensor.is_pinned():
        raise ValueError("host_tensor must be page-locked (pin_memory)")
    k = pairs.shape[0] if pairs.dim() else 0
    st = library().swap_blocks(_dev(pool_tensor, "pool"), L * two, nb * bb, bb, nb,
                               C.c_void_p(host_tensor.data_ptr()), host_tensor.shape[0],
                               _dev(pairs, "pairs") if k else None, k, 1 if to_host else 0,
                               _dev(device_status, "device_status"), _stream(stream))
    _check(st, "swap_blocks")


def copy_kernel(src, dst, stream=None):
    n = src.numel() * src.element_size()
    _check(library().pkv_copy_kernel(_dev(src, "src"), _dev(dst, "dst"), n, _stream(stream)),
           "pkv_copy_kernel")


def read_kernel(src, sink, stream=None):
    n = src.numel() * src.element_size()
    _check(library().pkv_read_kernel(_dev(src, "src"), n, _dev(sink, "sink"), _stream(stream)),
           "pkv_read_kernel")


def read_kernel_sink_floats() -> int:
    return int(library().pkv_read_kernel_sink_floats())
