"""Oracle for the host block pool: FIFO free list, refcounts, block tables, slots.

TEST INFRASTRUCTURE ONLY (see ``oracle/__init__``).

Follows "LLM inference tutorial" (xurj.top Tutorial/Detail/167):

* section 4.2, ``PagedKVCache.__init__``: the physical pool is a tensor
  ``[num_layers, 2, num_blocks, block_size, num_kv_heads, head_dim]`` and the
  free list starts as ``0 .. num_blocks-1``;
* section 4.2, ``allocate_sequence``: a new sequence takes the FRONT of the free
  list at once (FIFO ``pop(0)``) and starts with length 0; an empty free list
  is an error;
* section 4.2, ``append_token``: the token at position ``n`` lives in logical
  block ``n // block_size`` at offset ``n % block_size``; a new block is taken
  from the front of the free list when that logical block is not yet in the
  table;
* section 4.2, ``free_sequence``: the sequence's blocks go to the TAIL of the
  free list in table order;
* section 4.2, ``memory_usage``: used = total - free, utilisation in percent,
  GB = bytes / 1e9 with per-layer block bytes times the layer count;
* section 4.3, ``PrefixCacheManager``: shared prefixes are counted by
  reference; this oracle keeps the count per physical block and frees a block
  when its count reaches zero (the page leaves "keep or free" open at zero;
  freeing is the reading taken);
* "nano-vLLM architecture", section 4.3: ``block_bytes = 2 * num_layers *
  block_size * num_kv_heads * head_dim * dtype_size`` and ``available_blocks =
  free_memory // block_bytes``.

Plain Python: a ``collections.deque`` free list, dicts for tables and lengths.
"""
from __future__ import annotations

from collections import deque
from dataclasses import dataclass, field

# Status names mirror the C ABI's error classes so replays can compare outcomes.
OK = "ok"
INVALID_ARG = "invalid_arg"
NO_FREE_BLOCK = "no_free_block"
BAD_BLOCK = "bad_block"
REFCOUNT = "refcount"

DTYPE_BYTES = {"f32": 4, "bf16": 2, "fp8_e4m3": 1}


class PoolError(Exception):
    """Raised with one of the status names above."""

    def __init__(self, status: str, msg: str = ""):
        super().__init__(f"{status}: {msg}")
        self.status = status


def block_bytes(num_layers: int, block_size: int, num_kv_heads: int, head_dim: int,
                dtype_size: int) -> int:
    """Bytes of one physical block across all layers, K and V.

    "nano-vLLM architecture", section 4.3 memory-pool formula.
    """
    return 2 * num_layers * block_size * num_kv_heads * head_dim * dtype_size


def available_blocks(free_memory: int, bytes_per_block: int) -> int:
    """"nano-vLLM architecture", section 4.3: free_memory // block_bytes."""
    return free_memory // bytes_per_block


@dataclass
class Pool:
    """Host-side pool state: free list, refcounts, tables and lengths."""

    num_layers: int
    num_kv_heads: int
    head_dim: int
    block_size: int
    dtype_size: int
    num_blocks: int
    initial_free_order: list[int] | None = None
    free: deque = field(init=False)
    ref: list[int] = field(init=False)
    tables: dict = field(init=False, default_factory=dict)
    lens: dict = field(init=False, default_factory=dict)

    def __post_init__(self):
        if self.num_blocks <= 0 or self.block_size <= 0:
            raise PoolError(INVALID_ARG, "num_blocks and block_size must be > 0")
        order = (list(range(self.num_blocks)) if self.initial_free_order is None
                 else [int(b) for b in self.initial_free_order])
        if sorted(order) != list(range(self.num_blocks)):
            raise PoolError(INVALID_ARG, "initial_free_order is not a permutation")
        self.free = deque(order)
        self.ref = [0] * self.num_blocks
        self.tables = {}
        self.lens = {}

    # -- blocks (section 4.2 free list, section 4.3 reference counts) --------
    def block_alloc(self) -> int:
        if not self.free:
            raise PoolError(NO_FREE_BLOCK, "free list empty")
        b = self.free.popleft()
        self.ref[b] = 1
        return b

    def _check_id(self, b: int):
        if not (0 <= b < self.num_blocks):
            raise PoolError(BAD_BLOCK, f"block id {b} out of range")

    def block_ref(self, b: int):
        self._check_id(b)
        if self.ref[b] <= 0:
            raise PoolError(REFCOUNT, f"block {b} is free")
        self.ref[b] += 1

    def block_free(self, b: int):
        self._check_id(b)
        if self.ref[b] <= 0:
            raise PoolError(REFCOUNT, f"block {b} already free")
        self.ref[b] -= 1
        if self.ref[b] == 0:
            self.free.append(b)

    # -- sequences (section 4.2 allocate_sequence / append_token / free) -----
    def seq_create(self, sid: int):
        if sid in self.tables:
            raise PoolError(INVALID_ARG, f"sequence {sid} exists")
        b = self.block_alloc()
        self.tables[sid] = [b]
        self.lens[sid] = 0

    def seq_fork_prefix(self, dst: int, src: int, ntok: int):
        """New sequence ``dst`` sharing the first ``ntok`` tokens of ``src``.

        Only whole blocks are shared (``ntok`` a multiple of the block size),
        so the next token of ``dst`` opens a private block and no block is
        ever written through two tables (copy-on-write is not needed).
        """
        if dst in self.tables or src not in self.tables:
            raise PoolError(INVALID_ARG, "bad fork ids")
        if ntok <= 0 or ntok % self.block_size or ntok > self.lens[src]:
            raise PoolError(INVALID_ARG, "fork length must be whole blocks of src")
        shared = self.tables[src][: ntok // self.block_size]
        for b in shared:
            self.block_ref(b)
        self.tables[dst] = list(shared)
        self.lens[dst] = ntok

    def _needs_block(self, sid: int, extra: int) -> bool:
        n = self.lens[sid] + extra
        return n // self.block_size >= len(self.tables[sid])

    def _append_one(self, sid: int) -> int:
        n = self.lens[sid]
        blk, off = divmod(n, self.block_size)
        if blk >= len(self.tables[sid]):
            self.tables[sid].append(self.block_alloc())
        slot = self.tables[sid][blk] * self.block_size + off
        self.lens[sid] = n + 1
        return slot

    def seq_append_slots(self, sids: list[int]) -> list[int]:
        """Append one token to each listed sequence; return the slot of each.

        All-or-nothing: if the free list cannot cover every new block the
        call fails before changing anything.  Repeated ids are refused.
        """
        if len(set(sids)) != len(sids):
            raise PoolError(INVALID_ARG, "repeated sequence id")
        for s in sids:
            if s not in self.tables:
                raise PoolError(INVALID_ARG, f"unknown sequence {s}")
        need = sum(1 for s in sids if self._needs_block(s, 0))
        if need > len(self.free):
            raise PoolError(NO_FREE_BLOCK, f"need {need}, have {len(self.free)}")
        return [self._append_one(s) for s in sids]

    def seq_append_tokens(self, sid: int, n: int) -> list[int]:
        """Append ``n`` tokens to one sequence (a prompt); all-or-nothing."""
        if sid not in self.tables:
            raise PoolError(INVALID_ARG, f"unknown sequence {sid}")
        if n < 0:
            raise PoolError(INVALID_ARG, "negative count")
        have = len(self.tables[sid]) * self.block_size
        need = max(0, -(-(self.lens[sid] + n - have) // self.block_size))
        if need > len(self.free):
            raise PoolError(NO_FREE_BLOCK, f"need {need}, have {len(self.free)}")
        return [self._append_one(sid) for _ in range(n)]

    def seq_free(self, sid: int):
        if sid not in self.tables:
            raise PoolError(INVALID_ARG, f"unknown sequence {sid}")
        for b in self.tables[sid]:
            self.block_free(b)
        del self.tables[sid]
        del self.lens[sid]

    # -- views ----------------------------------------------------------------
    def block_table(self, sid: int) -> list[int]:
        return list(self.tables[sid])

    def padded_tables(self, sids: list[int], max_blocks: int, pad: int = -1):
        """``[len(sids), max_blocks]`` table rows padded with ``pad``, and lens."""
        rows, lens = [], []
        for s in sids:
            t = self.tables[s]
            if len(t) > max_blocks:
                raise PoolError(INVALID_ARG, "table longer than max_blocks")
            rows.append(t + [pad] * (max_blocks - len(t)))
            lens.append(self.lens[s])
        return rows, lens

    def stats(self) -> dict:
        """Section 4.2 ``memory_usage``, with block bytes over all layers."""
        bb = block_bytes(self.num_layers, self.block_size, self.num_kv_heads,
                         self.head_dim, self.dtype_size)
        used = self.num_blocks - len(self.free)
        return {
            "total_blocks": self.num_blocks,
            "used_blocks": used,
            "free_blocks": len(self.free),
            "utilization": used / self.num_blocks * 100.0,
            "block_bytes": bb,
            "total_bytes": self.num_blocks * bb,
            "used_bytes": used * bb,
            "total_memory_gb": self.num_blocks * bb / 1e9,
            "used_memory_gb": used * bb / 1e9,
        }
