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
* section 4.2, the class docstring: copy-on-write for beam search.  A fork
  shares the source's blocks, including a partly filled last block; the first
  write into a block whose count is above one first moves the writer to a
  fresh block (front of the free list) and records (old, new) in a list of
  pending block copies, which the caller executes on the device before it
  writes the token (``take_copies``);
* section 4.3, ``PrefixCacheManager``: ``cache_prefix`` remembers the blocks of
  a token prefix with count 1 (here the cache also holds one reference on each
  of those blocks, so they outlive the sequence that wrote them);
  ``get_cached_prefix`` tries the query's prefixes from the longest down and a
  hit adds one to the count; ``release_prefix`` takes one off, and at zero the
  entry is dropped together with its block references (the "free" reading of
  the page's "keep or free").  Entries are keyed by the token tuple itself, so
  there are no hash collisions to resolve;
* "ToPG framework", section 2.3: pages managed by an LRU policy, so contexts
  can outgrow device memory.  Reading taken (the policy is not spelled out):
  the pool orders resident sequences by their last append (least recently
  used first, ties by id); a sequence swapped out moves its private blocks
  (count 1) to host slots taken from a FIFO host free list, its shared blocks
  stay on the device, and it takes no appends, forks or batch views until it
  is swapped back in, when each host block gets a device block from the
  free-list front.  Each swap returns the (source, destination) pairs the
  caller copies on the device;
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

DTYPE_BYTES = {"f32": 4, "bf16": 2, "fp8_e4m3": 1, "int8": 1}


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
    copies: list = field(init=False, default_factory=list)
    prefix: dict = field(init=False, default_factory=dict)
    host_free: deque = field(init=False, default_factory=deque)
    host_blocks: int = field(init=False, default=0)
    on_host: dict = field(init=False, default_factory=dict)      # sid -> set of table indices
    last_use: dict = field(init=False, default_factory=dict)
    clock: int = field(init=False, default=0)

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
        self.copies = []
        self.prefix = {}
        self.host_free = deque()
        self.host_blocks = 0
        self.on_host = {}
        self.last_use = {}
        self.clock = 0

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
    def _touch(self, sid: int):
        self.clock += 1
        self.last_use[sid] = self.clock

    def _resident(self, sid: int):
        if sid not in self.tables:
            raise PoolError(INVALID_ARG, f"unknown sequence {sid}")
        if sid in self.on_host:
            raise PoolError(INVALID_ARG, f"sequence {sid} is swapped out")

    def seq_create(self, sid: int):
        if sid in self.tables:
            raise PoolError(INVALID_ARG, f"sequence {sid} exists")
        b = self.block_alloc()
        self.tables[sid] = [b]
        self.lens[sid] = 0
        self._touch(sid)

    def seq_fork_prefix(self, dst: int, src: int, ntok: int):
        """New sequence ``dst`` sharing the first ``ntok`` tokens of ``src``.

        The ``ceil(ntok / block_size)`` blocks holding them gain a reference;
        a partly filled last block is shared too and copied on the first
        write into it (by either sequence).  ``ntok == len(src)`` is a full
        fork (a beam).
        """
        if dst in self.tables or src not in self.tables or src in self.on_host:
            raise PoolError(INVALID_ARG, "bad fork ids")
        if ntok <= 0 or ntok > self.lens[src]:
            raise PoolError(INVALID_ARG, "fork length must be 1 .. len(src)")
        shared = self.tables[src][: -(-ntok // self.block_size)]
        for b in shared:
            self.block_ref(b)
        self.tables[dst] = list(shared)
        self.lens[dst] = ntok
        self._touch(dst)

    def _shared_target(self, sid: int) -> bool:
        """The block the next token of ``sid`` goes to exists and is shared."""
        blk = self.lens[sid] // self.block_size
        t = self.tables[sid]
        return blk < len(t) and self.ref[t[blk]] > 1

    def _needs_block(self, sid: int, extra: int) -> bool:
        n = self.lens[sid] + extra
        return n // self.block_size >= len(self.tables[sid]) or (
            extra == 0 and self._shared_target(sid))

    def _append_one(self, sid: int) -> int:
        n = self.lens[sid]
        blk, off = divmod(n, self.block_size)
        t = self.tables[sid]
        if blk >= len(t):
            t.append(self.block_alloc())
        elif self.ref[t[blk]] > 1:          # copy-on-write
            new = self.block_alloc()
            self.copies.append((t[blk], new))
            self.block_free(t[blk])
            t[blk] = new
        slot = t[blk] * self.block_size + off
        self.lens[sid] = n + 1
        return slot

    def seq_append_slots(self, sids: list[int]) -> list[int]:
        """Append one token to each listed sequence; return the slot of each.

        All-or-nothing: if the free list cannot cover every new or
        copied-on-write block the call fails before changing anything.
        Repeated ids are refused.
        """
        if len(set(sids)) != len(sids):
            raise PoolError(INVALID_ARG, "repeated sequence id")
        for s in sids:
            self._resident(s)
        need = sum(1 for s in sids if self._needs_block(s, 0))
        if need > len(self.free):
            raise PoolError(NO_FREE_BLOCK, f"need {need}, have {len(self.free)}")
        out = []
        for s in sids:
            out.append(self._append_one(s))
            self._touch(s)
        return out

    def seq_append_tokens(self, sid: int, n: int) -> list[int]:
        """Append ``n`` tokens to one sequence (a prompt); all-or-nothing."""
        self._resident(sid)
        if n < 0:
            raise PoolError(INVALID_ARG, "negative count")
        have = len(self.tables[sid]) * self.block_size
        need = max(0, -(-(self.lens[sid] + n - have) // self.block_size))
        if n > 0 and self._shared_target(sid):
            need += 1
        if need > len(self.free):
            raise PoolError(NO_FREE_BLOCK, f"need {need}, have {len(self.free)}")
        out = [self._append_one(sid) for _ in range(n)]
        self._touch(sid)
        return out

    def take_copies(self) -> list[tuple[int, int]]:
        """The pending (source block, new block) copies, oldest first; clears them."""
        out, self.copies = self.copies, []
        return out

    # -- prefix cache (section 4.3 PrefixCacheManager) ------------------------
    def prefix_insert(self, tokens, sid: int):
        """``cache_prefix``: the blocks holding ``sid``'s first ``len(tokens)``
        tokens are remembered under ``tokens`` with count 1."""
        key = tuple(int(t) for t in tokens)
        if (sid not in self.tables or sid in self.on_host or not key or len(key) > self.lens[sid]
                or key in self.prefix):
            raise PoolError(INVALID_ARG, "bad prefix insert")
        blocks = self.tables[sid][: -(-len(key) // self.block_size)]
        for b in blocks:
            self.block_ref(b)
        self.prefix[key] = {"blocks": list(blocks), "count": 1}

    def prefix_lookup(self, tokens):
        """``get_cached_prefix``: (blocks, length) of the longest cached prefix
        of ``tokens``, trying lengths from the longest down, or None.  A hit
        adds one to that entry's count."""
        key = tuple(int(t) for t in tokens)
        for length in range(len(key), 0, -1):
            e = self.prefix.get(key[:length])
            if e is not None:
                e["count"] += 1
                return list(e["blocks"]), length
        return None

    def seq_create_from_prefix(self, sid: int, tokens) -> int:
        """New sequence whose first tokens come from the longest cached prefix
        of ``tokens`` (its blocks gain a reference); without a hit, a plain
        ``seq_create``.  Returns the number of tokens taken from the cache."""
        if sid in self.tables:
            raise PoolError(INVALID_ARG, f"sequence {sid} exists")
        hit = self.prefix_lookup(tokens)
        if hit is None:
            self.seq_create(sid)
            return 0
        blocks, length = hit
        for b in blocks:
            self.block_ref(b)
        self.tables[sid] = blocks
        self.lens[sid] = length
        self._touch(sid)
        return length

    def prefix_release(self, tokens):
        """``release_prefix``: one fewer; at zero the entry and its block
        references go."""
        key = tuple(int(t) for t in tokens)
        e = self.prefix.get(key)
        if e is None:
            raise PoolError(INVALID_ARG, "prefix not cached")
        e["count"] -= 1
        if e["count"] == 0:
            del self.prefix[key]
            for b in e["blocks"]:
                self.block_free(b)

    def prefix_count(self, tokens) -> int:
        e = self.prefix.get(tuple(int(t) for t in tokens))
        return 0 if e is None else e["count"]

    def seq_free(self, sid: int):
        if sid not in self.tables:
            raise PoolError(INVALID_ARG, f"unknown sequence {sid}")
        host = self.on_host.pop(sid, set())
        for j, b in enumerate(self.tables[sid]):
            if j in host:
                self.host_free.append(b)
            else:
                self.block_free(b)
        del self.tables[sid]
        del self.lens[sid]
        del self.last_use[sid]

    # -- swap to host memory (ToPG section 2.3, LRU) ---------------------------
    def host_init(self, num_host_blocks: int):
        """Host swap area of ``num_host_blocks`` block slots, FIFO free list."""
        if self.host_blocks or num_host_blocks <= 0:
            raise PoolError(INVALID_ARG, "host area already set or empty")
        self.host_blocks = num_host_blocks
        self.host_free = deque(range(num_host_blocks))

    def lru_order(self) -> list[int]:
        """Resident sequences, least recently appended first (ties by id)."""
        return sorted((s for s in self.tables if s not in self.on_host),
                      key=lambda s: (self.last_use[s], s))

    def seq_swap_out(self, sid: int) -> list[tuple[int, int]]:
        """Move the sequence's private blocks (count 1) to host slots; returns
        the (device block, host slot) pairs, in table order, for the copy."""
        self._resident(sid)
        priv = [j for j, b in enumerate(self.tables[sid]) if self.ref[b] == 1]
        if len(priv) > len(self.host_free):
            raise PoolError(NO_FREE_BLOCK, f"need {len(priv)} host blocks")
        pairs = []
        t = self.tables[sid]
        for j in priv:
            h = self.host_free.popleft()
            pairs.append((t[j], h))
            self.block_free(t[j])
            t[j] = h
        self.on_host[sid] = set(priv)
        return pairs

    def seq_swap_in(self, sid: int) -> list[tuple[int, int]]:
        """Give every host block of a swapped-out sequence a device block from
        the free-list front; returns the (host slot, device block) pairs."""
        if sid not in self.on_host:
            raise PoolError(INVALID_ARG, f"sequence {sid} is not swapped out")
        host = sorted(self.on_host[sid])
        if len(host) > len(self.free):
            raise PoolError(NO_FREE_BLOCK, f"need {len(host)} device blocks")
        pairs = []
        t = self.tables[sid]
        for j in host:
            b = self.block_alloc()
            pairs.append((t[j], b))
            self.host_free.append(t[j])
            t[j] = b
        del self.on_host[sid]
        self._touch(sid)
        return pairs

    # -- views ----------------------------------------------------------------
    def block_table(self, sid: int) -> list[int]:
        return list(self.tables[sid])

    def padded_tables(self, sids: list[int], max_blocks: int, pad: int = -1):
        """``[len(sids), max_blocks]`` table rows padded with ``pad``, and lens."""
        rows, lens = [], []
        for s in sids:
            self._resident(s)
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
