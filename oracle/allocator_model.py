"""Reference model of the host block allocator -- TEST INFRASTRUCTURE ONLY.

A plain-Python restatement of the block-manager policy, written independently
of the library's C++ allocator, used to check that library's block tables and
refcounts exactly.  Only tests, the smoke check and the benchmark's CPU leg use
it.

What it models:

* A flat pool of ``num_blocks`` physical blocks of ``block_size`` (16) tokens
  and per-sequence block tables mapping logical block j to a physical id
  ("Capítulo 8 -- Gestión de caché KV de nueva generación", section 8.1;
  "PagedAttention y Gestión de KV-Cache", section 2 figure).
* A free list of unused blocks; blocks go back to it when a request ends or is
  cancelled, otherwise memory leaks ("PagedAttention y Gestión de KV-Cache",
  section 4.02, cleanup on cancel).
* A reference count per block, so several sequences can point at one block
  (shared prompts, best-of-n branches) ("Capítulo 8 ...", section 8.1).
* Copy-on-write: a sequence that is about to append into a block it shares
  gets a private copy first ("PagedAttention y Gestión de KV-Cache",
  section 3.01; "KV Cache y PagedAttention", "Cómo PagedAttention soluciona
  esto").

Policy details the pages leave open, and the reading taken:

* The free list is a LIFO stack that initially pops 0, 1, 2, ...; freed blocks
  are pushed and reused first.
* ``alloc(n)`` is all-or-nothing.
* ``free`` / ``incref`` validate the whole request before changing anything.
* COW applies only when the next token falls inside an existing block
  (position % block_size != 0) whose refcount is above 1: a new block is
  allocated, the old one is decref'ed, the table entry is rewritten and the
  pair (old, new) is returned for a device copy of the block contents.
"""
from __future__ import annotations

from collections import Counter


class OutOfBlocks(Exception):
    pass


class InvalidRequest(Exception):
    pass


class AllocatorModel:
    def __init__(self, num_blocks: int, block_size: int = 16):
        if num_blocks <= 0:
            raise InvalidRequest("num_blocks must be positive")
        self.num_blocks = num_blocks
        self.block_size = block_size
        self.refcount = [0] * num_blocks
        # top of the stack is the end of the list: pops give 0, 1, 2, ...
        self.free_stack = list(range(num_blocks - 1, -1, -1))

    # ------------------------------------------------------------ operations
    def alloc(self, n: int) -> list[int]:
        if n < 0:
            raise InvalidRequest("negative count")
        if n > len(self.free_stack):
            raise OutOfBlocks(f"need {n}, have {len(self.free_stack)}")
        ids = []
        for _ in range(n):
            b = self.free_stack.pop()
            self.refcount[b] = 1
            ids.append(b)
        return ids

    def free(self, ids) -> None:
        ids = list(ids)
        for b, c in Counter(ids).items():
            if not (0 <= b < self.num_blocks) or self.refcount[b] < c:
                raise InvalidRequest(f"free of block {b} with refcount "
                                     f"{self.refcount[b] if 0 <= b < self.num_blocks else '-'}")
        for b in ids:
            self.refcount[b] -= 1
            if self.refcount[b] == 0:
                self.free_stack.append(b)

    def incref(self, ids) -> None:
        ids = list(ids)
        for b in ids:
            if not (0 <= b < self.num_blocks) or self.refcount[b] == 0:
                raise InvalidRequest(f"incref of unallocated block {b}")
        for b in ids:
            self.refcount[b] += 1

    def cow_prepare(self, table_row: list[int], ctx_len: int):
        """Make the block that receives token ``ctx_len`` private.

        Returns the (src, dst) pair to copy, or None.  ``table_row`` is
        rewritten in place when a copy is needed.
        """
        j, off = divmod(ctx_len, self.block_size)
        if off == 0:
            return None
        b = table_row[j]
        if self.refcount[b] <= 1:
            return None
        new = self.alloc(1)[0]
        self.refcount[b] -= 1
        table_row[j] = new
        return (b, new)

    # ------------------------------------------------------- prefix cache
    # Prompt hashing in block-size chunks ("Capítulo 8 -- Gestión de caché KV de
    # nueva generación", section 8.3): a request whose leading full blocks are
    # cached points its table at them; blocks are registered after prefill.
    # Reading taken: the cache owns one reference per mapped block; lookups stop
    # at the first miss; eviction removes least-recently-used entries that no
    # request references (ties by lower block id).
    def _prefix_init(self):
        if not hasattr(self, "prefix"):
            self.prefix = {}      # hash -> [block, last_use]
            self.tick = 0
            self.lookups = 0
            self.hits = 0

    def prefix_lookup(self, hashes):
        self._prefix_init()
        self.tick += 1
        self.lookups += len(hashes)
        ids = []
        for h in hashes:
            e = self.prefix.get(int(h))
            if e is None:
                break
            e[1] = self.tick
            self.refcount[e[0]] += 1
            ids.append(e[0])
        self.hits += len(ids)
        return ids

    def prefix_register(self, hashes, ids):
        self._prefix_init()
        for b in ids:
            if not (0 <= b < self.num_blocks) or self.refcount[b] == 0:
                raise InvalidRequest(f"register of unallocated block {b}")
        self.tick += 1
        for h, b in zip(hashes, ids):
            if int(h) in self.prefix:
                continue
            self.prefix[int(h)] = [b, self.tick]
            self.refcount[b] += 1

    def prefix_evict(self, max_blocks):
        self._prefix_init()
        cand = sorted((e[1], e[0], h) for h, e in self.prefix.items() if self.refcount[e[0]] == 1)
        n = 0
        for _, b, h in cand[:max_blocks]:
            del self.prefix[h]
            self.refcount[b] = 0
            self.free_stack.append(b)
            n += 1
        return n

    # ----------------------------------------------------------------- views
    def stats(self):
        used = sum(1 for r in self.refcount if r > 0)
        shared = sum(1 for r in self.refcount if r > 1)
        return used, self.num_blocks - used, shared

    def check_invariants(self, tables=None) -> None:
        assert all(r >= 0 for r in self.refcount)
        assert len(set(self.free_stack)) == len(self.free_stack), "duplicate in free list"
        free_set = set(self.free_stack)
        for b, r in enumerate(self.refcount):
            assert (r == 0) == (b in free_set), f"block {b}: rc {r}, free {b in free_set}"
        if tables is not None:
            refs = Counter(b for row in tables for b in row)
            for b in range(self.num_blocks):
                assert refs.get(b, 0) == self.refcount[b], (
                    f"block {b}: {refs.get(b, 0)} table refs vs refcount {self.refcount[b]}")


def slot_of(table_row, pos: int, block_size: int = 16) -> int:
    """Physical slot of logical token ``pos``: table[pos // B] * B + pos % B."""
    j, off = divmod(pos, block_size)
    return table_row[j] * block_size + off


def blocks_for(tokens: int, block_size: int = 16) -> int:
    return (tokens + block_size - 1) // block_size


def internal_waste(reserved_tokens: int, used_tokens: int) -> float:
    """Fraction of a reservation left unused (internal fragmentation)."""
    return 1.0 - used_tokens / reserved_tokens


def fnv1a64(data: bytes, h: int = 0xCBF29CE484222325) -> int:
    """64-bit FNV-1a (Fowler, Noll, Vo): per byte, h ^= b; h *= 0x100000001B3."""
    for b in data:
        h ^= b
        h = (h * 0x100000001B3) & 0xFFFFFFFFFFFFFFFF
    return h


def prefix_chain_hashes(tokens, parent: int = 0, block_size: int = 16):
    """Chain hash of each full block: FNV-1a-64 of the previous block's hash
    (8 little-endian bytes) followed by the block's token ids (4 little-endian
    bytes each); the first block chains from `parent`."""
    out = []
    prev = parent
    for j in range(len(tokens) // block_size):
        data = prev.to_bytes(8, "little") + b"".join(
            (int(t) & 0xFFFFFFFF).to_bytes(4, "little")
            for t in tokens[j * block_size:(j + 1) * block_size])
        prev = fnv1a64(data)
        out.append(prev)
    return out
