"""Host-side block pool, block tables, slot mapping and copy-on-write bookkeeping.

This is the memory-manager side of PagedAttention, kept on the host: it decides which
physical block holds which logical block of a sequence and produces the three arrays
the GPU kernels consume (block tables, slot mapping, copy-on-write pairs).  It never
touches K/V data.

What it follows:

* A pool of fixed-size physical blocks shared by every request; a sequence takes a new
  block only when its last block is full, from wherever the pool has a free one
  (ultralytics.com glossary "PagedAttention", section "페이징의 작동 방식";
  gufacode.com "PagedAttention:KV cache 的页表革命", section "按需分配 demo":
  ceil(20/16) = 2 blocks, the 33rd token takes a third block).
* A block table maps logical block i of a sequence to a physical block id, read in
  logical order (vasteelab.pages.dev "PagedAttentionとは？", section
  "tokenを固定長blockへ分ける", table [7, 2, 11] for 12 tokens at 4 tokens per block).
* Token position ``pos`` lives at slot ``table[pos // bs] * bs + pos % bs`` — the
  write ``key_pool[block_table[pos // block_size], pos % block_size] = key`` of the
  ultralytics.com PyTorch example, flattened to one slot index.
* Blocks carry reference counts; several tables may point at one block; a sequence
  that must write into a block that another sequence still uses first gets its own
  copy (copy-on-write; vasteelab.pages.dev section "Copy-on-Writeで共通prefixを共有できる",
  ultralytics.com section "시퀀스 간 블록 공유").  The last remaining holder writes
  in place.
* Finished sequences return their blocks to the pool (ya.zerocoder.ru
  "Что такое PagedAttention", section "Учебная трасса: рост последовательности").
* Prefix caching on top of the pool (:class:`PrefixCache`): a full block is identified
  by the hash of its parent block's identity, the tokens it holds and the request's
  model conditions (adapter id, multimodal input hashes), so a later prompt that starts
  with the same tokens under the same conditions reuses the blocks instead of computing
  them again (vasteelab.pages.dev "PagedAttentionとは？", section "Prefix Cachingとの違い").
"""
from __future__ import annotations

import hashlib
from collections import OrderedDict, deque
from dataclasses import dataclass, field
from typing import Iterable, List, Optional, Sequence, Tuple


class PoolExhausted(RuntimeError):
    """Raised when a block is needed and the pool has no free block left."""


class BlockAllocator:
    """Free list + reference counts over ``num_blocks`` physical blocks.

    ``free_order`` fixes the order in which free blocks are handed out (a shuffled
    order gives scattered tables, as on the pages); by default blocks come out
    0, 1, 2, ...
    """

    def __init__(self, num_blocks: int, block_size: int,
                 free_order: Optional[Iterable[int]] = None):
        if num_blocks <= 0 or block_size <= 0:
            raise ValueError("num_blocks and block_size must be positive")
        self.num_blocks = int(num_blocks)
        self.block_size = int(block_size)
        order = list(range(num_blocks)) if free_order is None else [int(b) for b in free_order]
        if sorted(order) != list(range(num_blocks)):
            raise ValueError("free_order must be a permutation of range(num_blocks)")
        self._free = deque(order)
        self.refcount = [0] * num_blocks

    @property
    def num_free(self) -> int:
        return len(self._free)

    def allocate(self) -> int:
        if not self._free:
            raise PoolExhausted("no free block in the pool")
        b = self._free.popleft()
        assert self.refcount[b] == 0
        self.refcount[b] = 1
        return b

    def incref(self, block: int) -> None:
        if self.refcount[block] <= 0:
            raise ValueError(f"block {block} is not allocated")
        self.refcount[block] += 1

    def decref(self, block: int) -> None:
        if self.refcount[block] <= 0:
            raise ValueError(f"block {block} is not allocated")
        self.refcount[block] -= 1
        if self.refcount[block] == 0:
            self._free.append(block)

    def is_free(self, block: int) -> bool:
        return self.refcount[block] == 0


RELEASED = -1  # table entry of a block released after it left a sliding window


@dataclass
class SequenceBlocks:
    """One sequence's block table and its number of cached tokens."""
    blocks: List[int] = field(default_factory=list)
    length: int = 0
    released: int = 0  # leading table entries released after they left a sliding window

    def slot(self, pos: int, block_size: int) -> int:
        if not 0 <= pos < len(self.blocks) * block_size:
            raise IndexError(f"position {pos} is outside the table")
        b = self.blocks[pos // block_size]
        if b == RELEASED:
            raise IndexError(f"position {pos} lies in a released block")
        return b * block_size + pos % block_size


def blocks_needed(num_tokens: int, block_size: int) -> int:
    """ceil(num_tokens / block_size): e.g. 33 tokens at 16 per block need 3 blocks."""
    return -(-int(num_tokens) // int(block_size))


class BlockManager:
    """Block tables for a set of sequences over one :class:`BlockAllocator`."""

    def __init__(self, allocator: BlockAllocator):
        self.alloc = allocator
        self.bs = allocator.block_size
        self.seqs: dict = {}

    # -- sequence lifetime -------------------------------------------------
    def add_sequence(self, seq_id, num_tokens: int = 0) -> List[int]:
        """Register a sequence and reserve blocks for its first ``num_tokens``
        tokens; returns their slots in position order."""
        if seq_id in self.seqs:
            raise ValueError(f"sequence {seq_id} exists")
        self.seqs[seq_id] = SequenceBlocks()
        slots = []
        for _ in range(num_tokens):
            slot, pair = self.append_token(seq_id)
            assert pair is None
            slots.append(slot)
        return slots

    def fork(self, parent_id, child_id) -> None:
        """The child shares every block of the parent (reference counts go up)."""
        if child_id in self.seqs:
            raise ValueError(f"sequence {child_id} exists")
        p = self.seqs[parent_id]
        for b in p.blocks:
            if b != RELEASED:
                self.alloc.incref(b)
        self.seqs[child_id] = SequenceBlocks(list(p.blocks), p.length, p.released)

    def free_sequence(self, seq_id) -> None:
        s = self.seqs.pop(seq_id)
        for b in s.blocks:
            if b != RELEASED:
                self.alloc.decref(b)

    def release_outside_window(self, seq_id, window: int) -> List[int]:
        """Sliding window of ``window`` positions: give back every block whose
        positions all lie before the last ``window`` ones (attention never reads them
        again); their table entries become RELEASED.  Returns the released ids
        (ya.zerocoder.ru, section "Где подход не решает задачу": a limited attention
        window frees the blocks that have left it)."""
        s = self.seqs[seq_id]
        first_kept = max(0, s.length - int(window)) // self.bs  # block holding the window's first position
        out = []
        for i in range(s.released, min(first_kept, len(s.blocks))):
            self.alloc.decref(s.blocks[i])
            out.append(s.blocks[i])
            s.blocks[i] = RELEASED
        s.released = max(s.released, min(first_kept, len(s.blocks)))
        return out

    # -- growth ------------------------------------------------------------
    def append_token(self, seq_id) -> Tuple[int, Optional[Tuple[int, int]]]:
        """Reserve the slot for the next token of ``seq_id``.

        A new block is taken only when the last one is full.  If the target block is
        shared (reference count > 1), the sequence first gets a private copy: the
        returned pair ``(src, dst)`` must be copied on the device before the token is
        written.  Returns ``(slot, pair_or_None)``.
        """
        s = self.seqs[seq_id]
        pair = None
        if s.length == len(s.blocks) * self.bs:
            s.blocks.append(self.alloc.allocate())
        else:
            last = s.blocks[s.length // self.bs]
            if self.alloc.refcount[last] > 1:
                new = self.alloc.allocate()
                self.alloc.decref(last)
                s.blocks[s.length // self.bs] = new
                pair = (last, new)
        slot = s.slot(s.length, self.bs)
        s.length += 1
        return slot, pair

    # -- export ------------------------------------------------------------
    def block_table_rows(self, seq_ids: Sequence, max_blocks: Optional[int] = None,
                         pad: int = -1) -> List[List[int]]:
        rows = [list(self.seqs[i].blocks) for i in seq_ids]
        mb = max_blocks if max_blocks is not None else max((len(r) for r in rows), default=0)
        out = []
        for r in rows:
            if len(r) > mb:
                raise ValueError("table longer than max_blocks")
            out.append(r + [pad] * (mb - len(r)))
        return out

    def unused_slots(self, seq_id) -> int:
        """Internal fragmentation: reserved slots that hold no token."""
        s = self.seqs[seq_id]
        return len(s.blocks) * self.bs - s.length

    # -- structural checks -------------------------------------------------
    def check_structure(self, held: Iterable[int] = ()) -> None:
        """Structural correctness: every table entry is an allocated block (or, in a
        leading run, a block released after it left a sliding window), each
        sequence's table covers its tokens exactly, reference counts equal the number
        of table entries pointing at each block plus the references ``held`` by other
        owners (a prefix cache), and no free block is referenced (ya.zerocoder.ru,
        section "Учебная трасса: рост последовательности": the table references
        existing blocks, reference counts balance, frees leave nothing dangling)."""
        counts = [0] * self.alloc.num_blocks
        for b in held:
            counts[b] += 1
        for sid, s in self.seqs.items():
            if len(s.blocks) != blocks_needed(s.length, self.bs):
                raise AssertionError(f"sequence {sid}: {len(s.blocks)} blocks for {s.length} tokens")
            released = 0
            while released < len(s.blocks) and s.blocks[released] == RELEASED:
                released += 1
            for b in s.blocks[released:]:
                if not 0 <= b < self.alloc.num_blocks:
                    raise AssertionError(f"sequence {sid}: block {b} outside the pool")
                counts[b] += 1
            if released and released * self.bs >= s.length:
                raise AssertionError(f"sequence {sid}: the block holding its last token was released")
        for b in range(self.alloc.num_blocks):
            if counts[b] != self.alloc.refcount[b]:
                raise AssertionError(f"block {b}: refcount {self.alloc.refcount[b]} but {counts[b]} references")
        free = list(self.alloc._free)
        if len(set(free)) != len(free):
            raise AssertionError("a block is on the free list twice")
        for b in free:
            if counts[b] != 0:
                raise AssertionError(f"free block {b} is still referenced")
        if len(free) + sum(1 for c in counts if c > 0) != self.alloc.num_blocks:
            raise AssertionError("a block is neither free nor referenced")


def validate_cow_pairs(pairs: Sequence[Tuple[int, int]], num_blocks: int) -> None:
    """Copy pairs are applied in parallel on the device, so destinations must be
    distinct and no destination may also be a source."""
    dsts = [d for _, d in pairs]
    srcs = {s for s, _ in pairs}
    if len(set(dsts)) != len(dsts):
        raise ValueError("duplicate copy destination")
    for s, d in pairs:
        if not (0 <= s < num_blocks and 0 <= d < num_blocks):
            raise ValueError(f"pair ({s}, {d}) outside the pool")
        if d in srcs:
            raise ValueError(f"block {d} is both a source and a destination")


class PrefixCache:
    """Reuse of full blocks computed for earlier prompts, over a :class:`BlockManager`.

    A full block's identity is a hash chained from its parent's: H(parent identity,
    the block's tokens, the request's extra keys such as an adapter id or multimodal
    input hashes).  Equal identities mean equal tokens at equal positions under equal
    conditions, hence equal keys and values, so the block can be shared.  Only full
    blocks are identified (a partial block still grows).  The cache keeps one reference
    to every block it identifies, so a block outlives the sequences that computed it
    until :meth:`evict` drops it (least recently used first, and only blocks no
    sequence holds).  Blocks are identified when their prompt is added: the cache write
    of that step puts their keys and values in place before any later attention reads
    them.
    """

    def __init__(self, manager: BlockManager):
        self.mgr = manager
        self.by_hash: "OrderedDict[bytes, int]" = OrderedDict()  # identity -> block, oldest use first

    @staticmethod
    def block_hash(parent: Optional[bytes], tokens: Sequence[int], extra: Sequence = ()) -> bytes:
        h = hashlib.sha256()
        h.update(parent if parent is not None else bytes(32))
        h.update(len(tokens).to_bytes(4, "little"))
        for t in tokens:
            h.update(int(t).to_bytes(8, "little", signed=True))
        h.update(repr(tuple(extra)).encode())
        return h.digest()

    def add_prompt(self, seq_id, tokens: Sequence[int], extra: Sequence = ()) -> Tuple[List[int], int]:
        """Register ``seq_id`` with a prompt.  Its longest run of leading full blocks
        whose identities are cached is shared (reference counts go up); blocks are
        reserved for the rest, and the new full blocks are identified.  At least the
        last token is always computed (a prompt cached whole gives back its last block
        and computes it again).  Returns (slots of the tokens still to compute, in
        position order, number of cached tokens)."""
        mgr, bs = self.mgr, self.mgr.bs
        if seq_id in mgr.seqs:
            raise ValueError(f"sequence {seq_id} exists")
        tokens = list(tokens)
        nfull = len(tokens) // bs
        ids, parent = [], None
        for i in range(nfull):
            parent = self.block_hash(parent, tokens[i * bs:(i + 1) * bs], extra)
            ids.append(parent)
        reused = []
        for h in ids:
            b = self.by_hash.get(h)
            if b is None:
                break
            reused.append(b)
        if reused and len(reused) * bs == len(tokens):
            reused.pop()
        for i, b in enumerate(reused):
            mgr.alloc.incref(b)
            self.by_hash.move_to_end(ids[i])
        cached = len(reused) * bs
        mgr.seqs[seq_id] = SequenceBlocks(blocks=list(reused), length=cached)
        slots = []
        for _ in range(len(tokens) - cached):
            slot, pair = mgr.append_token(seq_id)
            assert pair is None  # new tokens go to fresh blocks: reused blocks are full
            slots.append(slot)
        blocks = mgr.seqs[seq_id].blocks
        for i in range(len(reused), nfull):
            if ids[i] not in self.by_hash:
                self.by_hash[ids[i]] = blocks[i]
                mgr.alloc.incref(blocks[i])  # the cache's own reference
        return slots, cached

    def held(self) -> List[int]:
        """The blocks the cache holds a reference to."""
        return list(self.by_hash.values())

    def evict(self, n: int) -> int:
        """Drop up to ``n`` identified blocks that no sequence holds, least recently
        used first, returning them to the pool; returns how many were dropped."""
        dropped = 0
        for h in list(self.by_hash):
            if dropped >= n:
                break
            b = self.by_hash[h]
            if self.mgr.alloc.refcount[b] == 1:
                del self.by_hash[h]
                self.mgr.alloc.decref(b)
                dropped += 1
        return dropped

