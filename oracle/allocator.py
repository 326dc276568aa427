"""Oracle for the host block allocator: a plain restatement of the pages'
block manager.  TEST INFRASTRUCTURE ONLY (tests/, smoke and bench's
baseline legs may import it; the library never does).

Restated from:
* mini-runtime "ch.12 Paged KV Cache" §2.2 (BlockTable: block ids in logical
  order, first-block offset, capacity = num_blocks * block_size - offset),
  §2.3 (KVCacheManager: a FIFO deque of free block ids; allocate computes
  ceil(num_tokens / block_size) and pops that many from the left, or returns
  False and changes nothing when too few are free), §2.4 (ref_count:
  inc_ref when another holder shares a block, dec_ref when a holder lets go,
  the block returns to the free queue when its count reaches zero), §3.1
  (vLLM shares blocks with copy-on-write plus ref_count).
* "vLLM PagedAttention source notes" §2.1 (allocate / free / append_slot /
  can_allocate; decode_append adds a slot to the last block while it has
  room, else allocates a new block), §3 (fragmentation ratio).

Readings where the pages are silent:
* A released block goes to the right end of the free deque (deque
  semantics: popleft to allocate, append to release).
* Appending tokens to a sequence first fills its last block, then takes
  fresh blocks from the left of the deque, in order.  If the free blocks do
  not suffice for the whole append, nothing changes.
* Copy-on-write: when an append writes into a block whose ref_count is above
  one, that block is replaced in this sequence's table by a fresh block from
  the deque (dec_ref on the shared one); the caller copies the shared block's
  contents into the fresh one.  The fresh block is taken before the blocks
  the append needs beyond it.
* Fork shares every block of the source (inc_ref each) with the same offset
  and length; a prefix hit shares given blocks and covers given tokens.

Parity pins: tests/test_allocator.py (the chapter's exercises, FIFO order,
all-or-nothing allocation, ref-count order independence, capacity, the
fragmentation formula, and brute-force invariants).  No function here is
"parity unpinned".
"""

from __future__ import annotations

import collections
from dataclasses import dataclass, field
from typing import Dict, List, Optional, Sequence


class NoBlocks(Exception):
    """Fewer free blocks than an operation needs (nothing was changed)."""


@dataclass
class BlockTable:
    """ch.12 §2.2: physical block ids in logical order plus the first-block
    offset; capacity = num_blocks * block_size - offset."""
    block_ids: List[int] = field(default_factory=list)
    offset: int = 0
    num_tokens: int = 0

    def capacity(self, block_size: int) -> int:
        return len(self.block_ids) * block_size - self.offset


class KVCacheManager:
    def __init__(self, num_blocks: int, block_size: int, free_order: Optional[Sequence[int]] = None):
        self.block_size = block_size
        self.num_blocks = num_blocks
        order = list(range(num_blocks)) if free_order is None else [int(x) for x in free_order]
        if sorted(order) != list(range(num_blocks)):
            raise ValueError("free_order must be a permutation of the block ids")
        self.ref_count = [0] * num_blocks
        self.free = collections.deque(order)
        self.seqs: Dict[int, BlockTable] = {}

    # -- block level (ch.12 §2.3, §2.4) ---------------------------------------
    def num_free(self) -> int:
        return len(self.free)

    def allocate_blocks(self, n: int) -> List[int]:
        """Pop n ids from the left of the free deque, or raise NoBlocks and
        change nothing."""
        if n > len(self.free):
            raise NoBlocks(n)
        out = [self.free.popleft() for _ in range(n)]
        for b in out:
            self.ref_count[b] = 1
        return out

    def inc_ref(self, b: int) -> None:
        if self.ref_count[b] <= 0:
            raise ValueError(f"block {b} is free")
        self.ref_count[b] += 1

    def dec_ref(self, b: int) -> None:
        if self.ref_count[b] <= 0:
            raise ValueError(f"block {b} is free")
        self.ref_count[b] -= 1
        if self.ref_count[b] == 0:
            self.free.append(b)

    def can_allocate(self, num_tokens: int) -> bool:
        """vLLM notes §2.1: enough free blocks for a new request."""
        return -(-num_tokens // self.block_size) <= len(self.free)

    # -- sequences (BlockTable) -----------------------------------------------
    def seq_new(self, sid: int, offset: int = 0) -> None:
        if sid in self.seqs:
            raise ValueError(f"sequence {sid} exists")
        if not 0 <= offset < self.block_size:
            raise ValueError("offset must be in [0, block_size)")
        self.seqs[sid] = BlockTable([], offset, 0)

    def seq_share(self, sid: int, blocks: Sequence[int], num_tokens: int) -> None:
        """Prefix hit (ch.12 §2.4): the new sequence reuses already allocated
        blocks (inc_ref each) and covers num_tokens tokens of them."""
        t = self.seqs[sid]
        if t.block_ids:
            raise ValueError("sharing starts a sequence")
        span = -(-(t.offset + num_tokens) // self.block_size) if num_tokens > 0 else 0
        if num_tokens < 0 or span != len(blocks):
            raise ValueError("the shared blocks must be exactly the blocks the tokens span")
        for b in blocks:
            self.inc_ref(int(b))
        t.block_ids = [int(b) for b in blocks]
        t.num_tokens = num_tokens

    def seq_append(self, sid: int, num_tokens: int):
        """Append tokens (prefill or decode).  Returns (slots, cow) where
        slots are the appended tokens' slot numbers and cow is the list of
        (shared block, fresh block) pairs whose contents the caller copies."""
        t = self.seqs[sid]
        bs = self.block_size
        if num_tokens == 0:
            return [], []
        start = t.offset + t.num_tokens            # table position of the first new token
        end = start + num_tokens
        blocks_after = -(-end // bs) if end > 0 else 0
        new_blocks = max(0, blocks_after - len(t.block_ids))
        # the block the first new token lands in, if it exists and is shared
        first_blk = start // bs
        cow_needed = (num_tokens > 0 and first_blk < len(t.block_ids)
                      and self.ref_count[t.block_ids[first_blk]] > 1)
        need = new_blocks + (1 if cow_needed else 0)
        if need > len(self.free):
            raise NoBlocks(need)
        cow = []
        if cow_needed:
            old = t.block_ids[first_blk]
            fresh = self.allocate_blocks(1)[0]
            self.dec_ref(old)
            t.block_ids[first_blk] = fresh
            cow.append((old, fresh))
        t.block_ids.extend(self.allocate_blocks(new_blocks))
        slots = [t.block_ids[p // bs] * bs + p % bs for p in range(start, end)]
        t.num_tokens += num_tokens
        return slots, cow

    def seq_append_batch(self, sids: Sequence[int], counts: Optional[Sequence[int]] = None):
        """One decode step for many sequences: seq_append on each in order,
        all or nothing (on NoBlocks the whole state is restored)."""
        import copy
        if len(set(sids)) != len(sids) or any(s not in self.seqs for s in sids):
            raise ValueError("unknown or repeated sequence id")
        saved = copy.deepcopy((self.ref_count, self.free, self.seqs))
        slots, cows = [], []
        try:
            for i, sid in enumerate(sids):
                sl, cw = self.seq_append(sid, 1 if counts is None else int(counts[i]))
                slots.extend(sl)
                cows.extend(cw)
        except NoBlocks:
            self.ref_count, self.free, self.seqs = saved
            raise
        return slots, cows

    def seq_fork(self, src: int, dst: int) -> None:
        s = self.seqs[src]
        if dst in self.seqs:
            raise ValueError(f"sequence {dst} exists")
        for b in s.block_ids:
            self.inc_ref(b)
        self.seqs[dst] = BlockTable(list(s.block_ids), s.offset, s.num_tokens)

    def seq_free(self, sid: int) -> None:
        """vLLM notes §2.1 free / minivLLM free_request: every block of the
        sequence is released (dec_ref)."""
        t = self.seqs.pop(sid)
        for b in t.block_ids:
            self.dec_ref(b)

    def seq_table(self, sid: int) -> BlockTable:
        return self.seqs[sid]

    # -- accounting (vLLM notes §3) ---------------------------------------------
    def fragmentation(self):
        """(allocated blocks, used token slots, ratio) over live blocks: each
        allocated block counted once; a slot is used when some sequence holds
        a token in it."""
        used = set()
        for t in self.seqs.values():
            for i in range(t.num_tokens):
                p = t.offset + i
                used.add((t.block_ids[p // self.block_size], p % self.block_size))
        allocated = sum(1 for c in self.ref_count if c > 0)
        ratio = 0.0 if allocated == 0 else (allocated * self.block_size - len(used)) / (
            allocated * self.block_size)
        return allocated, len(used), ratio
