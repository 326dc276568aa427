"""The host block allocator: the oracle allocator pinned to what the pages
fix, and the library's C++ allocator (through the C ABI) bit-exact against
the oracle on seeded random operation traces.  CPU only."""

import os
import random

import numpy as np
import pytest

import oracle
from oracle import allocator as OA
import paged_kv_cache_blk_gb300 as pkv
from paged_kv_cache_blk_gb300 import PkvError

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _rows(path):
    return [l.split() for l in open(path) if l.strip() and not l.startswith("#")]


# ---------------------------------------------------------------------------
# invariants every state must satisfy
# ---------------------------------------------------------------------------

def check_invariants(m, extra=None):
    """Every block is free (ref 0, once in the deque) or held: its ref_count
    is the number of sequences holding it plus the references the caller
    holds directly (`extra`)."""
    holders = [0] * m.num_blocks
    for b in (extra or []):
        holders[b] += 1
    for t in m.seqs.values():
        span = -(-(t.offset + t.num_tokens) // m.block_size) if t.num_tokens else 0
        assert len(t.block_ids) == span
        assert 0 <= t.offset < m.block_size
        for b in t.block_ids:
            holders[b] += 1
    free = list(m.free)
    assert len(free) == len(set(free))
    for b in range(m.num_blocks):
        if b in free:
            assert m.ref_count[b] == 0 and holders[b] == 0
        else:
            assert m.ref_count[b] == holders[b] > 0


# ---------------------------------------------------------------------------
# pins for the oracle allocator
# ---------------------------------------------------------------------------

def pin_exercise(M):
    for n, bs, blocks, slots, last, util, frag in _rows(
            os.path.join(GOLDEN, "exercise_30_tokens.txt")):
        n, bs, blocks = int(n), int(bs), int(blocks)
        m = M(64, bs)
        m.seq_new(1)
        m.seq_append(1, n)
        assert len(m.seq_table(1).block_ids) == blocks
        assert m.seq_table(1).capacity(bs) == int(slots)
        a, used, ratio = m.fragmentation()
        assert (a, used) == (blocks, n) and ratio == float(frag)


def pin_fifo(M):
    order = [5, 3, 9, 0, 7, 1, 2, 4, 6, 8]
    m = M(10, 4, order)
    assert m.allocate_blocks(3) == [5, 3, 9]
    m.dec_ref(3)
    assert list(m.free) == [0, 7, 1, 2, 4, 6, 8, 3]      # released to the back
    assert m.allocate_blocks(2) == [0, 7]


def pin_all_or_nothing(M):
    m = M(4, 4)
    m.seq_new(1)
    m.seq_append(1, 10)                                  # 3 blocks
    before = (list(m.free), list(m.seq_table(1).block_ids), m.seq_table(1).num_tokens)
    with pytest.raises(OA.NoBlocks):
        m.seq_append(1, 7)                               # needs 2 more, 1 free
    assert (list(m.free), list(m.seq_table(1).block_ids), m.seq_table(1).num_tokens) == before
    with pytest.raises(OA.NoBlocks):
        m.allocate_blocks(2)
    assert list(m.free) == before[0]
    assert not m.can_allocate(5) and m.can_allocate(4)


def pin_decode_append(M):
    """vLLM notes §2.1 decode_append: a slot in the last block while it has
    room, otherwise a new block."""
    m = M(8, 4)
    m.seq_new(1, offset=1)
    slots, _ = m.seq_append(1, 3)                        # rows 1..3 of block 0
    assert slots == [1, 2, 3] and m.num_free() == 7
    s, _ = m.seq_append(1, 1)                            # block full: a new block
    assert s == [4 * 1 + 0] and m.num_free() == 6
    s, _ = m.seq_append(1, 1)
    assert s == [5] and m.num_free() == 6
    t = m.seq_table(1)
    assert t.capacity(4) == 2 * 4 - 1                    # ch.12 §2.2
    for i in range(t.num_tokens):
        assert oracle.slot_of(t.block_ids, t.offset, i, 4) == ([1, 2, 3, 4, 5])[i]


def pin_ref_count_order(M):
    """ch.12 exercise: a block held twice, both holders finish in either
    order: the block is freed exactly once, when the second one lets go."""
    finals = []
    for order in ((1, 2), (2, 1)):
        m = M(6, 4)
        m.seq_new(1)
        m.seq_append(1, 4)
        m.seq_fork(1, 2)
        b = m.seq_table(1).block_ids[0]
        assert m.ref_count[b] == 2
        m.seq_free(order[0])
        assert m.ref_count[b] == 1 and b not in m.free
        m.seq_free(order[1])
        assert m.ref_count[b] == 0 and list(m.free).count(b) == 1
        finals.append((list(m.free), list(m.ref_count)))
    assert finals[0] == finals[1]


def pin_copy_on_write(M):
    m = M(8, 4)
    m.seq_new(1)
    m.seq_append(1, 6)                                   # blocks 0, 1 (block 1 half full)
    m.seq_fork(1, 2)
    slots, cow = m.seq_append(2, 1)                      # writes into shared block 1
    assert cow == [(1, 2)] and slots == [2 * 4 + 2]
    assert m.seq_table(2).block_ids == [0, 2] and m.seq_table(1).block_ids == [0, 1]
    assert m.ref_count[1] == 1 and m.ref_count[2] == 1 and m.ref_count[0] == 2
    s1, cow1 = m.seq_append(1, 1)                        # block 1 is private again
    assert cow1 == [] and s1 == [1 * 4 + 2]


def pin_prefix_share(M):
    m = M(16, 4)
    m.seq_new(1)
    m.seq_append(1, 12)                                  # blocks 0..2
    m.seq_new(2, offset=0)
    m.seq_share(2, m.seq_table(1).block_ids[:2], 8)      # prefix hit on 2 blocks
    assert [m.ref_count[b] for b in (0, 1, 2)] == [2, 2, 1]
    slots, cow = m.seq_append(2, 1)                      # block boundary: fresh block, no copy
    assert cow == [] and slots == [3 * 4]
    with pytest.raises(ValueError):
        m.seq_new(3)
        m.seq_share(3, [0, 1], 9)                        # 9 tokens span 3 blocks
    check_invariants(m)


def pin_fragmentation_formula(M):
    m = M(32, 16)
    for sid, n in ((1, 30), (2, 17), (3, 16)):
        m.seq_new(sid)
        m.seq_append(sid, n)
    a, used, ratio = m.fragmentation()
    assert (a, used) == (2 + 2 + 1, 63)
    assert ratio == oracle.fragmentation_ratio(5, 16, 63)


PINS = [pin_exercise, pin_fifo, pin_all_or_nothing, pin_decode_append, pin_ref_count_order,
        pin_copy_on_write, pin_prefix_share, pin_fragmentation_formula]


@pytest.mark.parametrize("pin", PINS, ids=[p.__name__ for p in PINS])
def test_oracle_allocator_pins(pin):
    pin(OA.KVCacheManager)


# planted mistakes: each broken allocator must fail some pin ----------------

class _Lifo(OA.KVCacheManager):
    def allocate_blocks(self, n):
        if n > len(self.free):
            raise OA.NoBlocks(n)
        out = [self.free.pop() for _ in range(n)]
        for b in out:
            self.ref_count[b] = 1
        return out


class _FreeAtOne(OA.KVCacheManager):
    def dec_ref(self, b):
        self.ref_count[b] = 0
        if b not in self.free:
            self.free.append(b)


class _NoCow(OA.KVCacheManager):
    def seq_append(self, sid, n):
        rc = self.ref_count
        self.ref_count = [min(c, 1) for c in rc]
        try:
            slots, _ = super().seq_append(sid, n)
        finally:
            fixed = self.ref_count
            self.ref_count = [max(a, b) if a else 0 for a, b in zip(rc, fixed)]
        return slots, []


class _Partial(OA.KVCacheManager):
    def seq_append(self, sid, n):
        t = self.seqs[sid]
        while True:
            try:
                return super().seq_append(sid, n)
            except OA.NoBlocks:
                if not self.free:
                    raise
                t.block_ids.append(self.allocate_blocks(1)[0])


@pytest.mark.parametrize("broken", [_Lifo, _FreeAtOne, _NoCow, _Partial],
                         ids=["lifo", "free-at-one", "no-cow", "partial-alloc"])
def test_pins_catch_broken_allocators(broken):
    failed = 0
    for pin in PINS:
        try:
            pin(broken)
        except (AssertionError, IndexError, ValueError, OA.NoBlocks):
            failed += 1
    assert failed >= 1


# ---------------------------------------------------------------------------
# the C++ allocator against the oracle
# ---------------------------------------------------------------------------

class Pair:
    """Runs each operation on both allocators and compares the outcome."""

    def __init__(self, num_blocks, bs, order):
        self.o = OA.KVCacheManager(num_blocks, bs, order)
        self.c = pkv.Allocator(num_blocks, bs, order)
        self.N, self.bs = num_blocks, bs

    def run(self, name, *args):
        err_o = err_c = None
        ro = rc = None
        try:
            ro = getattr(self.o, name)(*args)
        except OA.NoBlocks:
            err_o = "PKV_ERR_NO_BLOCKS"
        except (ValueError, KeyError, IndexError):
            err_o = "bad"
        try:
            rc = getattr(self.c, name)(*args)
        except PkvError as e:
            err_c = "PKV_ERR_NO_BLOCKS" if e.name == "PKV_ERR_NO_BLOCKS" else "bad"
        assert err_o == err_c, (name, args, err_o, err_c)
        if err_o is None and name == "seq_append":
            assert list(ro[0]) == rc[0].tolist() and ro[1] == rc[1]
        if err_o is None and name == "allocate_blocks":
            assert ro == rc
            self.last_alloc = list(ro)
        return err_o

    def compare(self):
        assert self.o.num_free() == self.c.num_free()
        assert [self.o.ref_count[b] for b in range(self.N)] == [
            self.c.ref_count(b) for b in range(self.N)]
        sids = sorted(self.o.seqs)
        if sids:
            mb = max(1, max(len(t.block_ids) for t in self.o.seqs.values()))
            tables, lens, offs = self.c.seq_tables(sids, mb)
            for i, sid in enumerate(sids):
                t = self.o.seqs[sid]
                assert tables[i].tolist() == t.block_ids + [-1] * (mb - len(t.block_ids))
                assert lens[i] == t.num_tokens and offs[i] == t.offset
        a, u, f = self.c.stats()
        ao, uo, fo = self.o.fragmentation()
        assert (a, u) == (ao, uo) and abs(f - fo) < 1e-12


@pytest.mark.parametrize("seed", range(6))
def test_cpp_allocator_matches_oracle(seed):
    rng = random.Random(seed)
    bs = rng.choice([1, 2, 4, 16])
    N = rng.choice([8, 24, 64])
    order = list(range(N))
    rng.shuffle(order)
    p = Pair(N, bs, order)
    next_id = 0
    held = []          # references the trace holds directly (not through a sequence)
    for step in range(400):
        live = sorted(p.o.seqs)
        op = rng.random()
        if op < 0.2 or not live:
            p.run("seq_new", next_id, rng.randrange(bs))
            next_id += 1
        elif op < 0.55:
            p.run("seq_append", rng.choice(live), rng.choice([0, 1, 1, 1, 3, bs, 2 * bs + 1]))
        elif op < 0.65:
            p.run("seq_fork", rng.choice(live), next_id)
            next_id += 1
        elif op < 0.78:
            p.run("seq_free", rng.choice(live))
        elif op < 0.88:
            src = p.o.seqs[rng.choice(live)]
            p.run("seq_new", next_id, src.offset)
            k = rng.randint(0, src.num_tokens)
            span = -(-(src.offset + k) // bs) if k else 0
            p.run("seq_share", next_id, src.block_ids[:span], k)
            next_id += 1
        elif op < 0.94:
            n = rng.randint(0, 3)
            if p.run("allocate_blocks", n) is None:
                held.extend(_last_allocated(p, n))
        else:
            if rng.random() < 0.5 or not held:
                # take another reference on a block in use
                used = [b for b in range(N) if p.o.ref_count[b] > 0]
                if used:
                    b = rng.choice(used)
                    p.run("inc_ref", b)
                    held.append(b)
                else:
                    p.run("inc_ref", rng.randrange(N))            # a free block: refused
            else:
                b = held.pop(rng.randrange(len(held)))
                p.run("dec_ref", b)
        # errors on both sides must agree too
        if rng.random() < 0.05:
            p.run("seq_free", 10_000_000)
            p.run("seq_append", rng.choice(sorted(p.o.seqs) or [0]), 10 * N * bs)
        p.compare()
        check_invariants(p.o, held)


def _last_allocated(p, n):
    return p.last_alloc if n else []


def test_cpp_allocator_refuses_bad_input():
    with pytest.raises(PkvError):
        pkv.Allocator(8, 3)
    with pytest.raises(PkvError):
        pkv.Allocator(4, 4, [0, 1, 1, 3])
    a = pkv.Allocator(4, 4)
    with pytest.raises(PkvError):
        a.seq_new(1, 4)
    a.seq_new(1)
    with pytest.raises(PkvError):
        a.seq_new(1)
    with pytest.raises(PkvError):
        a.dec_ref(2)                                     # free block
    with pytest.raises(PkvError) as e:
        a.seq_append(1, 17)
    assert e.value.name == "PKV_ERR_NO_BLOCKS"
    a.seq_append(1, 5)
    with pytest.raises(PkvError) as e:
        a.seq_tables([1], 1)
    assert e.value.name == "PKV_ERR_CAPACITY"
    assert a.ref_count(99) == -1


@pytest.mark.parametrize("seed", range(4))
def test_batched_append_matches_oracle(seed):
    rng = random.Random(100 + seed)
    bs, N = 4, 40
    order = list(range(N))
    rng.shuffle(order)
    o = OA.KVCacheManager(N, bs, order)
    c = pkv.Allocator(N, bs, order)
    nid = 0
    for step in range(60):
        live = sorted(o.seqs)
        r = rng.random()
        if r < 0.25 or len(live) < 2:
            for m in (o, c):
                m.seq_new(nid, rng.randrange(bs)) if m is o else None
            c.seq_new(nid, o.seqs[nid].offset)
            nid += 1
        elif r < 0.4:
            o.seq_fork(live[0], nid)
            c.seq_fork(live[0], nid)
            nid += 1
        elif r < 0.5:
            o.seq_free(live[-1])
            c.seq_free(live[-1])
        live = sorted(o.seqs)
        sids = rng.sample(live, rng.randint(1, len(live)))
        counts = [rng.choice([0, 1, 1, 2, bs + 1]) for _ in sids]
        try:
            ro = o.seq_append_batch(sids, counts)
            err_o = None
        except OA.NoBlocks:
            err_o = "PKV_ERR_NO_BLOCKS"
        try:
            rc = c.seq_append_batch(sids, counts)
            err_c = None
        except PkvError as e:
            err_c = e.name
        assert err_o == err_c
        if err_o is None:
            assert list(ro[0]) == rc[0].tolist() and ro[1] == rc[1]
        assert o.num_free() == c.num_free()
        assert [o.ref_count[b] for b in range(N)] == [c.ref_count(b) for b in range(N)]
    with pytest.raises(PkvError):
        c.seq_append_batch([sorted(o.seqs)[0]] * 2)          # repeated id


def test_batched_append_copy_on_write_order():
    """Two forks of one sequence append in the same step: the first copies
    the shared last block, the second then holds it alone and writes in place."""
    for M in (OA.KVCacheManager, lambda n, b: pkv.Allocator(n, b)):
        m = M(8, 4)
        m.seq_new(1)
        m.seq_append(1, 2)
        m.seq_fork(1, 2)
        slots, cow = m.seq_append_batch([1, 2])
        assert len(cow) == 1 and cow[0][0] == 0
        assert list(slots) == [cow[0][1] * 4 + 2, 0 * 4 + 2]
