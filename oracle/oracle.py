"""Oracle for the paged KV cache hot path: a plain, slow CPU restatement.

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
CPU-baseline leg of ``bench.py`` may import this module.  The CUDA library
never calls it, and it imports nothing from the library.

Pages restated here (cited by title and section):

* "step14_2 - index_select gather" (mini-vLLM tutorial): the per-block gather
  loop (section "Problem"), the flat-index gather (section "Solution"), and the
  scatter that writes with the same indices (section "Relation to step14_1").
* "vLLM PagedAttention source notes": the pool layout and ``slot_mapping``
  (§2.2), the gather-then-standard-attention decode (§2.3), the
  fragmentation ratio (§3).
* "mini-runtime ch.12 Paged KV Cache": the BlockTable with its first-block
  offset and capacity (§2.2), block-granular allocation (§2.3), the
  logical-contiguous / physical-arbitrary mapping (§2.1 figure) and the
  exercises at the end of the chapter.

Representation.  A pool is a numpy array ``[num_blocks, num_layers,
block_size, num_kv_heads, head_dim]``; bf16 pools hold the raw uint16 bit
patterns and fp32 pools hold float32, so copies are bit copies.  Attention
widens the stored values exactly to fp64 and works in fp64 throughout.

Readings where the pages are silent:

* Logical token ``i`` of a sequence with first-block offset ``off`` sits at
  table position ``p = off + i``; its block is ``table[p // bs]`` and its row
  ``p % bs``.  The step14_2 formulas are the ``off == 0`` case.
* ``slot_mapping`` entries equal to ``-1`` are skipped; any other negative
  entry, an entry past the pool, or a repeated slot is rejected.
* The decode query attends to every one of the ``seq_len`` tokens (no mask);
  query head ``h`` reads kv head ``h // (Hq // Hkv)``; ``seq_len == 0`` gives
  an all-zero output row.

Parity pins: every function here is checked in ``tests/test_oracle_pins.py``
against the pages' worked examples, closed forms, a library attention routine
and brute-force enumeration.  No function is "parity unpinned".
"""

from __future__ import annotations

import math
from typing import Iterable, List, Optional, Sequence

import numpy as np

__all__ = [
    "blocks_needed", "capacity", "last_block_fill", "fragmentation_ratio",
    "slot_of", "build_slot_mapping", "write_slots", "gather_loop",
    "gather_indexed", "gather_batch", "widen", "attention_fp64",
    "decode_attention", "decode_attention_pairs", "split_partials",
    "combine_partials", "copy_blocks", "swap_out", "swap_in", "prefill_attention",
    "prefill_attention_rows",
]


# ---------------------------------------------------------------------------
# block arithmetic
# ---------------------------------------------------------------------------

def blocks_needed(num_tokens: int, block_size: int, offset: int = 0) -> int:
    """Blocks a sequence of ``num_tokens`` spans when its first token sits at
    row ``offset`` of its first block.

    mini-runtime ch.12 §2.3, allocation flow: a request of ``num_tokens`` needs
    ``ceil(num_tokens / block_size)`` blocks (vLLM notes §2.1,
    ``prefill_allocate``, says the same); with a first-block offset (ch.12
    §2.2) the span starts ``offset`` rows into the first block.
    """
    if num_tokens < 0 or not (0 <= offset < block_size):
        raise ValueError("bad token count or offset")
    if num_tokens == 0:
        return 0
    return -(-(offset + num_tokens) // block_size)


def capacity(num_blocks: int, block_size: int, offset: int) -> int:
    """Tokens a BlockTable can hold: ``num_blocks * block_size - offset``
    (mini-runtime ch.12 §2.2, BlockTable field table)."""
    return num_blocks * block_size - offset


def last_block_fill(num_tokens: int, block_size: int, offset: int = 0) -> int:
    """Rows used in the last block of a sequence (ch.12 exercises: a partly
    filled last block is the only internal waste)."""
    if num_tokens <= 0:
        return 0
    return (offset + num_tokens - 1) % block_size + 1


def fragmentation_ratio(total_allocated_blocks: int, block_size: int,
                        total_used_tokens: int) -> float:
    """vLLM notes §3: (allocated slots - used tokens) / allocated slots."""
    slots = total_allocated_blocks * block_size
    return (slots - total_used_tokens) / slots


# ---------------------------------------------------------------------------
# logical -> physical index (slot_mapping)
# ---------------------------------------------------------------------------

def slot_of(block_table: Sequence[int], offset: int, i: int, block_size: int) -> int:
    """Physical slot of logical token ``i``.

    vLLM notes §2.2: ``slot = block_table[block_idx] * block_size + offset``
    where ``block_idx`` and the in-block offset are the quotient and remainder
    of the token position by the block size (step14_2, "Solution":
    ``positions // block_size`` and ``positions % block_size``).  The position
    is shifted by the BlockTable's first-block offset (ch.12 §2.2).
    """
    p = offset + i
    return int(block_table[p // block_size]) * block_size + p % block_size


def build_slot_mapping(block_tables: np.ndarray, offsets: np.ndarray,
                       token_seq: np.ndarray, token_pos: np.ndarray,
                       block_size: int) -> np.ndarray:
    """``slot_mapping`` for a token list: int64, ``-1`` for padding entries
    (``token_seq == -1``), else :func:`slot_of` (vLLM notes §2.2)."""
    T = len(token_seq)
    out = np.empty(T, dtype=np.int64)
    for t in range(T):
        b = int(token_seq[t])
        if b < 0:
            out[t] = -1
            continue
        out[t] = slot_of(block_tables[b], int(offsets[b]), int(token_pos[t]),
                         block_size)
    return out


# ---------------------------------------------------------------------------
# scatter (slot_mapping write)
# ---------------------------------------------------------------------------

def write_slots(k_cache: np.ndarray, v_cache: np.ndarray, layer: int,
                k_new: np.ndarray, v_new: np.ndarray,
                slot_mapping: np.ndarray) -> None:
    """Write token rows into the pools in place.

    step14_2, "Relation to step14_1": the write is the gather's indexing on
    the left-hand side, ``pool[physical_blocks, slot_indices] = K``.  vLLM
    notes §2.2: rows are addressed as ``[block_id, layer_idx, offset]`` and
    ``-1`` in ``slot_mapping`` is padding, which is not written.
    """
    N, L, bs = k_cache.shape[:3]
    seen = set()
    for t in range(len(slot_mapping)):
        s = int(slot_mapping[t])
        if s == -1:
            continue
        if s < 0 or s >= N * bs:
            raise IndexError(f"slot {s} outside the pool")
        if s in seen:
            raise ValueError(f"slot {s} written twice")
        seen.add(s)
        blk, j = divmod(s, bs)
        k_cache[blk, layer, j] = k_new[t]
        v_cache[blk, layer, j] = v_new[t]


# ---------------------------------------------------------------------------
# gather (block_table read)
# ---------------------------------------------------------------------------

def gather_loop(pool: np.ndarray, layer: int, block_table: Sequence[int],
                seq_len: int, offset: int = 0) -> np.ndarray:
    """Contiguous ``[seq_len, Hkv, D]`` copy of one sequence, block by block.

    step14_2, "Problem": walk the table in order, take ``min(block_size,
    remaining)`` rows from each block and concatenate.  Generalised with the
    first-block offset of ch.12 §2.2: the first block contributes rows from
    ``offset`` on, so that reading does not start at the block head.
    """
    bs = pool.shape[2]
    chunks: List[np.ndarray] = []
    remaining = seq_len
    start = offset
    for blk in block_table:
        if remaining <= 0:
            break
        take = min(bs - start, remaining)
        chunks.append(pool[int(blk), layer, start:start + take])
        remaining -= take
        start = 0
    if remaining > 0:
        raise IndexError("sequence longer than its table's capacity")
    if not chunks:
        return np.zeros((0,) + pool.shape[3:], dtype=pool.dtype)
    return np.concatenate(chunks, axis=0)


def gather_indexed(pool: np.ndarray, layer: int, block_table: Sequence[int],
                   seq_len: int, offset: int = 0) -> np.ndarray:
    """Same result as :func:`gather_loop` through one flat index.

    step14_2, "Solution": positions ``0..seq_len-1``, block index
    ``positions // block_size``, row ``positions % block_size``, physical
    block ``table[block index]``, one advanced-indexing read.  Positions are
    shifted by the first-block offset (ch.12 §2.2).
    """
    bs = pool.shape[2]
    positions = offset + np.arange(seq_len, dtype=np.int64)
    bt = np.asarray(block_table, dtype=np.int64)
    return pool[bt[positions // bs], layer, positions % bs]


def gather_batch(k_cache: np.ndarray, v_cache: np.ndarray, layer: int,
                 block_tables: np.ndarray, seq_lens: np.ndarray,
                 offsets: np.ndarray):
    """Every sequence gathered with :func:`gather_loop` and concatenated in
    batch order (vLLM notes §2.3, ``gather_kv_for_attention``)."""
    ks, vs = [], []
    for b in range(len(seq_lens)):
        ks.append(gather_loop(k_cache, layer, block_tables[b], int(seq_lens[b]),
                              int(offsets[b])))
        vs.append(gather_loop(v_cache, layer, block_tables[b], int(seq_lens[b]),
                              int(offsets[b])))
    return np.concatenate(ks, axis=0), np.concatenate(vs, axis=0)


# ---------------------------------------------------------------------------
# decode attention
# ---------------------------------------------------------------------------

def widen(x: np.ndarray) -> np.ndarray:
    """Stored values, exactly, as fp64.  bf16 bits are the upper half of an
    IEEE fp32 word, so shifting them up 16 bits gives the same number."""
    if x.dtype == np.uint16:
        return (x.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    if x.dtype == np.float32:
        return x.astype(np.float64)
    if x.dtype == np.float64:
        return x
    raise TypeError(f"unsupported element type {x.dtype}")


def attention_fp64(q: np.ndarray, k: np.ndarray, v: np.ndarray,
                   scale: float) -> np.ndarray:
    """Standard single-query attention in fp64 (vLLM notes §2.3: the gathered
    K/V go through ordinary multi-head attention).

    ``q`` is ``[D]``, ``k`` and ``v`` are ``[n, D]``:
    ``softmax(scale * k @ q) @ v``, with the maximum logit subtracted before
    exponentiation.  ``n == 0`` gives zeros.
    """
    if k.shape[0] == 0:
        return np.zeros(v.shape[1], dtype=np.float64)
    s = scale * (k @ q)
    p = np.exp(s - s.max())
    return (p @ v) / p.sum()


def decode_attention(k_cache: np.ndarray, v_cache: np.ndarray, layer: int,
                     q: np.ndarray, block_tables: np.ndarray,
                     seq_lens: np.ndarray, offsets: np.ndarray,
                     scale: float) -> np.ndarray:
    """Decode attention for a batch, ``[B, Hq, D]`` in fp64.

    vLLM notes §2.3 (minivLLM path): gather each sequence's K/V to contiguous
    ``[seq_len, Hkv, D]`` and run standard attention for its one query token.
    Query head ``h`` uses kv head ``h // (Hq // Hkv)``.
    """
    B, Hq, D = q.shape
    Hkv = k_cache.shape[3]
    if Hq % Hkv:
        raise ValueError("num_q_heads must be a multiple of num_kv_heads")
    group = Hq // Hkv
    qd = widen(q)
    out = np.zeros((B, Hq, D), dtype=np.float64)
    for b in range(B):
        kb = widen(gather_loop(k_cache, layer, block_tables[b], int(seq_lens[b]),
                               int(offsets[b])))
        vb = widen(gather_loop(v_cache, layer, block_tables[b], int(seq_lens[b]),
                               int(offsets[b])))
        for h in range(Hq):
            g = h // group
            out[b, h] = attention_fp64(qd[b, h], kb[:, g, :], vb[:, g, :], scale)
    return out


def decode_attention_pairs(k_cache: np.ndarray, v_cache: np.ndarray, layer: int,
                           q: np.ndarray, block_tables: np.ndarray,
                           seq_lens: np.ndarray, offsets: np.ndarray,
                           scale: float, pairs: Iterable) -> dict:
    """:func:`decode_attention` for selected ``(b, h)`` pairs only, gathering
    just the kv head each pair reads; returns ``{(b, h): [D] fp64}``."""
    Hq = q.shape[1]
    group = Hq // k_cache.shape[3]
    out = {}
    for b, h in pairs:
        g = h // group
        kb = gather_loop(k_cache[:, :, :, g:g + 1], layer, block_tables[b],
                         int(seq_lens[b]), int(offsets[b]))
        vb = gather_loop(v_cache[:, :, :, g:g + 1], layer, block_tables[b],
                         int(seq_lens[b]), int(offsets[b]))
        out[(b, h)] = attention_fp64(widen(q[b, h]), widen(kb[:, 0, :]),
                                     widen(vb[:, 0, :]), scale)
    return out


# ---------------------------------------------------------------------------
# split-K partials and their combination
# ---------------------------------------------------------------------------

def split_partials(q: np.ndarray, k: np.ndarray, v: np.ndarray, scale: float,
                   bounds: Sequence[int]):
    """Per-chunk softmax state over the token chunks ``[bounds[c],
    bounds[c+1])``: the chunk maximum ``m``, ``l = sum exp(s - m)`` and
    ``acc = sum exp(s - m) v`` (fp64).  The pages leave the split open; this
    is the plain definition of attention restricted to a chunk."""
    parts = []
    for c in range(len(bounds) - 1):
        lo, hi = bounds[c], bounds[c + 1]
        if hi <= lo:
            continue
        s = scale * (k[lo:hi] @ q)
        m = s.max()
        p = np.exp(s - m)
        parts.append((m, p.sum(), p @ v[lo:hi]))
    return parts


def combine_partials(parts, head_dim: int) -> np.ndarray:
    """Merge chunk states: with ``M = max_c m_c``, the output is
    ``sum_c e^(m_c - M) acc_c / sum_c e^(m_c - M) l_c``."""
    if not parts:
        return np.zeros(head_dim, dtype=np.float64)
    M = max(m for m, _, _ in parts)
    num = sum(math.exp(m - M) * acc for m, _, acc in parts)
    den = sum(math.exp(m - M) * l for m, l, _ in parts)
    return num / den


# ---------------------------------------------------------------------------
# block copy (copy-on-write) and swap between the pool and host memory
# ---------------------------------------------------------------------------

def _layers(pool: np.ndarray, layer: int):
    return slice(None) if layer < 0 else slice(layer, layer + 1)


def copy_blocks(k_cache: np.ndarray, v_cache: np.ndarray, layer: int,
                src: Sequence[int], dst: Sequence[int]) -> None:
    """Copy-on-write support (mini-runtime ch.12 §3.1: vLLM shares blocks
    with copy-on-write plus ref_count): block dst[i] receives the contents of
    block src[i], in one layer or (layer < 0) in every layer.  The pairs are
    applied in order; a destination is assumed not to be read as a source by
    another pair."""
    ls = _layers(k_cache, layer)
    for s_, d_ in zip(src, dst):
        k_cache[int(d_), ls] = k_cache[int(s_), ls]
        v_cache[int(d_), ls] = v_cache[int(s_), ls]


def swap_out(k_cache: np.ndarray, v_cache: np.ndarray, layer: int,
             blocks: Sequence[int]):
    """Preemption by swapping ("vLLM PagedAttention source notes" §2.4: move
    a request's KV from the GPU to the CPU): the listed blocks, in order, as
    contiguous host arrays [n, layers, bs, Hkv, D]."""
    ls = _layers(k_cache, layer)
    ks = np.stack([k_cache[int(b), ls] for b in blocks]) if len(blocks) else None
    vs = np.stack([v_cache[int(b), ls] for b in blocks]) if len(blocks) else None
    return ks, vs


def swap_in(k_cache: np.ndarray, v_cache: np.ndarray, layer: int,
            blocks: Sequence[int], host_k: np.ndarray, host_v: np.ndarray) -> None:
    """The reverse of :func:`swap_out`: host rows i go back into block
    blocks[i] (any free blocks; the table is updated by the allocator)."""
    ls = _layers(k_cache, layer)
    for i, b in enumerate(blocks):
        k_cache[int(b), ls] = host_k[i]
        v_cache[int(b), ls] = host_v[i]


# ---------------------------------------------------------------------------
# prefill attention (causal, over the paged cache)
# ---------------------------------------------------------------------------

def prefill_attention(k_cache: np.ndarray, v_cache: np.ndarray, layer: int, q: np.ndarray,
                      block_tables: np.ndarray, seq_lens: np.ndarray, offsets: np.ndarray,
                      cu_q: np.ndarray, scale: float) -> np.ndarray:
    """Prefill attention in fp64, ``[T, Hq, D]``.

    "vLLM PagedAttention source notes" §2.4 (prefill batch): the prompt
    tokens' K/V are in their blocks; each new token then attends to itself
    and to every earlier token of its sequence (causal attention; the plain
    reading, as the pages name no other mask).  The queries of sequence b are
    its last ``n = cu_q[b+1] - cu_q[b]`` tokens; query i sits at position
    ``P = seq_len - n + i`` and attends to keys ``0..P``, gathered block by
    block as in :func:`gather_loop`.  Query head h reads kv head
    ``h // (Hq // Hkv)``.
    """
    T, Hq, D = q.shape
    group = Hq // k_cache.shape[3]
    out = np.zeros((T, Hq, D), dtype=np.float64)
    qd = widen(q)
    for b in range(len(seq_lens)):
        n = int(cu_q[b + 1] - cu_q[b])
        if n == 0:
            continue
        L = int(seq_lens[b])
        kb = widen(gather_loop(k_cache, layer, block_tables[b], L, int(offsets[b])))
        vb = widen(gather_loop(v_cache, layer, block_tables[b], L, int(offsets[b])))
        for i in range(n):
            P = L - n + i
            for h in range(Hq):
                g = h // group
                out[int(cu_q[b]) + i, h] = attention_fp64(qd[int(cu_q[b]) + i, h],
                                                          kb[:P + 1, g], vb[:P + 1, g], scale)
    return out


def prefill_attention_rows(k_cache: np.ndarray, v_cache: np.ndarray, layer: int, q: np.ndarray,
                           block_tables: np.ndarray, seq_lens: np.ndarray, offsets: np.ndarray,
                           cu_q: np.ndarray, scale: float, rows: Iterable) -> dict:
    """:func:`prefill_attention` for selected ``(t, h)`` pairs only (``t`` a
    row of ``q``, ``h`` a query head): the same definition, evaluated where a
    full-size check samples it."""
    Hq = q.shape[1]
    group = Hq // k_cache.shape[3]
    out = {}
    for t, h in rows:
        b = int(np.searchsorted(cu_q, t, side="right") - 1)
        n = int(cu_q[b + 1] - cu_q[b])
        L = int(seq_lens[b])
        P = L - n + (t - int(cu_q[b]))
        g = h // group
        kb = widen(gather_loop(k_cache, layer, block_tables[b], P + 1, int(offsets[b])))
        vb = widen(gather_loop(v_cache, layer, block_tables[b], P + 1, int(offsets[b])))
        out[(t, h)] = attention_fp64(widen(q[t, h]), kb[:, g], vb[:, g], scale)
    return out

