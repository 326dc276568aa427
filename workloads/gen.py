"""Seeded synthetic workloads for the paged KV cache.

The five named workloads mirror the pages' setting: a block pool shaped
``[num_blocks, num_layers, block_size, num_kv_heads, head_dim]`` (vLLM notes
§2.2 and its PagedKVCache paragraph), block size 16 and 16384 blocks (mini-
runtime ch12 §4.2 decision table), block tables popped FIFO from a free list
(ch12 §2.3 KVCacheManager), first-block offsets from prefix sharing (ch12
§2.2) and ``-1`` padding in ``slot_mapping`` (vLLM notes §2.2).

Index structures are drawn with ``numpy.random.default_rng`` (PCG64, the same
stream on every platform).  Bulk K/V/Q values are drawn with a seeded
``torch.Generator`` on the target device as fp32 N(0, 1) and rounded once to
the pool dtype (round-to-nearest-even for bf16); both the oracle and the CUDA
path consume exactly those bits.

Sizing a block table needs the number of blocks a sequence spans,
``ceil((offset + seq_len) / block_size)``: that is workload layout, not the
method's slot or copy arithmetic, which lives in ``oracle/`` and the library.
"""

from __future__ import annotations

import collections
import math
from dataclasses import dataclass, field
from typing import Optional

import numpy as np
import torch

DTYPES = {"f32": torch.float32, "bf16": torch.bfloat16, "i8": torch.uint8}


@dataclass(frozen=True)
class PoolSpec:
    """Shape of one K (or V) pool tensor ``[N, L, bs, Hkv, D]``; an ``"i8"``
    pool is bytes ``[N, L, bs, row_bytes]`` whose token rows hold Hkv * D int8
    codes, then Hkv fp32 scales, then padding to a multiple of 16 bytes."""

    num_blocks: int
    num_layers: int
    block_size: int
    num_kv_heads: int
    head_dim: int
    dtype: str  # "f32" | "bf16" | "i8"

    @property
    def torch_dtype(self) -> torch.dtype:
        return DTYPES[self.dtype]

    @property
    def elem_size(self) -> int:
        return {"f32": 4, "bf16": 2, "i8": 1}[self.dtype]

    @property
    def row_elems(self) -> int:
        """Elements of one token row (all kv heads)."""
        return self.num_kv_heads * self.head_dim

    @property
    def row_bytes(self) -> int:
        if self.dtype == "i8":
            return self.row_elems + (4 * self.num_kv_heads + 15) // 16 * 16
        return self.row_elems * self.elem_size

    @property
    def shape(self):
        if self.dtype == "i8":
            return (self.num_blocks, self.num_layers, self.block_size, self.row_bytes)
        return (self.num_blocks, self.num_layers, self.block_size,
                self.num_kv_heads, self.head_dim)

    @property
    def bytes_per_tensor(self) -> int:
        return self.num_blocks * self.num_layers * self.block_size * self.row_bytes


@dataclass
class Batch:
    """Per-sequence view of the cache: what a BlockTable holds (ch12 §2.2).

    ``block_tables[b, k]`` is the physical block holding logical block ``k`` of
    sequence ``b``; entries past the blocks the sequence spans are ``-1``.
    Logical token ``i`` of sequence ``b`` sits at in-table position
    ``offsets[b] + i``.  ``cu_seqlens`` is the packed output layout used by the
    gather (sequence ``b`` occupies rows ``cu_seqlens[b]:cu_seqlens[b+1]``).
    """

    block_tables: np.ndarray  # int32 [B, max_blocks]
    seq_lens: np.ndarray      # int32 [B]
    offsets: np.ndarray       # int32 [B]
    cu_seqlens: np.ndarray    # int64 [B+1]

    @property
    def batch(self) -> int:
        return int(self.seq_lens.shape[0])

    @property
    def max_blocks(self) -> int:
        return int(self.block_tables.shape[1])

    @property
    def total_tokens(self) -> int:
        return int(self.cu_seqlens[-1])


@dataclass
class TokenStream:
    """Tokens whose K/V rows are to be written into the pool.

    Token ``t`` is logical position ``token_pos[t]`` of sequence
    ``token_seq[t]`` of the accompanying :class:`Batch`; ``token_seq[t] == -1``
    marks a padding entry that must not be written.
    """

    token_seq: np.ndarray  # int32 [T]
    token_pos: np.ndarray  # int32 [T]

    @property
    def num_tokens(self) -> int:
        return int(self.token_seq.shape[0])

    @property
    def num_valid(self) -> int:
        return int((self.token_seq >= 0).sum())


@dataclass
class Workload:
    name: str
    description: str
    pool: PoolSpec
    layer: int
    seed: int
    batch: Batch                         # sequences read by gather / decode
    tokens: Optional[TokenStream] = None  # rows written by the scatter
    token_batch: Optional[Batch] = None   # tables the scatter tokens refer to
    num_q_heads: Optional[int] = None
    scale: Optional[float] = None
    k_boost_frac: float = 0.0            # fraction of pool rows whose K is x3
    k_boost: float = 3.0
    notes: dict = field(default_factory=dict)

    @property
    def scatter_batch(self) -> Batch:
        return self.token_batch if self.token_batch is not None else self.batch


# --------------------------------------------------------------------------
# index structure helpers
# --------------------------------------------------------------------------

def _span_blocks(seq_len: int, offset: int, block_size: int) -> int:
    if seq_len <= 0:
        return 0
    return -(-(offset + seq_len) // block_size)


def _pack(tables, seq_lens, offsets) -> Batch:
    B = len(tables)
    width = max([len(t) for t in tables] + [1])
    bt = np.full((B, width), -1, dtype=np.int32)
    for b, t in enumerate(tables):
        bt[b, :len(t)] = np.asarray(t, dtype=np.int32)
    lens = np.asarray(seq_lens, dtype=np.int32)
    offs = np.asarray(offsets, dtype=np.int32)
    cu = np.zeros(B + 1, dtype=np.int64)
    cu[1:] = np.cumsum(lens.astype(np.int64))
    return Batch(bt, lens, offs, cu)


def _all_tokens(batch: Batch) -> TokenStream:
    """Every token of every sequence, packed in sequence order."""
    seq = np.repeat(np.arange(batch.batch, dtype=np.int32), batch.seq_lens)
    pos = np.concatenate([np.arange(n, dtype=np.int32) for n in batch.seq_lens]
                         or [np.zeros(0, np.int32)])
    return TokenStream(seq.astype(np.int32), pos.astype(np.int32))


class FreeList:
    """FIFO free-block queue popped from the left (ch12 §2.3, FIFO allocation)."""

    def __init__(self, order):
        self.q = collections.deque(int(x) for x in order)

    def pop(self, n: int):
        if n > len(self.q):
            raise RuntimeError("free list exhausted")
        return [self.q.popleft() for _ in range(n)]


# --------------------------------------------------------------------------
# the five named workloads
# --------------------------------------------------------------------------

def _tiny(seed: int) -> Workload:
    spec = PoolSpec(64, 1, 16, 4, 64, "f32")
    rng = np.random.default_rng(seed)
    table = rng.permutation(spec.num_blocks)[:7]
    batch = _pack([table], [100], [0])
    return Workload(
        name="tiny", seed=seed, pool=spec, layer=0, batch=batch,
        tokens=_all_tokens(batch), num_q_heads=4, scale=1.0 / math.sqrt(64),
        description="pool 64x1x16x4x64 fp32; one sequence of 100 tokens over 7 "
                    "seeded-permutation blocks; scatter 100, gather [100,4,64], "
                    "decode with 4 query heads, scale 1/8")


def _gather_scatter(seed: int) -> Workload:
    spec = PoolSpec(16384, 32, 16, 8, 128, "bf16")
    rng = np.random.default_rng(seed)
    B = 32
    lens = rng.integers(512, 4096 + 1, size=B)
    free = FreeList(rng.permutation(spec.num_blocks))
    tables = [free.pop(_span_blocks(int(n), 0, spec.block_size)) for n in lens]
    batch = _pack(tables, lens, np.zeros(B, np.int32))
    return Workload(
        name="gather_scatter", seed=seed, pool=spec, layer=0, batch=batch,
        tokens=_all_tokens(batch),
        description="pool 16384x32x16x8x128 bf16 (layer 0); 32 sequences, "
                    "seq_len U[512,4096]; tables popped FIFO from a seeded "
                    "shuffled free list; scatter all tokens then gather each")


def _decode_gqa(seed: int) -> Workload:
    spec = PoolSpec(16384, 32, 16, 8, 128, "bf16")
    rng = np.random.default_rng(seed)
    B = 64
    lens = rng.integers(1024, 8192 + 1, size=B)
    # The last block of every sequence is private: distinct across the batch
    # and in no other sequence's table, so a decode-step append never hits the
    # same row twice and never writes a block another sequence reads in the
    # same step.  The other blocks are drawn per sequence without replacement
    # and may repeat across sequences (the batch spans more blocks than the
    # pool holds).
    last = rng.permutation(spec.num_blocks)[:B]
    tables = []
    for b in range(B):
        nblk = _span_blocks(int(lens[b]), 0, spec.block_size)
        others = rng.permutation(spec.num_blocks)
        others = others[~np.isin(others, last)][:nblk - 1]
        tables.append(list(others) + [int(last[b])])
    batch = _pack(tables, lens, np.zeros(B, np.int32))
    # one new token per sequence: its last logical position
    tokens = TokenStream(np.arange(B, dtype=np.int32), (lens - 1).astype(np.int32))
    return Workload(
        name="decode_gqa", seed=seed, pool=spec, layer=7, batch=batch,
        tokens=tokens, num_q_heads=32, scale=1.0 / math.sqrt(128),
        description="pool 16384x32x16x8x128 bf16 (layer 7), Hq=32 (GQA 4); "
                    "batch 64, seq_len U[1024,8192]; random non-contiguous "
                    "block tables; one query token per sequence")


def _long_splitk(seed: int) -> Workload:
    spec = PoolSpec(65536, 4, 16, 8, 128, "bf16")
    rng = np.random.default_rng(seed)
    B = 8
    lens = rng.integers(32768, 131072 + 1, size=B)
    free = FreeList(rng.permutation(spec.num_blocks))
    tables = [free.pop(_span_blocks(int(n), 0, spec.block_size)) for n in lens]
    batch = _pack(tables, lens, np.zeros(B, np.int32))
    tokens = TokenStream(np.arange(B, dtype=np.int32), (lens - 1).astype(np.int32))
    return Workload(
        name="long_splitk", seed=seed, pool=spec, layer=2, batch=batch,
        tokens=tokens, num_q_heads=32, scale=1.0 / math.sqrt(128),
        k_boost_frac=0.01,
        description="pool 65536x4x16x8x128 bf16 (layer 2), Hq=32; batch 8, "
                    "seq_len U[32768,131072]; tables from one seeded "
                    "permutation; K x3 on 1% of pool rows (peaked softmax)")


def _prefix_mix(seed: int) -> Workload:
    spec = PoolSpec(32768, 8, 16, 8, 128, "bf16")
    rng = np.random.default_rng(seed)
    bs = spec.block_size
    free = FreeList(rng.permutation(spec.num_blocks))
    prefix = free.pop(64)
    B = 256
    offs = rng.integers(0, bs, size=B)
    suffix = rng.integers(16, 2048 + 1, size=B)
    tables, lens = [], []
    for b in range(B):
        # tokens start at row offs[b] of prefix block 0 and run to the end of
        # the 64-block prefix; the private suffix starts on a fresh block
        lens.append(64 * bs - int(offs[b]) + int(suffix[b]))
        tables.append(prefix + free.pop(_span_blocks(int(suffix[b]), 0, bs)))
    batch = _pack(tables, lens, offs)
    # prefill scatter: 8192 entries, each padding with probability 0.1; the
    # valid entries, in order, fill 8 new prompts on freshly popped blocks
    T = 8192
    pad = rng.random(T) < 0.1
    n_valid = int((~pad).sum())
    cuts = np.sort(rng.choice(np.arange(1, n_valid), size=7, replace=False))
    plens = np.diff(np.concatenate([[0], cuts, [n_valid]])).astype(np.int32)
    ptables = [free.pop(_span_blocks(int(n), 0, bs)) for n in plens]
    pbatch = _pack(ptables, plens, np.zeros(len(plens), np.int32))
    seq = np.full(T, -1, np.int32)
    pos = np.full(T, -1, np.int32)
    valid = _all_tokens(pbatch)
    seq[~pad] = valid.token_seq
    pos[~pad] = valid.token_pos
    return Workload(
        name="prefix_mix", seed=seed, pool=spec, layer=0, batch=batch,
        tokens=TokenStream(seq, pos), token_batch=pbatch, num_q_heads=32,
        scale=1.0 / math.sqrt(128),
        notes={"prefix_blocks": prefix},
        description="pool 32768x8x16x8x128 bf16 (layer 0), Hq=32; 256 decode "
                    "sequences sharing a 64-block prefix, first-block offset "
                    "U[0,15], private suffix U[16,2048]; prefill scatter of 8192 "
                    "entries with ~10% padding (-1)")


CONFIGS = {
    "tiny": (_tiny, 0),
    "gather_scatter": (_gather_scatter, 1),
    "decode_gqa": (_decode_gqa, 2),
    "long_splitk": (_long_splitk, 3),
    "prefix_mix": (_prefix_mix, 4),
}


def make_workload(name: str, seed: Optional[int] = None) -> Workload:
    fn, default_seed = CONFIGS[name]
    return fn(default_seed if seed is None else seed)


def small_workload(*, seed: int, num_blocks: int = 64, num_layers: int = 2,
                   block_size: int = 16, num_kv_heads: int = 2, head_dim: int = 64,
                   dtype: str = "bf16", batch: int = 3, min_len: int = 0,
                   max_len: int = 100, offsets: bool = True, layer: int = 1,
                   num_q_heads: Optional[int] = None, shared_prefix: int = 0,
                   lens=None) -> Workload:
    """A small seeded workload for sweeps: ragged lengths, optional offsets,
    optional shared prefix blocks, tables from a FIFO shuffled free list."""
    spec = PoolSpec(num_blocks, num_layers, block_size, num_kv_heads, head_dim, dtype)
    rng = np.random.default_rng(seed)
    if lens is None:
        lens = rng.integers(min_len, max_len + 1, size=batch)
    lens = np.asarray(lens, dtype=np.int64)
    batch = len(lens)
    offs = (rng.integers(0, block_size, size=batch) if offsets
            else np.zeros(batch, np.int64))
    offs = np.where(lens > 0, offs, 0)
    free = FreeList(rng.permutation(num_blocks))
    prefix = free.pop(shared_prefix) if shared_prefix else []
    tables = []
    for b in range(batch):
        nblk = _span_blocks(int(lens[b]), int(offs[b]), block_size)
        own = max(nblk - len(prefix), 0)
        tables.append((prefix[:nblk] if prefix else []) + free.pop(own))
    bt = _pack(tables, lens, offs)
    hq = num_q_heads if num_q_heads is not None else num_kv_heads
    return Workload(
        name="small", seed=seed, pool=spec, layer=layer, batch=bt,
        tokens=_all_tokens(bt), num_q_heads=hq,
        scale=1.0 / math.sqrt(head_dim), description="small sweep case")


# --------------------------------------------------------------------------
# bulk values
# --------------------------------------------------------------------------

_CHUNK_BLOCKS = 2048


def new_pool(spec: PoolSpec, device) -> tuple:
    """Zeroed K and V pool tensors of ``spec``'s shape on ``device``."""
    k = torch.zeros(spec.shape, dtype=spec.torch_dtype, device=device)
    v = torch.zeros(spec.shape, dtype=spec.torch_dtype, device=device)
    return k, v


def fill_pool(k_cache: torch.Tensor, v_cache: torch.Tensor, spec: PoolSpec,
              layer: int, seed: int, k_boost_frac: float = 0.0,
              k_boost: float = 3.0) -> None:
    """Fill one layer of both pools with N(0,1) drawn in fp32 on the pool's
    device, in fixed chunks of blocks (the stream does not depend on memory),
    then round once to the pool dtype.  With ``k_boost_frac`` > 0, exactly
    ``round(frac * N * bs)`` seeded token rows of K are multiplied by
    ``k_boost`` in fp32 before rounding."""
    dev = k_cache.device
    g = torch.Generator(device=dev)
    g.manual_seed(seed * 7919 + 17)
    N, bs = spec.num_blocks, spec.block_size
    boost = None
    if k_boost_frac > 0:
        rng = np.random.default_rng(seed * 104729 + 3)
        nrows = N * bs
        pick = rng.permutation(nrows)[:int(round(k_boost_frac * nrows))]
        mask = np.zeros(nrows, dtype=bool)
        mask[pick] = True
        boost = torch.from_numpy(mask.reshape(N, bs)).to(dev)
    row_shape = (spec.num_kv_heads, spec.head_dim)
    for lo in range(0, N, _CHUNK_BLOCKS):
        hi = min(N, lo + _CHUNK_BLOCKS)
        kk = torch.randn((hi - lo, bs) + row_shape, generator=g, device=dev,
                         dtype=torch.float32)
        if boost is not None:
            kk = torch.where(boost[lo:hi, :, None, None], kk * k_boost, kk)
        k_cache[lo:hi, layer].copy_(kk.to(spec.torch_dtype))
        vv = torch.randn((hi - lo, bs) + row_shape, generator=g, device=dev,
                         dtype=torch.float32)
        v_cache[lo:hi, layer].copy_(vv.to(spec.torch_dtype))


def fill_pool_i8(k_cache: torch.Tensor, v_cache: torch.Tensor, spec: PoolSpec,
                 layer: int, seed: int, k_boost_frac: float = 0.0,
                 k_boost: float = 3.0) -> None:
    """Fill one layer of two int8 pools with seeded random rows: codes are
    N(0,1) * 42 rounded and clipped to [-127, 127] (the spread of absmax-coded
    Gaussian rows), stored as the bytes code + 128, scales are uniform in
    [0.01, 0.04] (a Gaussian head's absmax / 127), padding bytes are random.  With ``k_boost_frac`` > 0 the
    K scales of that fraction of token rows are multiplied by ``k_boost``.
    Drawn on the pool's device in fixed chunks of blocks."""
    dev = k_cache.device
    g = torch.Generator(device=dev)
    g.manual_seed(seed * 7919 + 29)
    N, bs, H, D = spec.num_blocks, spec.block_size, spec.num_kv_heads, spec.head_dim
    R = spec.row_bytes
    boost = None
    if k_boost_frac > 0:
        rng = np.random.default_rng(seed * 104729 + 5)
        nrows = N * bs
        pick = rng.permutation(nrows)[:int(round(k_boost_frac * nrows))]
        mask = np.zeros(nrows, dtype=bool)
        mask[pick] = True
        boost = torch.from_numpy(mask.reshape(N, bs)).to(dev)
    for lo in range(0, N, _CHUNK_BLOCKS):
        hi = min(N, lo + _CHUNK_BLOCKS)
        for which, pool in ((0, k_cache), (1, v_cache)):
            rows = torch.randint(0, 256, (hi - lo, bs, R), generator=g, device=dev,
                                 dtype=torch.uint8)
            codes = torch.randn((hi - lo, bs, H * D), generator=g, device=dev) * 42.0
            codes = codes.round().clamp_(-127, 127).to(torch.int8)
            sc = torch.rand((hi - lo, bs, H), generator=g, device=dev) * 0.03 + 0.01
            if which == 0 and boost is not None:
                sc = torch.where(boost[lo:hi, :, None], sc * k_boost, sc)
            rows[:, :, :H * D] = (codes.to(torch.int16) + 128).to(torch.uint8)  # offset binary
            rows[:, :, H * D:H * D + 4 * H] = sc.contiguous().view(torch.uint8).view(
                hi - lo, bs, 4 * H)
            pool[lo:hi, layer].copy_(rows)


def rand_rows(shape, dtype: str, seed: int, device) -> torch.Tensor:
    """N(0,1) drawn in fp32 on ``device`` and rounded once to ``dtype``."""
    g = torch.Generator(device=device)
    g.manual_seed(seed * 6151 + 5)
    x = torch.randn(shape, generator=g, device=device, dtype=torch.float32)
    return x.to(DTYPES[dtype])


def to_numpy_bits(t: torch.Tensor) -> np.ndarray:
    """Host numpy copy of ``t``: fp32 as float32, bf16 as its uint16 bits."""
    t = t.detach().cpu().contiguous()
    if t.dtype == torch.bfloat16:
        return t.view(torch.int16).numpy().view(np.uint16)
    if t.dtype in (torch.float32, torch.uint8):
        return t.numpy()
    raise TypeError(f"unsupported dtype {t.dtype}")
