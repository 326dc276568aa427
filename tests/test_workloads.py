"""The seeded workload generators: determinism and the structure each named
workload promises (no pools are allocated here; index structure only)."""

import numpy as np
import torch

import oracle
from workloads import CONFIGS, make_workload, small_workload, rand_rows, fill_pool, PoolSpec


def _check_batch(w):
    bt = w.batch
    bs = w.pool.block_size
    assert bt.block_tables.dtype == np.int32 and bt.seq_lens.dtype == np.int32
    assert bt.cu_seqlens[0] == 0
    assert np.array_equal(np.diff(bt.cu_seqlens), bt.seq_lens)
    for b in range(bt.batch):
        nb = oracle.blocks_needed(int(bt.seq_lens[b]), bs, int(bt.offsets[b]))
        row = bt.block_tables[b]
        assert np.all(row[:nb] >= 0) and np.all(row[:nb] < w.pool.num_blocks)
        assert np.all(row[nb:] == -1)
        assert len(set(row[:nb].tolist())) == nb        # distinct within a sequence
        assert 0 <= bt.offsets[b] < bs
        assert bt.seq_lens[b] <= oracle.capacity(bt.max_blocks, bs, int(bt.offsets[b]))


def test_all_configs_deterministic_and_valid():
    for name in CONFIGS:
        a = make_workload(name)
        b = make_workload(name)
        assert np.array_equal(a.batch.block_tables, b.batch.block_tables)
        assert np.array_equal(a.batch.seq_lens, b.batch.seq_lens)
        _check_batch(a)
        if a.tokens is not None:
            assert np.array_equal(a.tokens.token_seq, b.tokens.token_seq)


def test_tiny_shape():
    w = make_workload("tiny")
    assert w.pool == PoolSpec(64, 1, 16, 4, 64, "f32")
    assert w.batch.seq_lens.tolist() == [100]
    assert (w.batch.block_tables[0] >= 0).sum() == 7
    assert w.tokens.num_tokens == 100 and w.num_q_heads == 4 and w.scale == 0.125


def test_gather_scatter_fifo_distinct():
    w = make_workload("gather_scatter")
    assert w.batch.batch == 32
    assert w.batch.seq_lens.min() >= 512 and w.batch.seq_lens.max() <= 4096
    used = w.batch.block_tables[w.batch.block_tables >= 0]
    assert len(np.unique(used)) == len(used)          # one free list, FIFO
    assert w.tokens.num_tokens == w.batch.total_tokens


def test_decode_gqa_last_blocks_private():
    w = make_workload("decode_gqa")
    bt = w.batch
    last = [bt.block_tables[b, oracle.blocks_needed(int(bt.seq_lens[b]), 16) - 1]
            for b in range(bt.batch)]
    assert len(set(last)) == bt.batch
    assert np.array_equal(w.tokens.token_pos, bt.seq_lens - 1)
    # no sequence reads a block that another sequence's new token goes into
    for b in range(bt.batch):
        n = oracle.blocks_needed(int(bt.seq_lens[b]), 16)
        others = set(bt.block_tables[b, :n - 1].tolist())
        assert not (others & (set(last) - {last[b]})), b


def test_long_splitk_fits_pool():
    w = make_workload("long_splitk")
    used = w.batch.block_tables[w.batch.block_tables >= 0]
    assert len(np.unique(used)) == len(used) <= w.pool.num_blocks
    assert w.k_boost_frac == 0.01


def test_prefix_mix_structure():
    w = make_workload("prefix_mix")
    bt = w.batch
    prefix = w.notes["prefix_blocks"]
    assert np.all(bt.block_tables[:, :64] == np.array(prefix))
    assert bt.offsets.min() >= 0 and bt.offsets.max() <= 15
    sfx = bt.seq_lens - (1024 - bt.offsets)
    assert sfx.min() >= 16 and sfx.max() <= 2048
    ts = w.tokens
    assert ts.num_tokens == 8192
    frac = 1 - ts.num_valid / ts.num_tokens
    assert 0.08 < frac < 0.12
    # prefill blocks are fresh: disjoint from every decode block
    pb = w.token_batch.block_tables
    dec = set(bt.block_tables[bt.block_tables >= 0].tolist())
    assert not dec & set(pb[pb >= 0].tolist())
    _ = oracle.build_slot_mapping(w.token_batch.block_tables, w.token_batch.offsets,
                                  ts.token_seq, ts.token_pos, 16)


def test_small_workload_sweeps():
    for seed in range(5):
        w = small_workload(seed=seed, shared_prefix=2, min_len=0, max_len=60)
        _check_batch(w)


def test_fill_pool_and_rows_are_seeded():
    spec = PoolSpec(8, 2, 4, 2, 8, "bf16")
    k1 = torch.zeros(spec.shape, dtype=torch.bfloat16)
    v1 = torch.zeros_like(k1)
    k2, v2 = torch.zeros_like(k1), torch.zeros_like(k1)
    fill_pool(k1, v1, spec, 1, seed=3, k_boost_frac=0.25)
    fill_pool(k2, v2, spec, 1, seed=3, k_boost_frac=0.25)
    assert torch.equal(k1, k2) and torch.equal(v1, v2)
    assert k1[:, 0].abs().sum() == 0 and k1[:, 1].abs().sum() > 0
    assert torch.equal(rand_rows((5, 2, 8), "f32", 1, "cpu"), rand_rows((5, 2, 8), "f32", 1, "cpu"))
