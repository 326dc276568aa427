"""GPU parity: the CUDA path through the C ABI against the oracle on the same
seeded inputs.  Index work and copies must match bit for bit; attention must
agree within max-abs 2e-2 for bf16 and 1e-5 for fp32.

The five named workloads run at full size (decode outputs of the two largest
are sampled (b, h) pairs the oracle computes one by one); the sweeps use small
pools that span several blocks and stages with ragged tails."""

import math
import zlib

import numpy as np
import pytest
import torch

import oracle
import paged_kv_cache_blk_gb300 as pkv
from workloads import (PoolSpec, TokenStream, make_workload, rand_rows, small_workload,
                       to_numpy_bits)

from gpu_util import (dev_batch, gpu_decode, gpu_gather, gpu_slots, host_layer, make_pools,
                      max_abs, need_gpu, oracle_slots, tol, widen_out)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def dev():
    d = need_gpu()
    pkv.set_decode_ctas(0)
    pkv.set_validate(False)
    yield d
    torch.cuda.empty_cache()


def _scatter_case(w, dev, batch, tokens, check_layer=True):
    """slots + scatter on the GPU and in the oracle; returns pools and host copies."""
    k, v = make_pools(w, dev)
    pool = pkv.Pool(k, v)
    kh0, vh0 = host_layer(k, w.layer), host_layer(v, w.layer)
    T = tokens.num_tokens
    row = (w.pool.num_kv_heads, w.pool.head_dim)
    k_new = rand_rows((T,) + row, w.pool.dtype, w.seed * 31 + 1, dev)
    v_new = rand_rows((T,) + row, w.pool.dtype, w.seed * 31 + 2, dev)
    sm = gpu_slots(pool, batch, tokens, dev)
    pkv.write_slots(pool, w.layer, k_new, v_new, sm)
    sm_ref = oracle_slots(w, batch, tokens)
    assert np.array_equal(sm.cpu().numpy(), sm_ref), "slot mapping differs"
    oracle.write_slots(kh0, vh0, 0, to_numpy_bits(k_new), to_numpy_bits(v_new), sm_ref)
    if check_layer:
        assert np.array_equal(host_layer(k, w.layer), kh0), "K layer differs after scatter"
        assert np.array_equal(host_layer(v, w.layer), vh0), "V layer differs after scatter"
    return pool, k, v, kh0, vh0


# ---------------------------------------------------------------------------
# the five named workloads
# ---------------------------------------------------------------------------

def test_tiny_full_path(dev):
    w = make_workload("tiny")
    pool, k, v, kh, vh = _scatter_case(w, dev, w.batch, w.tokens)
    ko, vo = gpu_gather(pool, w.layer, w.batch, dev)
    kr, vr = oracle.gather_batch(kh, vh, 0, w.batch.block_tables, w.batch.seq_lens,
                                 w.batch.offsets)
    assert ko.shape == (100, 4, 64)
    assert np.array_equal(to_numpy_bits(ko), kr) and np.array_equal(to_numpy_bits(vo), vr)
    q = rand_rows((1, w.num_q_heads, w.pool.head_dim), "f32", 77, dev)
    out = gpu_decode(pool, w.layer, q, w.scale, w.batch, dev)
    ref = oracle.decode_attention(kh, vh, 0, to_numpy_bits(q), w.batch.block_tables,
                                  w.batch.seq_lens, w.batch.offsets, w.scale)
    assert max_abs(widen_out(out), ref) <= 1e-5


def test_gather_scatter_full(dev):
    w = make_workload("gather_scatter")
    pool, k, v, kh, vh = _scatter_case(w, dev, w.batch, w.tokens)
    ko, vo = gpu_gather(pool, w.layer, w.batch, dev)
    kr, vr = oracle.gather_batch(kh, vh, 0, w.batch.block_tables, w.batch.seq_lens,
                                 w.batch.offsets)
    assert np.array_equal(to_numpy_bits(ko), kr)
    assert np.array_equal(to_numpy_bits(vo), vr)
    del pool, k, v, ko, vo
    torch.cuda.empty_cache()


def test_decode_gqa_full(dev):
    w = make_workload("decode_gqa")
    k, v = make_pools(w, dev)
    pool = pkv.Pool(k, v)
    q = rand_rows((w.batch.batch, w.num_q_heads, w.pool.head_dim), "bf16", 91, dev)
    out = gpu_decode(pool, w.layer, q, w.scale, w.batch, dev)
    kh, vh = host_layer(k, w.layer), host_layer(v, w.layer)
    ref = oracle.decode_attention(kh, vh, 0, to_numpy_bits(q), w.batch.block_tables,
                                  w.batch.seq_lens, w.batch.offsets, w.scale)
    assert max_abs(widen_out(out), ref) <= 2e-2
    # the decode step: append one token per sequence, then attend
    T = w.tokens.num_tokens
    k_new = rand_rows((T, 8, 128), "bf16", 92, dev)
    v_new = rand_rows((T, 8, 128), "bf16", 93, dev)
    sm = gpu_slots(pool, w.batch, w.tokens, dev)
    pkv.write_slots(pool, w.layer, k_new, v_new, sm)
    out2 = gpu_decode(pool, w.layer, q, w.scale, w.batch, dev)
    sm_ref = oracle_slots(w, w.batch, w.tokens)
    assert np.array_equal(sm.cpu().numpy(), sm_ref)
    oracle.write_slots(kh, vh, 0, to_numpy_bits(k_new), to_numpy_bits(v_new), sm_ref)
    ref2 = oracle.decode_attention(kh, vh, 0, to_numpy_bits(q), w.batch.block_tables,
                                   w.batch.seq_lens, w.batch.offsets, w.scale)
    assert max_abs(widen_out(out2), ref2) <= 2e-2
    assert np.array_equal(host_layer(k, w.layer), kh)
    del pool, k, v
    torch.cuda.empty_cache()


def test_long_splitk_full_sampled(dev):
    w = make_workload("long_splitk")
    k, v = make_pools(w, dev)
    pool = pkv.Pool(k, v)
    B = w.batch.batch
    q = rand_rows((B, w.num_q_heads, w.pool.head_dim), "bf16", 95, dev)
    out = gpu_decode(pool, w.layer, q, w.scale, w.batch, dev)
    assert torch.isfinite(out.float()).all()
    kh, vh = host_layer(k, w.layer), host_layer(v, w.layer)
    pairs = [(b, h) for b in range(B) for h in (0, 5, 18, 31)]
    ref = oracle.decode_attention_pairs(kh, vh, 0, to_numpy_bits(q), w.batch.block_tables,
                                        w.batch.seq_lens, w.batch.offsets, w.scale, pairs)
    got = widen_out(out)
    err = max(max_abs(got[b, h], r) for (b, h), r in ref.items())
    assert err <= 2e-2, err
    del pool, k, v
    torch.cuda.empty_cache()


def test_prefix_mix_full(dev):
    w = make_workload("prefix_mix")
    # prefill scatter with ~10% padding: whole layer bit-exact
    pool, k, v, kh, vh = _scatter_case(w, dev, w.token_batch, w.tokens)
    # decode of the 256 prefix-sharing sequences (offsets in the first block)
    B = w.batch.batch
    q = rand_rows((B, w.num_q_heads, w.pool.head_dim), "bf16", 97, dev)
    out = gpu_decode(pool, w.layer, q, w.scale, w.batch, dev)
    pairs = [(b, (7 * b) % w.num_q_heads) for b in range(0, B, 3)]
    ref = oracle.decode_attention_pairs(kh, vh, 0, to_numpy_bits(q), w.batch.block_tables,
                                        w.batch.seq_lens, w.batch.offsets, w.scale, pairs)
    got = widen_out(out)
    err = max(max_abs(got[b, h], r) for (b, h), r in ref.items())
    assert err <= 2e-2, err
    # gather of the first 32 sequences (first-block offsets honoured)
    sub = _sub_batch(w.batch, 32)
    ko, vo = gpu_gather(pool, w.layer, sub, dev)
    kr, vr = oracle.gather_batch(kh, vh, 0, sub.block_tables, sub.seq_lens, sub.offsets)
    assert np.array_equal(to_numpy_bits(ko), kr) and np.array_equal(to_numpy_bits(vo), vr)
    del pool, k, v
    torch.cuda.empty_cache()


def _sub_batch(batch, n):
    from workloads.gen import Batch
    return Batch(batch.block_tables[:n].copy(), batch.seq_lens[:n].copy(),
                 batch.offsets[:n].copy(), batch.cu_seqlens[:n + 1].copy())


# ---------------------------------------------------------------------------
# sweeps on small pools
# ---------------------------------------------------------------------------

SWEEP = [
    # dtype, head_dim, num_kv_heads, group, block_size, layer, max_len
    ("bf16", 128, 8, 4, 16, 1, 120),
    ("bf16", 128, 8, 1, 16, 0, 90),
    ("bf16", 128, 8, 2, 16, 2, 70),
    ("bf16", 128, 8, 8, 16, 1, 70),
    ("bf16", 64, 8, 4, 16, 1, 100),
    ("bf16", 128, 4, 4, 16, 1, 100),
    ("bf16", 128, 2, 8, 16, 0, 100),
    ("bf16", 64, 1, 8, 16, 2, 100),
    ("bf16", 128, 1, 1, 16, 1, 60),
    ("bf16", 128, 8, 4, 8, 1, 100),
    ("bf16", 128, 8, 4, 32, 1, 140),
    ("bf16", 128, 8, 4, 4, 1, 60),
    ("bf16", 64, 4, 2, 64, 0, 200),
    ("bf16", 128, 8, 4, 1, 1, 20),
    # boxes taller than a stage (kv heads x stage rows < 8): the extra rows
    # come from the next layer, or from past the pool on the last layer
    ("bf16", 64, 1, 4, 2, 2, 30),
    ("bf16", 128, 2, 4, 1, 2, 20),
    ("bf16", 64, 1, 8, 4, 0, 40),
    ("bf16", 128, 1, 2, 1, 2, 12),
    ("f32", 64, 4, 1, 16, 0, 100),
    ("f32", 128, 8, 4, 16, 1, 100),
    ("f32", 128, 2, 2, 8, 1, 80),
    ("f32", 64, 8, 8, 16, 1, 70),
    ("f32", 64, 1, 4, 32, 2, 90),
]


@pytest.mark.parametrize("dtype,D,hkv,G,bs,layer,max_len", SWEEP,
                         ids=["-".join(map(str, c)) for c in SWEEP])
def test_small_path_sweep(dev, dtype, D, hkv, G, bs, layer, max_len):
    seed = zlib.crc32(repr((dtype, D, hkv, G, bs, layer)).encode()) % 1000
    w = small_workload(seed=seed, num_blocks=max(64, 4 * (max_len // bs + 2)), num_layers=3,
                       block_size=bs, num_kv_heads=hkv, head_dim=D, dtype=dtype, batch=5,
                       min_len=0, max_len=max_len, layer=layer, num_q_heads=hkv * G)
    pool, k, v, kh, vh = _scatter_case(w, dev, w.batch, w.tokens)
    ko, vo = gpu_gather(pool, w.layer, w.batch, dev)
    kr, vr = oracle.gather_batch(kh, vh, 0, w.batch.block_tables, w.batch.seq_lens,
                                 w.batch.offsets)
    assert np.array_equal(to_numpy_bits(ko), kr) and np.array_equal(to_numpy_bits(vo), vr)
    q = rand_rows((w.batch.batch, w.num_q_heads, D), dtype, seed + 5, dev)
    ref = oracle.decode_attention(kh, vh, 0, to_numpy_bits(q), w.batch.block_tables,
                                  w.batch.seq_lens, w.batch.offsets, w.scale)
    for ctas in (0, 1, 3):
        pkv.set_decode_ctas(ctas)
        try:
            out = gpu_decode(pool, w.layer, q, w.scale, w.batch, dev)
        finally:
            pkv.set_decode_ctas(0)
        assert max_abs(widen_out(out), ref) <= tol(dtype), ctas


@pytest.mark.parametrize("ctas", [1, 2, 3, 7, 64, 152, 500, 3000])
def test_decode_split_counts(dev, ctas):
    w = small_workload(seed=11, num_blocks=512, num_layers=2, block_size=16, num_kv_heads=8,
                       head_dim=128, dtype="bf16", batch=6, min_len=1, max_len=900,
                       num_q_heads=32, shared_prefix=3)
    k, v = make_pools(w, dev)
    pool = pkv.Pool(k, v)
    q = rand_rows((6, 32, 128), "bf16", 12, dev)
    ref = oracle.decode_attention(host_layer(k, w.layer), host_layer(v, w.layer), 0,
                                  to_numpy_bits(q), w.batch.block_tables, w.batch.seq_lens,
                                  w.batch.offsets, w.scale)
    pkv.set_decode_ctas(ctas)
    try:
        out = gpu_decode(pool, w.layer, q, w.scale, w.batch, dev)
    finally:
        pkv.set_decode_ctas(0)
    assert max_abs(widen_out(out), ref) <= 2e-2


def test_seq_len_and_offset_edges(dev):
    lens = [0, 1, 15, 16, 17, 31, 32, 33, 47, 48, 49, 0, 1, 2, 255]
    for seed in range(3):
        w = small_workload(seed=50 + seed, num_blocks=256, num_layers=1, block_size=16,
                           num_kv_heads=8, head_dim=128, dtype="bf16", lens=lens, layer=0,
                           num_q_heads=32)
        pool, k, v, kh, vh = _scatter_case(w, dev, w.batch, w.tokens)
        ko, vo = gpu_gather(pool, 0, w.batch, dev)
        kr, vr = oracle.gather_batch(kh, vh, 0, w.batch.block_tables, w.batch.seq_lens,
                                     w.batch.offsets)
        assert np.array_equal(to_numpy_bits(ko), kr) and np.array_equal(to_numpy_bits(vo), vr)
        q = rand_rows((len(lens), 32, 128), "bf16", seed, dev)
        out = gpu_decode(pool, 0, q, w.scale, w.batch, dev)
        ref = oracle.decode_attention(kh, vh, 0, to_numpy_bits(q), w.batch.block_tables,
                                      w.batch.seq_lens, w.batch.offsets, w.scale)
        assert max_abs(widen_out(out), ref) <= 2e-2
        assert torch.count_nonzero(out[0]) == 0           # seq_len 0 -> zeros


def test_every_offset_with_identity_table(dev):
    """Identity tables: gathered sequences are contiguous runs of the layer."""
    spec = PoolSpec(8, 2, 16, 2, 64, "bf16")
    from workloads.gen import _pack
    tables = [list(range(8))] * 16
    offs = list(range(16))
    lens = [8 * 16 - o for o in offs]
    batch = _pack(tables, lens, offs)
    k = rand_rows(spec.shape, "bf16", 3, dev)
    v = rand_rows(spec.shape, "bf16", 4, dev)
    pool = pkv.Pool(k, v)
    ko, vo = gpu_gather(pool, 1, batch, dev)
    flat = k[:, 1].reshape(8 * 16, 2, 64)
    for b, o in enumerate(offs):
        lo, hi = batch.cu_seqlens[b], batch.cu_seqlens[b + 1]
        assert torch.equal(ko[lo:hi], flat[o:])


def test_every_layer(dev):
    w = small_workload(seed=21, num_blocks=64, num_layers=4, block_size=16, num_kv_heads=4,
                       head_dim=128, dtype="bf16", batch=3, min_len=10, max_len=200,
                       num_q_heads=16)
    spec = w.pool
    k = rand_rows(spec.shape, "bf16", 1, dev)
    v = rand_rows(spec.shape, "bf16", 2, dev)
    pool = pkv.Pool(k, v)
    q = rand_rows((3, 16, 128), "bf16", 3, dev)
    for layer in range(spec.num_layers):
        out = gpu_decode(pool, layer, q, w.scale, w.batch, dev)
        ref = oracle.decode_attention(host_layer(k, layer), host_layer(v, layer), 0,
                                      to_numpy_bits(q), w.batch.block_tables, w.batch.seq_lens,
                                      w.batch.offsets, w.scale)
        assert max_abs(widen_out(out), ref) <= 2e-2, layer


def test_batch_larger_than_one_launch(dev):
    """More sequences than one partial-pass launch takes (2048): split on the host."""
    B = 2600
    w = small_workload(seed=31, num_blocks=4096, num_layers=1, block_size=16, num_kv_heads=2,
                       head_dim=64, dtype="bf16", batch=B, min_len=0, max_len=20, layer=0,
                       num_q_heads=4, offsets=True)
    k, v = make_pools(w, dev)
    pool = pkv.Pool(k, v)
    q = rand_rows((B, 4, 64), "bf16", 32, dev)
    out = gpu_decode(pool, 0, q, w.scale, w.batch, dev)
    ref = oracle.decode_attention(host_layer(k, 0), host_layer(v, 0), 0, to_numpy_bits(q),
                                  w.batch.block_tables, w.batch.seq_lens, w.batch.offsets,
                                  w.scale)
    assert max_abs(widen_out(out), ref) <= 2e-2


def test_peaked_softmax(dev):
    """A key far above the rest dominates: the output is (nearly) its value row."""
    w = small_workload(seed=41, num_blocks=64, num_layers=1, block_size=16, num_kv_heads=8,
                       head_dim=128, dtype="bf16", lens=[300, 17], layer=0, num_q_heads=32,
                       offsets=False)
    k, v = make_pools(w, dev)
    q = rand_rows((2, 32, 128), "bf16", 42, dev)
    # plant K rows proportional to q for kv head 0 at token 123 of sequence 0
    blk = int(w.batch.block_tables[0, 123 // 16])
    k[blk, 0, 123 % 16, 0] = (q[0, 0].float() * 4).to(torch.bfloat16)
    pool = pkv.Pool(k, v)
    out = gpu_decode(pool, 0, q, 1.0, w.batch, dev)
    ref = oracle.decode_attention(host_layer(k, 0), host_layer(v, 0), 0, to_numpy_bits(q),
                                  w.batch.block_tables, w.batch.seq_lens, w.batch.offsets, 1.0)
    assert max_abs(widen_out(out), ref) <= 2e-2


def test_nondefault_stream(dev):
    w = small_workload(seed=61, num_blocks=128, num_layers=2, block_size=16, num_kv_heads=8,
                       head_dim=128, dtype="bf16", batch=4, min_len=1, max_len=300,
                       num_q_heads=32)
    k, v = make_pools(w, dev)
    pool = pkv.Pool(k, v)
    q = rand_rows((4, 32, 128), "bf16", 62, dev)
    s = torch.cuda.Stream(dev)
    with torch.cuda.stream(s):
        out = gpu_decode(pool, w.layer, q, w.scale, w.batch, dev)
    s.synchronize()
    ref = oracle.decode_attention(host_layer(k, w.layer), host_layer(v, w.layer), 0,
                                  to_numpy_bits(q), w.batch.block_tables, w.batch.seq_lens,
                                  w.batch.offsets, w.scale)
    assert max_abs(widen_out(out), ref) <= 2e-2


def test_decode_events_hook(dev):
    w = small_workload(seed=71, num_blocks=128, num_layers=1, block_size=16, num_kv_heads=8,
                       head_dim=128, dtype="bf16", batch=4, min_len=100, max_len=300,
                       num_q_heads=32, layer=0)
    k, v = make_pools(w, dev)
    pool = pkv.Pool(k, v)
    q = rand_rows((4, 32, 128), "bf16", 72, dev)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(); e1.record()
    pkv.set_decode_events(e0, e1)
    try:
        gpu_decode(pool, 0, q, w.scale, w.batch, dev)
    finally:
        pkv.set_decode_events(None, None)
    torch.cuda.synchronize()
    assert e0.elapsed_time(e1) > 0


def test_cuda_graph_replay_with_changing_inputs(dev):
    """A decode step captured once in a CUDA graph and replayed with new
    queries and new token rows each time must match the oracle every time
    (nothing launch-specific may be baked into the graph)."""
    w = small_workload(seed=91, num_blocks=256, num_layers=2, block_size=16, num_kv_heads=8,
                       head_dim=128, dtype="bf16", batch=6, min_len=40, max_len=900,
                       num_q_heads=32, offsets=True)
    k, v = make_pools(w, dev)
    pool = pkv.Pool(k, v)
    bt, lens, offs, _ = dev_batch(w.batch, dev)
    B = w.batch.batch
    # the step appends the last token of every sequence, then attends
    seq = torch.arange(B, dtype=torch.int32, device=dev)
    pos = lens - 1
    q = torch.empty((B, 32, 128), dtype=torch.bfloat16, device=dev)
    kn = torch.empty((B, 8, 128), dtype=torch.bfloat16, device=dev)
    vn = torch.empty_like(kn)
    out = torch.empty_like(q)
    slots = torch.empty(B, dtype=torch.int64, device=dev)
    ws = torch.empty(pkv.decode_workspace_size(B, 32, 128, dev), dtype=torch.uint8, device=dev)

    def step():
        pkv.build_slot_mapping(pool, bt, offs, seq, pos, slots)
        pkv.write_slots(pool, w.layer, kn, vn, slots)
        pkv.decode_attention(pool, w.layer, q, w.scale, bt, lens, offs, out, ws)

    q.copy_(rand_rows(q.shape, "bf16", 1, dev)); kn.copy_(rand_rows(kn.shape, "bf16", 2, dev))
    vn.copy_(rand_rows(vn.shape, "bf16", 3, dev))
    side = torch.cuda.Stream(dev)
    side.wait_stream(torch.cuda.current_stream(dev))
    with torch.cuda.stream(side):
        step()
    torch.cuda.current_stream(dev).wait_stream(side)
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        step()
    kh, vh = host_layer(k, w.layer), host_layer(v, w.layer)
    tokens = TokenStream(np.arange(B, dtype=np.int32), (w.batch.seq_lens - 1).astype(np.int32))
    sm_ref = oracle.build_slot_mapping(w.batch.block_tables, w.batch.offsets, tokens.token_seq,
                                       tokens.token_pos, 16)
    for r in range(4):
        q.copy_(rand_rows(q.shape, "bf16", 10 + r, dev))
        kn.copy_(rand_rows(kn.shape, "bf16", 20 + r, dev))
        vn.copy_(rand_rows(vn.shape, "bf16", 30 + r, dev))
        graph.replay()
        torch.cuda.synchronize()
        oracle.write_slots(kh, vh, 0, to_numpy_bits(kn), to_numpy_bits(vn), sm_ref)
        ref = oracle.decode_attention(kh, vh, 0, to_numpy_bits(q), w.batch.block_tables,
                                      w.batch.seq_lens, w.batch.offsets, w.scale)
        assert max_abs(widen_out(out), ref) <= 2e-2, r
