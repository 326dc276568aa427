"""GPU parity for shared-prefix decode (pkv_decode_attention_shared_prefix).

The result must be the oracle's decode attention over each sequence's tokens
(max-abs 2e-2 for bf16), exactly as for pkv_decode_attention: the call only
reads the shared prefix blocks once for the whole batch.  Cases: ragged
lengths with first-block offsets, sequences that end inside the prefix or
are empty, every head grouping and block size the prefix pass supports,
prefixes split over many CTAs, a prefix that covers every token, the
prefix-mix workload at full size, the validate-mode contract checks, and
shapes that take the plain path."""

import numpy as np
import pytest
import torch

import oracle
import paged_kv_cache_blk_gb300 as pkv
from paged_kv_cache_blk_gb300 import PkvError
from workloads import PoolSpec, fill_pool, make_workload, new_pool, rand_rows, to_numpy_bits
from workloads.gen import FreeList, _pack

from gpu_util import dev_batch, gpu_decode, host_layer, max_abs, need_gpu, widen_out

pytestmark = pytest.mark.gpu

TOL = 2e-2


@pytest.fixture(scope="module")
def dev():
    d = need_gpu()
    pkv.set_validate(False)
    pkv.set_decode_ctas(0)
    pkv.device_error(clear=True)
    return d


def _case(dev, seed, lens, P, bs=16, hkv=8, G=4, offsets=True, layer=1, dtype="bf16",
          D=128):
    """A batch whose tables start with the same P prefix blocks (sequence 0
    spans all of them); each sequence then has private blocks."""
    rng = np.random.default_rng(seed)
    lens = np.asarray(lens, np.int64)
    B = len(lens)
    offs = rng.integers(0, bs, size=B) if offsets else np.zeros(B, np.int64)
    offs = np.where(lens > 0, offs, 0)
    span = [-(-(int(o) + int(L)) // bs) if L > 0 else 0 for o, L in zip(offs, lens)]
    assert span[0] >= P
    N = P + sum(max(0, s - P) for s in span) + 16
    free = FreeList(rng.permutation(N))
    prefix = free.pop(P)
    tables = [prefix[:s] + free.pop(max(0, s - P)) for s in span]
    batch = _pack(tables, lens, offs)
    spec = PoolSpec(N, 2, bs, hkv, D, dtype)
    k, v = new_pool(spec, dev)
    fill_pool(k, v, spec, layer, seed)
    q = rand_rows((B, hkv * G, D), dtype, seed + 7, dev)
    return spec, batch, k, v, q, layer


def _run(dev, batch, k, v, q, layer, P, scale=128 ** -0.5):
    pool = pkv.Pool(k, v)
    bt, lens, offs, _ = dev_batch(batch, dev)
    out = torch.full_like(q, float("nan"))
    ws = torch.empty(pkv.decode_shared_prefix_workspace_size(pool, batch.batch, q.shape[1], P),
                     dtype=torch.uint8, device=dev)
    pkv.decode_attention_shared_prefix(pool, layer, q, scale, bt, lens, offs, P, out, ws)
    torch.cuda.synchronize()
    return pool, out


def _oracle(batch, k, v, q, layer, scale=128 ** -0.5):
    return oracle.decode_attention(host_layer(k, layer), host_layer(v, layer), 0,
                                   to_numpy_bits(q), batch.block_tables, batch.seq_lens,
                                   batch.offsets, scale)


CASES = [
    # lens, P, bs, hkv, G
    ([900, 300, 257, 1000, 129, 700, 512, 1, 800, 64, 999, 300], 8, 16, 8, 4),
    ([700] + [40, 0, 130, 5, 16, 17, 127, 128, 129] * 3, 8, 16, 8, 4),   # inside the prefix, empty
    ([2100] + list(range(100, 3000, 41)), 40, 16, 8, 4),                    # 72 sequences, splits
    ([800, 600, 1500], 16, 16, 2, 8),
    ([800, 600, 1500, 90], 16, 16, 4, 2),
    ([800, 600, 1500, 90], 16, 16, 8, 1),
    ([640, 300, 999], 20, 32, 8, 4),
    ([640, 300, 999], 40, 8, 8, 4),
    ([1200, 333, 1100], 9, 128, 2, 4),
    ([1024, 1000, 1010, 1023], 64, 16, 8, 4),                               # prefix covers all
]


@pytest.mark.parametrize("lens,P,bs,hkv,G", CASES,
                         ids=[f"B{len(c[0])}-P{c[1]}-bs{c[2]}-H{c[3]}G{c[4]}" for c in CASES])
def test_shared_prefix_matches_oracle(dev, lens, P, bs, hkv, G):
    seed = 300 + len(lens) + P + bs + G
    spec, batch, k, v, q, layer = _case(dev, seed, lens, P, bs=bs, hkv=hkv, G=G)
    pool, out = _run(dev, batch, k, v, q, layer, P)
    got = widen_out(out)
    assert np.isfinite(got).all()
    assert max_abs(got, _oracle(batch, k, v, q, layer)) <= TOL
    # and the plain decode path of the same batch agrees
    ref = gpu_decode(pool, layer, q, 128 ** -0.5, batch, dev)
    assert max_abs(got, widen_out(ref)) <= TOL
    assert pkv.device_error(clear=True) == "PKV_OK"


def test_shared_prefix_forced_grids(dev):
    """The suffix pass split over 1, 3 and 997 CTAs (segments merged with the
    prefix states in every arrangement)."""
    lens = [1500, 700, 33, 1200, 260]
    spec, batch, k, v, q, layer = _case(dev, 341, lens, 12)
    want = _oracle(batch, k, v, q, layer)
    for ctas in (1, 3, 997):
        pkv.set_decode_ctas(ctas)
        try:
            _, out = _run(dev, batch, k, v, q, layer, 12)
        finally:
            pkv.set_decode_ctas(0)
        assert max_abs(widen_out(out), want) <= TOL, ctas


def test_shared_prefix_zero_prefix_and_plain_shapes(dev):
    lens = [300, 50, 129]
    spec, batch, k, v, q, layer = _case(dev, 351, lens, 4)
    _, out = _run(dev, batch, k, v, q, layer, 0)          # no prefix: the plain path
    assert max_abs(widen_out(out), _oracle(batch, k, v, q, layer)) <= TOL
    # fp32 pools and head_dim 64 take the plain path (same result)
    spec, batch, k, v, q, layer = _case(dev, 352, lens, 4, dtype="f32", D=64, hkv=4, G=2)
    _, out = _run(dev, batch, k, v, q, layer, 4, scale=64 ** -0.5)
    want = _oracle(batch, k, v, q, layer, scale=64 ** -0.5)
    assert max_abs(widen_out(out), want) <= 1e-5


def test_shared_prefix_validate_mode(dev):
    lens = [600, 300, 200]
    spec, batch, k, v, q, layer = _case(dev, 361, lens, 8)
    pool = pkv.Pool(k, v)
    bt, lens_t, offs, _ = dev_batch(batch, dev)
    out = torch.zeros_like(q)
    ws = torch.empty(pkv.decode_shared_prefix_workspace_size(pool, 3, q.shape[1], 8),
                     dtype=torch.uint8, device=dev)
    pkv.set_validate(True)
    try:
        pkv.decode_attention_shared_prefix(pool, layer, q, 128 ** -0.5, bt, lens_t, offs, 8,
                                           out, ws)
        torch.cuda.synchronize()
        bad = bt.clone()
        bad[1, 3] = int(batch.block_tables[0, 8])        # disagrees with row 0 in the prefix
        with pytest.raises(PkvError) as e:
            pkv.decode_attention_shared_prefix(pool, layer, q, 128 ** -0.5, bad, lens_t, offs, 8,
                                               out, ws)
        assert e.value.name == "PKV_ERR_INDEX"
        with pytest.raises(PkvError) as e:                 # more prefix blocks than the table
            pkv.decode_attention_shared_prefix(pool, layer, q, 128 ** -0.5, bt, lens_t, offs,
                                               bt.shape[1] + 1, out, ws)
        assert e.value.name == "PKV_ERR_INVALID_ARG"
        small = ws[:64]
        with pytest.raises(PkvError) as e:
            pkv.decode_attention_shared_prefix(pool, layer, q, 128 ** -0.5, bt, lens_t, offs, 8,
                                               out, small)
        assert e.value.name == "PKV_ERR_WORKSPACE"
    finally:
        pkv.set_validate(False)
        pkv.device_error(clear=True)


def test_shared_prefix_prefix_mix_full(dev):
    """The prefix-mix workload at full size (256 sequences, one 64-block
    prefix, offsets U[0,15]): sampled (b, h) against the oracle, every output
    against the plain decode path."""
    w = make_workload("prefix_mix")
    k, v = new_pool(w.pool, dev)
    fill_pool(k, v, w.pool, w.layer, w.seed)
    B = w.batch.batch
    q = rand_rows((B, w.num_q_heads, w.pool.head_dim), "bf16", 97, dev)
    pool = pkv.Pool(k, v)
    bt, lens, offs, _ = dev_batch(w.batch, dev)
    out = torch.full_like(q, float("nan"))
    ws = torch.empty(pkv.decode_shared_prefix_workspace_size(pool, B, w.num_q_heads, 64),
                     dtype=torch.uint8, device=dev)
    pkv.decode_attention_shared_prefix(pool, w.layer, q, w.scale, bt, lens, offs, 64, out, ws)
    torch.cuda.synchronize()
    got = widen_out(out)
    assert np.isfinite(got).all()
    ref = widen_out(gpu_decode(pool, w.layer, q, w.scale, w.batch, dev))
    assert max_abs(got, ref) <= TOL
    kh, vh = host_layer(k, w.layer), host_layer(v, w.layer)
    pairs = [(b, (5 * b) % w.num_q_heads) for b in range(0, B, 3)]
    want = oracle.decode_attention_pairs(kh, vh, 0, to_numpy_bits(q), w.batch.block_tables,
                                         w.batch.seq_lens, w.batch.offsets, w.scale, pairs)
    err = max(max_abs(got[b, h], r) for (b, h), r in want.items())
    assert err <= TOL, err
    assert pkv.device_error(clear=True) == "PKV_OK"
    del pool, k, v
    torch.cuda.empty_cache()
