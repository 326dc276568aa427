"""GPU parity for whole-block moves (copy-on-write copy, swap out / in to
page-locked host memory) and an allocator-driven serving scenario: the
library's C++ allocator and the oracle allocator build the same tables, the
device path (copy-on-write copies, scatter, decode) is compared with the
oracle path.  Bad inputs here are all ones the host or kernel checks catch."""

import numpy as np
import pytest
import torch

import oracle
from oracle import allocator as OA
import paged_kv_cache_blk_gb300 as pkv
from paged_kv_cache_blk_gb300 import PkvError
from workloads import PoolSpec, rand_rows, to_numpy_bits

from gpu_util import gpu_decode, max_abs, need_gpu, widen_out

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def dev():
    d = need_gpu()
    pkv.set_validate(False)
    pkv.set_decode_ctas(0)
    pkv.device_error(clear=True)
    return d


def _pool(dev, spec, seed):
    k = rand_rows(spec.shape, spec.dtype, seed, dev)
    v = rand_rows(spec.shape, spec.dtype, seed + 1, dev)
    return k, v


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_copy_blocks_matches_oracle(dev, dtype):
    spec = PoolSpec(64, 3, 16, 4, 64, dtype)
    k, v = _pool(dev, spec, 3)
    pool = pkv.Pool(k, v)
    kh, vh = to_numpy_bits(k), to_numpy_bits(v)
    rng = np.random.default_rng(4)
    for layer in (-1, 0, 2):
        ids = rng.permutation(64)
        src, dst = ids[:10], ids[10:20]
        pkv.copy_blocks(pool, layer, torch.from_numpy(src.astype(np.int32)).to(dev),
                        torch.from_numpy(dst.astype(np.int32)).to(dev))
        oracle.copy_blocks(kh, vh, layer, src, dst)
        assert np.array_equal(to_numpy_bits(k), kh) and np.array_equal(to_numpy_bits(v), vh)


def test_swap_round_trip(dev):
    spec = PoolSpec(128, 4, 16, 8, 128, "bf16")
    k, v = _pool(dev, spec, 5)
    pool = pkv.Pool(k, v)
    kh, vh = to_numpy_bits(k), to_numpy_bits(v)
    rng = np.random.default_rng(6)
    out_ids = rng.permutation(128)[:20]
    for layer in (-1, 2):
        L = 4 if layer < 0 else 1
        hk = torch.empty((20, L, 16, 8, 128), dtype=torch.bfloat16, pin_memory=True)
        hv = torch.empty_like(hk, pin_memory=True)
        pkv.swap_out(pool, layer, torch.from_numpy(out_ids.astype(np.int32)).to(dev), hk, hv)
        torch.cuda.synchronize()
        rk, rv = oracle.swap_out(kh, vh, layer, out_ids)
        assert np.array_equal(to_numpy_bits(hk), rk) and np.array_equal(to_numpy_bits(hv), rv)
        in_ids = rng.permutation(128)[:20]
        pkv.swap_in(pool, layer, torch.from_numpy(in_ids.astype(np.int32)).to(dev), hk, hv)
        torch.cuda.synchronize()
        oracle.swap_in(kh, vh, layer, in_ids, rk, rv)
        assert np.array_equal(to_numpy_bits(k), kh) and np.array_equal(to_numpy_bits(v), vh)


def test_swap_refuses_pageable_and_short_buffers(dev):
    spec = PoolSpec(16, 2, 16, 2, 64, "bf16")
    k, v = _pool(dev, spec, 7)
    pool = pkv.Pool(k, v)
    ids = torch.arange(4, dtype=torch.int32, device=dev)
    pageable = torch.empty((4, 2, 16, 2, 64), dtype=torch.bfloat16)
    with pytest.raises(PkvError) as e:
        pkv.swap_out(pool, -1, ids, pageable, pageable)
    assert e.value.name == "PKV_ERR_INVALID_ARG"
    short = torch.empty((3, 2, 16, 2, 64), dtype=torch.bfloat16, pin_memory=True)
    with pytest.raises(PkvError) as e:
        pkv.swap_in(pool, -1, ids, short, short)
    assert e.value.name == "PKV_ERR_INVALID_ARG"


def test_copy_blocks_bad_ids(dev):
    spec = PoolSpec(16, 1, 16, 2, 64, "bf16")
    k, v = _pool(dev, spec, 8)
    pool = pkv.Pool(k, v)
    before = k.clone()
    src = torch.tensor([1, 99], dtype=torch.int32, device=dev)
    dst = torch.tensor([2, 3], dtype=torch.int32, device=dev)
    pkv.copy_blocks(pool, -1, src, dst)                   # fast path: bad pair skipped
    assert pkv.device_error() == "PKV_ERR_INDEX"
    assert torch.equal(k[2], before[1]) and torch.equal(k[3], before[3])
    pkv.set_validate(True)
    try:
        with pytest.raises(PkvError) as e:
            pkv.copy_blocks(pool, -1, dst, torch.tensor([4, -7], dtype=torch.int32, device=dev))
        assert e.value.name == "PKV_ERR_INDEX"
    finally:
        pkv.set_validate(False)


def test_allocator_driven_serving_scenario(dev):
    """Requests arrive, hit a shared prefix, fork, append with copy-on-write
    and get evicted; after every decode step the device output matches the
    oracle run on the oracle allocator's tables."""
    bs, N, Hkv, D, G = 16, 96, 8, 128, 4
    spec = PoolSpec(N, 2, bs, Hkv, D, "bf16")
    layer = 1
    k, v = _pool(dev, spec, 9)
    pool = pkv.Pool(k, v)
    kh, vh = to_numpy_bits(k), to_numpy_bits(v)
    rng = np.random.default_rng(10)
    order = rng.permutation(N)
    ca = pkv.Allocator(N, bs, order)
    oa = OA.KVCacheManager(N, bs, order)
    row = (Hkv, D)

    def both(name, *args):
        ro = getattr(oa, name)(*args)
        rc = getattr(ca, name)(*args)
        return ro, rc

    def write(sid, n, seed):
        (so, cow_o), (sc, cow_c) = both("seq_append", sid, n)
        assert list(so) == sc.tolist() and cow_o == cow_c
        if cow_c:
            src = torch.tensor([c[0] for c in cow_c], dtype=torch.int32, device=dev)
            dst = torch.tensor([c[1] for c in cow_c], dtype=torch.int32, device=dev)
            pkv.copy_blocks(pool, -1, src, dst)
            oracle.copy_blocks(kh, vh, -1, [c[0] for c in cow_o], [c[1] for c in cow_o])
        kn = rand_rows((n,) + row, "bf16", seed, dev)
        vn = rand_rows((n,) + row, "bf16", seed + 1, dev)
        pkv.write_slots(pool, layer, kn, vn, torch.from_numpy(sc).to(dev))
        oracle.write_slots(kh, vh, layer, to_numpy_bits(kn), to_numpy_bits(vn), np.array(so))

    # a long prompt, a prefix hit on it with an offset into the last shared block,
    # a fork (beam) of that, and a few independent requests
    both("seq_new", 0, 0)
    write(0, 150, 100)
    both("seq_new", 1, 0)
    t0 = oa.seq_table(0)
    both("seq_share", 1, t0.block_ids[:5], 70)      # 70 tokens span 5 blocks
    write(1, 30, 110)                               # copy-on-write in block 4
    both("seq_fork", 1, 2)
    write(2, 1, 120)                                # copy-on-write again
    for sid, n in ((3, 41), (4, 16), (5, 1)):
        both("seq_new", sid, int(rng.integers(0, bs)))
        write(sid, n, 130 + sid)
    live = [0, 1, 2, 3, 4, 5]
    for step in range(3):
        for sid in live:
            write(sid, 1, 200 + 10 * step + sid)
        mb = max(oa.seq_table(s).capacity(bs) // bs + 1 for s in live)
        tables, lens, offs = ca.seq_tables(live, mb)
        for i, sid in enumerate(live):
            t = oa.seq_table(sid)
            assert tables[i][:len(t.block_ids)].tolist() == t.block_ids
        q = rand_rows((len(live), Hkv * G, D), "bf16", 300 + step, dev)
        from workloads.gen import Batch
        batch = Batch(tables, lens, offs, np.concatenate([[0], np.cumsum(lens)]).astype(np.int64))
        out = gpu_decode(pool, layer, q, D ** -0.5, batch, dev)
        ref = oracle.decode_attention(kh, vh, layer, to_numpy_bits(q), tables, lens, offs,
                                      D ** -0.5)
        assert max_abs(widen_out(out), ref) <= 2e-2, step
        both("seq_free", live.pop(0))               # the oldest request leaves
        assert ca.num_free() == oa.num_free()
    assert np.array_equal(to_numpy_bits(k), kh)
