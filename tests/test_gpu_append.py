"""GPU parity for the fused slot mapping + scatter (pkv_append_tokens): the
pool and the returned slots must be bit-identical to the oracle's slot mapping
followed by its scatter (bf16, fp32 and int8 pools), padding tokens are
skipped, and tokens outside their tables are skipped and reported."""

import numpy as np
import pytest
import torch

import oracle
from oracle import quant as Q
import paged_kv_cache_blk_gb300 as pkv
from workloads import PoolSpec, fill_pool, fill_pool_i8, new_pool, rand_rows, small_workload
from workloads import to_numpy_bits

from gpu_util import dev_batch, need_gpu

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def dev():
    d = need_gpu()
    pkv.set_validate(False)
    pkv.device_error(clear=True)
    return d


def _tokens(w, rng, pad_frac=0.15):
    """Every token of the batch in a shuffled order, some marked padding."""
    seq = w.tokens.token_seq.copy()
    pos = w.tokens.token_pos.copy()
    order = rng.permutation(len(seq))
    seq, pos = seq[order], pos[order]
    seq[rng.random(len(seq)) < pad_frac] = -1
    return seq.astype(np.int32), pos.astype(np.int32)


@pytest.mark.parametrize("dtype", ["bf16", "f32", "i8"])
def test_append_matches_slot_mapping_then_scatter(dev, dtype):
    H, D = 4, 64
    w = small_workload(seed=31, num_blocks=96, batch=5, max_len=150, num_kv_heads=H,
                       head_dim=D, dtype="bf16" if dtype == "i8" else dtype)
    rng = np.random.default_rng(32)
    seq, pos = _tokens(w, rng)
    T = len(seq)
    if dtype == "i8":
        spec = PoolSpec(w.pool.num_blocks, w.pool.num_layers, w.pool.block_size, H, D, "i8")
        k = torch.zeros(spec.shape, dtype=torch.uint8, device=dev)
        v = torch.zeros_like(k)
        fill_pool_i8(k, v, spec, w.layer, 33)
        pool = pkv.Pool(k, v, H, D)
        in_dtype = "bf16"
    else:
        spec = w.pool
        k, v = new_pool(spec, dev)
        fill_pool(k, v, spec, w.layer, 33)
        pool = pkv.Pool(k, v)
        in_dtype = dtype
    kh, vh = to_numpy_bits(k), to_numpy_bits(v)
    kn = rand_rows((T, H, D), in_dtype, 34, dev)
    vn = rand_rows((T, H, D), in_dtype, 35, dev)
    bt, _, offs, _ = dev_batch(w.batch, dev)
    sm = torch.full((T,), -7, dtype=torch.int64, device=dev)
    pkv.append_tokens(pool, w.layer, bt, offs, torch.from_numpy(seq).to(dev),
                      torch.from_numpy(pos).to(dev), kn, vn, sm)
    torch.cuda.synchronize()
    ref_sm = oracle.build_slot_mapping(w.batch.block_tables, w.batch.offsets, seq, pos,
                                       spec.block_size)
    assert np.array_equal(sm.cpu().numpy(), ref_sm)
    if dtype == "i8":
        Q.write_slots_i8(kh, vh, w.layer, to_numpy_bits(kn), to_numpy_bits(vn), ref_sm, H, D)
    else:
        oracle.write_slots(kh, vh, w.layer, to_numpy_bits(kn), to_numpy_bits(vn), ref_sm)
    assert np.array_equal(to_numpy_bits(k), kh) and np.array_equal(to_numpy_bits(v), vh)
    assert pkv.device_error() == "PKV_OK"


def test_append_without_slot_output_and_bad_tokens(dev):
    w = small_workload(seed=41, num_blocks=48, batch=3, max_len=60)
    k, v = new_pool(w.pool, dev)
    fill_pool(k, v, w.pool, w.layer, 42)
    pool = pkv.Pool(k, v)
    kh, vh = to_numpy_bits(k), to_numpy_bits(v)
    seq = np.array([0, 1, 2, 5, 1, -1], np.int32)        # 5: no such sequence
    cap = int(w.batch.block_tables.shape[1]) * w.pool.block_size
    pos = np.array([0, 3, 1, 0, cap, 2], np.int32)        # cap: past the table row
    T = len(seq)
    H, D = w.pool.num_kv_heads, w.pool.head_dim
    kn = rand_rows((T, H, D), "bf16", 43, dev)
    vn = rand_rows((T, H, D), "bf16", 44, dev)
    bt, _, offs, _ = dev_batch(w.batch, dev)
    pkv.append_tokens(pool, w.layer, bt, offs, torch.from_numpy(seq).to(dev),
                      torch.from_numpy(pos).to(dev), kn, vn)
    err = pkv.device_error()
    assert err in ("PKV_ERR_INDEX", "PKV_ERR_CAPACITY")
    good = np.array([True, True, True, False, False, False])
    ref_sm = oracle.build_slot_mapping(w.batch.block_tables, w.batch.offsets,
                                       np.where(good, seq, -1).astype(np.int32), pos,
                                       w.pool.block_size)
    oracle.write_slots(kh, vh, w.layer, to_numpy_bits(kn), to_numpy_bits(vn), ref_sm)
    assert np.array_equal(to_numpy_bits(k), kh) and np.array_equal(to_numpy_bits(v), vh)
    pkv.set_validate(True)
    try:
        with pytest.raises(pkv.PkvError):
            pkv.append_tokens(pool, w.layer, bt, offs, torch.from_numpy(seq).to(dev),
                              torch.from_numpy(pos).to(dev), kn, vn)
    finally:
        pkv.set_validate(False)
