"""Bad inputs on the GPU, turned into statuses without any fault.

Every bad index used here is one the kernels check before any dereference
(block ids, slots, offsets, capacity, packed layout); host-visible mistakes
are refused before anything is enqueued.  Validate mode reports them as a
status; the fast path skips the bad accesses and records the sticky device
error word, read back with ``device_error()``."""

import numpy as np
import pytest
import torch

import paged_kv_cache_blk_gb300 as pkv
from paged_kv_cache_blk_gb300 import PkvError
from workloads import rand_rows, small_workload

from gpu_util import dev_batch, gpu_decode, gpu_gather, gpu_slots, make_pools, need_gpu

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def dev():
    d = need_gpu()
    pkv.set_validate(False)
    pkv.device_error(clear=True)
    yield d
    pkv.set_validate(False)


@pytest.fixture
def case(dev):
    w = small_workload(seed=5, num_blocks=64, num_layers=2, block_size=16, num_kv_heads=8,
                       head_dim=128, dtype="bf16", lens=[40, 70, 5], layer=1, num_q_heads=32,
                       offsets=True)
    k, v = make_pools(w, dev)
    return w, pkv.Pool(k, v)


def _expect(status, fn, *a):
    with pytest.raises(PkvError) as e:
        fn(*a)
    assert e.value.name == status, e.value


def _tables(w, dev, **edit):
    bt, lens, offs, cu = (x.clone() for x in dev_batch(w.batch, dev))
    if "blk" in edit:
        bt[1, 2] = edit["blk"]
    if "off" in edit:
        offs[0] = edit["off"]
    if "len" in edit:
        lens[2] = edit["len"]
    if "cu" in edit:
        cu[1] += edit["cu"]
    return bt, lens, offs, cu


def _decode(pool, w, dev, bt, lens, offs):
    q = rand_rows((3, 32, 128), "bf16", 1, dev)
    out = torch.full_like(q, 7.0)
    ws = torch.empty(pkv.decode_workspace_size(3, 32, 128, dev), dtype=torch.uint8, device=dev)
    pkv.decode_attention(pool, w.layer, q, w.scale, bt, lens, offs, out, ws)
    return out


def _gather(pool, w, dev, bt, lens, offs, cu):
    n = w.batch.total_tokens
    ko = torch.full((n, 8, 128), 3.0, dtype=torch.bfloat16, device=dev)
    vo = torch.full_like(ko, 3.0)
    pkv.gather(pool, w.layer, bt, lens, offs, cu, ko, vo)
    return ko, vo


@pytest.mark.parametrize("edit,status", [
    (dict(blk=64), "PKV_ERR_INDEX"),
    (dict(blk=-5), "PKV_ERR_INDEX"),
    (dict(off=16), "PKV_ERR_CAPACITY"),
    (dict(off=-1), "PKV_ERR_CAPACITY"),
    (dict(len=10_000), "PKV_ERR_CAPACITY"),
    (dict(len=-3), "PKV_ERR_CAPACITY"),
])
def test_validate_mode_tables(case, dev, edit, status):
    w, pool = case
    bt, lens, offs, cu = _tables(w, dev, **edit)
    pkv.set_validate(True)
    try:
        _expect(status, _decode, pool, w, dev, bt, lens, offs)
        if "len" not in edit:   # the packed layout follows the real lengths
            _expect(status, _gather, pool, w, dev, bt, lens, offs, cu)
    finally:
        pkv.set_validate(False)
    assert pkv.device_error() == "PKV_OK"


def test_validate_mode_packed_layout(case, dev):
    w, pool = case
    bt, lens, offs, cu = _tables(w, dev, cu=1)
    pkv.set_validate(True)
    try:
        _expect("PKV_ERR_INDEX", _gather, pool, w, dev, bt, lens, offs, cu)
    finally:
        pkv.set_validate(False)


def test_validate_mode_slots(case, dev):
    w, pool = case
    k_new = rand_rows((3, 8, 128), "bf16", 2, dev)
    pkv.set_validate(True)
    try:
        for bad in (-2, 64 * 16, 1 << 40):
            sm = torch.tensor([3, bad, -1], dtype=torch.int64, device=dev)
            before = pool.k_cache.clone()
            _expect("PKV_ERR_INDEX", pkv.write_slots, pool, w.layer, k_new, k_new, sm)
            assert torch.equal(before, pool.k_cache)      # nothing written at all
        seq = torch.tensor([0, 3, -1], dtype=torch.int32, device=dev)
        pos = torch.tensor([0, 0, 0], dtype=torch.int32, device=dev)
        bt, _, offs, _ = dev_batch(w.batch, dev)
        out = torch.empty(3, dtype=torch.int64, device=dev)
        _expect("PKV_ERR_INDEX", pkv.build_slot_mapping, pool, bt, offs, seq, pos, out)
        seq = torch.tensor([0, 1, 2], dtype=torch.int32, device=dev)
        pos = torch.tensor([0, 10_000, 0], dtype=torch.int32, device=dev)
        _expect("PKV_ERR_CAPACITY", pkv.build_slot_mapping, pool, bt, offs, seq, pos, out)
    finally:
        pkv.set_validate(False)


def test_fast_path_skips_bad_block(case, dev):
    w, pool = case
    good = gpu_gather(pool, w.layer, w.batch, dev)
    bt, lens, offs, cu = _tables(w, dev, blk=1 << 30)
    ko, vo = _gather(pool, w, dev, bt, lens, offs, cu)
    assert pkv.device_error() == "PKV_ERR_INDEX"
    assert pkv.device_error() == "PKV_OK"                     # cleared
    # rows of the bad block are left as they were; every other row is right
    c1 = int(w.batch.cu_seqlens[1])
    first = 2 * 16 - int(w.batch.offsets[1])                  # first row of logical block 2
    bad = slice(c1 + first, c1 + first + 16)
    mask = torch.ones(ko.shape[0], dtype=torch.bool, device=dev)
    mask[bad] = False
    assert torch.equal(ko[mask], good[0][mask]) and torch.equal(vo[mask], good[1][mask])
    assert torch.all(ko[bad] == 3.0)
    out = _decode(pool, w, dev, bt, lens, offs)
    assert pkv.device_error() == "PKV_ERR_INDEX"
    assert torch.isfinite(out.float()).all()


def test_fast_path_capacity_is_empty(case, dev):
    w, pool = case
    bt, lens, offs, cu = _tables(w, dev, len=10_000)
    out = _decode(pool, w, dev, bt, lens, offs)
    assert pkv.device_error() == "PKV_ERR_CAPACITY"
    assert torch.count_nonzero(out[2]) == 0                   # treated as empty


def test_fast_path_bad_slots(case, dev):
    w, pool = case
    k_new = rand_rows((4, 8, 128), "bf16", 3, dev)
    sm = torch.tensor([5, -2, 64 * 16 + 3, -1], dtype=torch.int64, device=dev)
    before = pool.k_cache.clone()
    pkv.write_slots(pool, w.layer, k_new, k_new, sm)
    assert pkv.device_error() == "PKV_ERR_INDEX"
    changed = (pool.k_cache != before).reshape(64, 2, 16, -1).any(-1)
    assert changed.sum() <= 1 and not changed[:, 0].any()
    assert torch.equal(pool.k_cache[0, w.layer, 5], k_new[0])


def test_host_refusals(case, dev):
    w, pool = case
    bt, lens, offs, cu = dev_batch(w.batch, dev)
    q = rand_rows((3, 32, 128), "bf16", 1, dev)
    out = torch.empty_like(q)
    ws = torch.empty(pkv.decode_workspace_size(3, 32, 128, dev), dtype=torch.uint8, device=dev)
    _expect("PKV_ERR_WORKSPACE", pkv.decode_attention, pool, w.layer, q, w.scale, bt, lens, offs,
            out, ws[:64])
    qm = torch.empty(3 * 32 * 128 + 8, dtype=torch.bfloat16, device=dev)[1:1 + 3 * 32 * 128]
    qm = qm.view(3, 32, 128)
    _expect("PKV_ERR_INVALID_ARG", pkv.decode_attention, pool, w.layer, qm, w.scale, bt, lens,
            offs, out, ws)
    _expect("PKV_ERR_INVALID_ARG", pkv.decode_attention, pool, 5, q, w.scale, bt, lens, offs,
            out, ws)
    q24 = rand_rows((3, 24, 128), "bf16", 1, dev)
    _expect("PKV_ERR_UNSUPPORTED", pkv.decode_attention, pool, w.layer, q24, w.scale, bt, lens,
            offs, torch.empty_like(q24), ws)
    assert pkv.device_error() == "PKV_OK"
