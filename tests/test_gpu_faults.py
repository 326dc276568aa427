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


# ---------------------------------------------------------------------------
# bounded waits that give up: a wait on a stage that nothing fills
# ---------------------------------------------------------------------------

def _run_with_stalled_stage(fn, limit_ns=1_000_000, validate=True, mode=1):
    """Run ``fn`` with every wait bounded by ``limit_ns`` and the test hook on
    (the first CTA of the launch leaves its first stage unfilled, so the waits
    on it can only give up).  Returns the status name and the seconds the call
    took, the device synchronised."""
    import time
    pkv.set_wait_limit_ns(limit_ns)
    pkv.set_debug_skip_fill(mode)
    pkv.set_validate(validate)
    t0 = time.perf_counter()
    name = "PKV_OK"
    try:
        fn()
        torch.cuda.synchronize()
    except PkvError as e:
        name = e.name
    finally:
        pkv.set_debug_skip_fill(0)
        pkv.set_wait_limit_ns(0)
        pkv.set_validate(False)
    torch.cuda.synchronize()
    return name, time.perf_counter() - t0


def _decode_case(dev, seed, batch=3, max_len=300):
    nblk = max(256, batch * (max_len // 16 + 2) + 16)
    w = small_workload(seed=seed, num_blocks=nblk, num_layers=2, block_size=16, num_kv_heads=8,
                       head_dim=128, dtype="bf16", batch=batch, min_len=1, max_len=max_len,
                       layer=1, num_q_heads=32, offsets=True)
    k, v = make_pools(w, dev)
    return w, pkv.Pool(k, v)


def test_wait_limit_setting(dev):
    assert pkv.get_wait_limit_ns() == 4_000_000_000
    pkv.set_wait_limit_ns(2_000_000)
    assert pkv.get_wait_limit_ns() == 2_000_000
    pkv.set_wait_limit_ns(0)
    assert pkv.get_wait_limit_ns() == 4_000_000_000
    for bad in (1, 999, 61_000_000_000):
        _expect("PKV_ERR_INVALID_ARG", pkv.set_wait_limit_ns, bad)


def test_decode_wait_gives_up_and_reports_timeout(dev):
    import oracle
    from workloads import to_numpy_bits
    from gpu_util import host_layer, max_abs, widen_out
    w, pool = _decode_case(dev, 201)
    q = rand_rows((w.batch.batch, 32, 128), "bf16", 202, dev)
    pkv.device_error(clear=True)
    name, secs = _run_with_stalled_stage(lambda: gpu_decode(pool, w.layer, q, w.scale, w.batch,
                                                            dev))
    assert name == "PKV_ERR_TIMEOUT"
    assert secs < 1.0, secs                 # one 1 ms bound, not minutes
    # validate mode reported and cleared the word; the context is healthy and
    # the next call is correct
    assert pkv.device_error(clear=True) == "PKV_OK"
    out = gpu_decode(pool, w.layer, q, w.scale, w.batch, dev)
    ref = oracle.decode_attention(host_layer(pool.k_cache, w.layer), host_layer(pool.v_cache, w.layer), 0,
                                  to_numpy_bits(q), w.batch.block_tables, w.batch.seq_lens,
                                  w.batch.offsets, w.scale)
    assert max_abs(widen_out(out), ref) <= 2e-2
    assert pkv.device_error(clear=True) == "PKV_OK"


def test_decode_give_up_without_validate_sets_the_word(dev):
    w, pool = _decode_case(dev, 203, batch=40, max_len=3000)
    q = rand_rows((w.batch.batch, 32, 128), "bf16", 204, dev)
    pkv.device_error(clear=True)
    name, secs = _run_with_stalled_stage(
        lambda: gpu_decode(pool, w.layer, q, w.scale, w.batch, dev), validate=False)
    assert name == "PKV_OK"                 # asynchronous: the status is in the word
    assert secs < 1.0, secs
    assert pkv.device_error(clear=True) == "PKV_ERR_TIMEOUT"
    assert pkv.device_error(clear=True) == "PKV_OK"


def test_decode_give_up_many_waves_ends_quickly(dev):
    """Every CTA of a grid of about 27 waves stalls: the first wave's waits
    give up at the 20 ms bound, and every CTA that starts later sees its
    launch's abort word and leaves at once.  Per-CTA bounds alone would take
    27 x 20 ms."""
    w, pool = _decode_case(dev, 205, batch=64, max_len=4000)
    q = rand_rows((w.batch.batch, 32, 128), "bf16", 206, dev)
    pkv.device_error(clear=True)
    pkv.set_decode_ctas(4096)
    try:
        name, secs = _run_with_stalled_stage(
            lambda: gpu_decode(pool, w.layer, q, w.scale, w.batch, dev), limit_ns=20_000_000,
            mode=2)
    finally:
        pkv.set_decode_ctas(0)
    assert name == "PKV_ERR_TIMEOUT"
    assert secs < 0.3, secs
    assert pkv.device_error(clear=True) == "PKV_OK"


def test_decode_step_give_up_then_correct(dev):
    """The fused decode step gives up the same way; a later launch, numbered
    differently, is not cut short by the earlier give-up even before the word
    is cleared."""
    import oracle
    from workloads import to_numpy_bits
    from gpu_util import host_layer, max_abs, widen_out
    w, pool = _decode_case(dev, 207, batch=8, max_len=900)
    B = w.batch.batch
    q = rand_rows((B, 32, 128), "bf16", 208, dev)
    kn = rand_rows((B, 8, 128), "bf16", 209, dev)
    vn = rand_rows((B, 8, 128), "bf16", 210, dev)
    bt, lens, offs, _ = dev_batch(w.batch, dev)
    ws = torch.empty(pkv.decode_workspace_size(B, 32, 128, dev), dtype=torch.uint8, device=dev)
    out = torch.empty_like(q)
    pkv.device_error(clear=True)
    name, _ = _run_with_stalled_stage(
        lambda: pkv.decode_step(pool, w.layer, q, w.scale, bt, lens, offs, kn, vn, out, ws),
        validate=False)
    assert name == "PKV_OK"
    # not cleared yet: the next launches, over a pool only the generator wrote,
    # still run to completion
    w2, pool2 = _decode_case(dev, 215, batch=8, max_len=900)
    q2 = rand_rows((B, 32, 128), "bf16", 216, dev)
    out2 = gpu_decode(pool2, w2.layer, q2, w2.scale, w2.batch, dev)
    torch.cuda.synchronize()
    ref = oracle.decode_attention(host_layer(pool2.k_cache, w2.layer),
                                  host_layer(pool2.v_cache, w2.layer), 0, to_numpy_bits(q2),
                                  w2.batch.block_tables, w2.batch.seq_lens, w2.batch.offsets,
                                  w2.scale)
    assert max_abs(widen_out(out2), ref) <= 2e-2
    assert pkv.device_error(clear=True) == "PKV_ERR_TIMEOUT"
    assert pkv.device_error(clear=True) == "PKV_OK"


def test_prefill_wait_gives_up_and_reports_timeout(dev):
    import oracle
    from workloads import PoolSpec, to_numpy_bits
    from workloads.gen import FreeList, _pack
    from gpu_util import max_abs, widen_out
    rng = np.random.default_rng(211)
    lens = [600, 260, 129]
    spec = PoolSpec(128, 2, 16, 2, 128, "bf16")
    free = FreeList(rng.permutation(spec.num_blocks))
    tables = [free.pop(-(-L // 16)) for L in lens]
    batch = _pack(tables, np.asarray(lens), np.zeros(3, np.int64))
    cu = np.concatenate([[0], np.cumsum(lens)]).astype(np.int64)
    k = rand_rows(spec.shape, "bf16", 212, dev)
    v = rand_rows(spec.shape, "bf16", 213, dev)
    q = rand_rows((int(cu[-1]), 8, 128), "bf16", 214, dev)
    pool = pkv.Pool(k, v)
    t = lambda a, dt: torch.from_numpy(np.ascontiguousarray(a)).to(dev, dt)
    args = (t(batch.block_tables, torch.int32), t(batch.seq_lens, torch.int32),
            t(batch.offsets, torch.int32), t(cu, torch.int64), max(lens))
    out = torch.zeros_like(q)
    scale = 128 ** -0.5
    pkv.device_error(clear=True)
    name, secs = _run_with_stalled_stage(
        lambda: pkv.prefill_attention(pool, 1, q, scale, *args, out))
    assert name == "PKV_ERR_TIMEOUT"
    assert secs < 1.0, secs
    assert pkv.device_error(clear=True) == "PKV_OK"
    pkv.prefill_attention(pool, 1, q, scale, *args, out)
    torch.cuda.synchronize()
    ref = oracle.prefill_attention(to_numpy_bits(k), to_numpy_bits(v), 1, to_numpy_bits(q),
                                   batch.block_tables, batch.seq_lens, batch.offsets, cu, scale)
    assert max_abs(widen_out(out), ref) <= 2e-2
    assert pkv.device_error(clear=True) == "PKV_OK"
