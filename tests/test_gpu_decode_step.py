"""GPU parity for the fused decode step (pkv_decode_step): after the call the
pool must be bit-identical to the oracle's slot mapping and scatter of each
sequence's new row at its last position, and the output must match the
oracle's decode attention over that pool.  The fused call must also agree
bit for bit with pkv_append_tokens followed by pkv_decode_attention, and a
second step must read the row the first one stored."""

import numpy as np
import pytest
import torch

import oracle
import paged_kv_cache_blk_gb300 as pkv
from workloads import fill_pool, new_pool, rand_rows, small_workload, to_numpy_bits

from gpu_util import dev_batch, max_abs, need_gpu, widen_out

pytestmark = pytest.mark.gpu

TOL = {"bf16": 2e-2, "f32": 1e-5}


@pytest.fixture(scope="module")
def dev():
    d = need_gpu()
    pkv.set_validate(False)
    pkv.set_decode_ctas(0)
    pkv.device_error(clear=True)
    return d


def _case(seed, dtype, H, D, bs, lens, offsets=True, spare=0):
    """A workload whose tables hold `spare` positions past each length."""
    w = small_workload(seed=seed, num_blocks=4 * (sum(lens) + spare * len(lens)) // bs + 64,
                       block_size=bs, num_kv_heads=H, head_dim=D, dtype=dtype,
                       lens=[L + spare if L > 0 else 0 for L in lens], offsets=offsets)
    w.batch.seq_lens[:] = np.asarray(lens, dtype=w.batch.seq_lens.dtype)
    return w


def _inputs(w, dev, G, dtype, seed):
    spec = w.pool
    k, v = new_pool(spec, dev)
    fill_pool(k, v, spec, w.layer, seed)
    B, H, D = w.batch.batch, spec.num_kv_heads, spec.head_dim
    kn = rand_rows((B, H, D), dtype, seed + 1, dev)
    vn = rand_rows((B, H, D), dtype, seed + 2, dev)
    q = rand_rows((B, H * G, D), dtype, seed + 3, dev)
    return k, v, kn, vn, q


def _oracle_step(kh, vh, w, kn, vn, q, scale, lens):
    """The oracle's decode step: slot of position len-1 for every non-empty
    sequence, scatter of its new row, decode attention over the result."""
    seqs = np.array([b for b in range(len(lens)) if lens[b] > 0], dtype=np.int32)
    pos = np.array([lens[b] - 1 for b in seqs], dtype=np.int32)
    sm = oracle.build_slot_mapping(w.batch.block_tables, w.batch.offsets, seqs, pos,
                                   w.pool.block_size)
    oracle.write_slots(kh, vh, w.layer, to_numpy_bits(kn)[seqs], to_numpy_bits(vn)[seqs], sm)
    return oracle.decode_attention(kh, vh, w.layer, to_numpy_bits(q), w.batch.block_tables,
                                   np.asarray(lens), w.batch.offsets, scale)


def _step(pool, w, q, kn, vn, lens_t, dev):
    bt, _, offs, _ = dev_batch(w.batch, dev)
    B, Hq, D = q.shape
    out = torch.full_like(q, float("nan"))
    ws = torch.empty(pkv.decode_workspace_size(B, Hq, D, dev), dtype=torch.uint8, device=dev)
    pkv.decode_step(pool, w.layer, q, w.scale, bt, lens_t, offs, kn, vn, out, ws)
    return out


CASES = [
    # dtype, H, G, D, bs, lens, ctas
    ("bf16", 2, 4, 128, 16, [300, 37, 129, 1, 16, 17], 0),
    ("bf16", 8, 4, 128, 16, [1000, 2, 15, 513], 0),
    ("bf16", 4, 1, 64, 32, [200, 64, 65], 0),
    ("bf16", 2, 8, 128, 8, [90, 0, 33, 0, 7], 0),
    ("f32", 4, 2, 64, 8, [120, 9, 1, 64], 0),
    ("f32", 2, 4, 128, 16, [250, 31], 0),
    ("bf16", 2, 4, 128, 16, [700, 333, 64, 5], 1),
    ("bf16", 2, 4, 128, 16, [700, 333, 64, 5], 3),
    ("bf16", 2, 4, 128, 16, [700, 333, 64, 5], 64),
    ("bf16", 2, 4, 128, 16, [700, 333, 64, 5], 997),
]


@pytest.mark.parametrize("dtype,H,G,D,bs,lens,ctas", CASES,
                         ids=[f"{c[0]}-H{c[1]}G{c[2]}D{c[3]}-bs{c[4]}-ctas{c[6]}-{i}"
                              for i, c in enumerate(CASES)])
def test_decode_step_matches_oracle(dev, dtype, H, G, D, bs, lens, ctas):
    seed = 7 + len(lens) + bs + ctas
    w = _case(seed, dtype, H, D, bs, lens)
    k, v, kn, vn, q = _inputs(w, dev, G, dtype, seed)
    kh, vh = to_numpy_bits(k), to_numpy_bits(v)
    pool = pkv.Pool(k, v)
    lens_t = torch.tensor(lens, dtype=torch.int32, device=dev)
    pkv.set_decode_ctas(ctas)
    try:
        out = _step(pool, w, q, kn, vn, lens_t, dev)
        torch.cuda.synchronize()
    finally:
        pkv.set_decode_ctas(0)
    ref = _oracle_step(kh, vh, w, kn, vn, q, w.scale, lens)
    assert np.array_equal(to_numpy_bits(k), kh) and np.array_equal(to_numpy_bits(v), vh)
    assert max_abs(widen_out(out), ref) <= TOL[dtype]
    assert pkv.device_error() == "PKV_OK"


def test_decode_step_equals_append_then_decode(dev):
    """Bit for bit: the fused step against pkv_append_tokens (token b at
    position len-1) followed by pkv_decode_attention on a copy of the pool."""
    lens = [2048, 517, 1, 64, 1000, 33, 4095, 16]
    w = _case(71, "bf16", 8, 128, 16, lens)
    k, v, kn, vn, q = _inputs(w, dev, 4, "bf16", 71)
    k2, v2 = k.clone(), v.clone()
    lens_t = torch.tensor(lens, dtype=torch.int32, device=dev)
    out = _step(pkv.Pool(k, v), w, q, kn, vn, lens_t, dev)
    bt, _, offs, _ = dev_batch(w.batch, dev)
    pool2 = pkv.Pool(k2, v2)
    B = len(lens)
    seq = torch.arange(B, dtype=torch.int32, device=dev)
    pkv.append_tokens(pool2, w.layer, bt, offs, seq, lens_t - 1, kn, vn, None)
    out2 = torch.empty_like(q)
    ws = torch.empty(pkv.decode_workspace_size(B, q.shape[1], 128, dev), dtype=torch.uint8,
                     device=dev)
    pkv.decode_attention(pool2, w.layer, q, w.scale, bt, lens_t, offs, out2, ws)
    torch.cuda.synchronize()
    assert torch.equal(k, k2) and torch.equal(v, v2)
    assert torch.equal(out.view(torch.int16), out2.view(torch.int16))


def test_two_steps_and_graph_replay(dev):
    """Two consecutive steps, captured once in a CUDA graph and replayed with
    new inputs: the second step attends to the row the first one stored."""
    lens = [300, 47, 129, 16]
    w = _case(81, "bf16", 2, 128, 16, lens, spare=2)
    k, v, kn, vn, q = _inputs(w, dev, 4, "bf16", 81)
    kh, vh = to_numpy_bits(k), to_numpy_bits(v)
    pool = pkv.Pool(k, v)
    bt, _, offs, _ = dev_batch(w.batch, dev)
    B, Hq, D = q.shape
    lens_t = torch.tensor(lens, dtype=torch.int32, device=dev)
    out = torch.empty_like(q)
    ws = torch.empty(pkv.decode_workspace_size(B, Hq, D, dev), dtype=torch.uint8, device=dev)
    # first use of the kernel outside the capture (decode only: the pool stays)
    pkv.decode_attention(pool, w.layer, q, w.scale, bt, lens_t, offs, out, ws)
    torch.cuda.synchronize()
    side = torch.cuda.Stream(dev)
    side.wait_stream(torch.cuda.current_stream(dev))
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.stream(side):
        with torch.cuda.graph(graph, stream=side):
            pkv.decode_step(pool, w.layer, q, w.scale, bt, lens_t, offs, kn, vn, out, ws)
    torch.cuda.current_stream(dev).wait_stream(side)
    # capture ran nothing: the pool is still the original one
    assert np.array_equal(to_numpy_bits(k), kh)
    for step in range(2):
        cur = [L + step for L in lens]
        kn.copy_(rand_rows(kn.shape, "bf16", 90 + step, dev))
        vn.copy_(rand_rows(vn.shape, "bf16", 95 + step, dev))
        q.copy_(rand_rows(q.shape, "bf16", 99 + step, dev))
        lens_t.copy_(torch.tensor(cur, dtype=torch.int32))
        graph.replay()
        torch.cuda.synchronize()
        ref = _oracle_step(kh, vh, w, kn, vn, q, w.scale, cur)
        assert np.array_equal(to_numpy_bits(k), kh) and np.array_equal(to_numpy_bits(v), vh)
        assert max_abs(widen_out(out), ref) <= 2e-2
    assert pkv.device_error() == "PKV_OK"


def test_decode_step_bad_block_is_skipped_and_reported(dev):
    """A table entry outside the pool.  In validate mode the call is refused
    before anything runs (the pool is unchanged).  Otherwise that block is
    skipped and reported, the sequence's new row is stored nowhere, and the
    other sequence's row lands in its slot."""
    lens = [100, 60]
    w = _case(91, "bf16", 2, 128, 16, lens)
    k, v, kn, vn, q = _inputs(w, dev, 2, "bf16", 91)
    N = w.pool.num_blocks
    bt_np = w.batch.block_tables.copy()
    last = (int(w.batch.offsets[1]) + lens[1] - 1) // 16
    bt_np[1, last] = N + 5
    kh, vh = to_numpy_bits(k), to_numpy_bits(v)
    pool = pkv.Pool(k, v)
    t = lambda a, dt: torch.from_numpy(np.ascontiguousarray(a)).to(dev, dt)
    args = (t(bt_np, torch.int32), t(np.asarray(lens), torch.int32),
            t(w.batch.offsets, torch.int32))
    out = torch.zeros_like(q)
    ws = torch.empty(pkv.decode_workspace_size(2, q.shape[1], 128, dev), dtype=torch.uint8,
                     device=dev)
    pkv.set_validate(True)
    try:
        with pytest.raises(pkv.PkvError) as e:
            pkv.decode_step(pool, w.layer, q, w.scale, *args, kn, vn, out, ws)
        assert e.value.name == "PKV_ERR_INDEX"
    finally:
        pkv.set_validate(False)
        pkv.device_error(clear=True)
    assert np.array_equal(to_numpy_bits(k), kh) and np.array_equal(to_numpy_bits(v), vh)
    pkv.decode_step(pool, w.layer, q, w.scale, *args, kn, vn, out, ws)
    torch.cuda.synchronize()
    assert pkv.device_error(clear=True) == "PKV_ERR_INDEX"
    seqs = np.array([0], dtype=np.int32)
    sm = oracle.build_slot_mapping(w.batch.block_tables, w.batch.offsets, seqs,
                                   np.array([lens[0] - 1], dtype=np.int32), 16)
    oracle.write_slots(kh, vh, w.layer, to_numpy_bits(kn)[seqs], to_numpy_bits(vn)[seqs], sm)
    assert np.array_equal(to_numpy_bits(k), kh) and np.array_equal(to_numpy_bits(v), vh)


I8_CASES = [
    # H, G, D, bs, lens, ctas
    (8, 4, 128, 16, [300, 37, 129, 1, 16, 17], 0),
    (2, 2, 64, 8, [90, 0, 33, 7], 0),
    (4, 4, 128, 16, [700, 333, 64, 5], 5),
]


@pytest.mark.parametrize("H,G,D,bs,lens,ctas", I8_CASES,
                         ids=[f"i8-H{c[0]}G{c[1]}D{c[2]}-bs{c[3]}-ctas{c[5]}" for c in I8_CASES])
def test_decode_step_int8_matches_oracle(dev, H, G, D, bs, lens, ctas):
    """int8 pools: the new rows are quantised into the pool exactly as the
    oracle's quantising scatter does (bit-exact), and attention over the
    dequantised pool matches within the bf16 tolerance."""
    from oracle import quant as Q
    from workloads import PoolSpec, fill_pool_i8
    seed = 101 + len(lens) + ctas
    w = _case(seed, "bf16", H, D, bs, lens)
    spec = PoolSpec(w.pool.num_blocks, w.pool.num_layers, bs, H, D, "i8")
    k = torch.zeros(spec.shape, dtype=torch.uint8, device=dev)
    v = torch.zeros_like(k)
    fill_pool_i8(k, v, spec, w.layer, seed)
    kh, vh = to_numpy_bits(k), to_numpy_bits(v)
    B = len(lens)
    kn = rand_rows((B, H, D), "bf16", seed + 1, dev)
    vn = rand_rows((B, H, D), "bf16", seed + 2, dev)
    q = rand_rows((B, H * G, D), "bf16", seed + 3, dev)
    pool = pkv.Pool(k, v, H, D)
    lens_t = torch.tensor(lens, dtype=torch.int32, device=dev)
    pkv.set_decode_ctas(ctas)
    try:
        out = _step(pool, w, q, kn, vn, lens_t, dev)
        torch.cuda.synchronize()
    finally:
        pkv.set_decode_ctas(0)
    seqs = np.array([b for b in range(B) if lens[b] > 0], dtype=np.int32)
    pos = np.array([lens[b] - 1 for b in seqs], dtype=np.int32)
    sm = oracle.build_slot_mapping(w.batch.block_tables, w.batch.offsets, seqs, pos, bs)
    Q.write_slots_i8(kh, vh, w.layer, to_numpy_bits(kn)[seqs], to_numpy_bits(vn)[seqs], sm, H, D)
    assert np.array_equal(to_numpy_bits(k), kh) and np.array_equal(to_numpy_bits(v), vh)
    ref = Q.decode_attention_i8(kh, vh, w.layer, to_numpy_bits(q), w.batch.block_tables,
                                np.asarray(lens), w.batch.offsets, w.scale)
    assert max_abs(widen_out(out), ref) <= 2e-2
    assert pkv.device_error() == "PKV_OK"


def test_decode_step_int8_equals_append_then_decode(dev):
    from workloads import PoolSpec, fill_pool_i8
    lens = [2048, 517, 1, 64, 1000, 33, 4095, 16]
    H, D, bs = 8, 128, 16
    w = _case(171, "bf16", H, D, bs, lens)
    spec = PoolSpec(w.pool.num_blocks, w.pool.num_layers, bs, H, D, "i8")
    k = torch.zeros(spec.shape, dtype=torch.uint8, device=dev)
    v = torch.zeros_like(k)
    fill_pool_i8(k, v, spec, w.layer, 171)
    k2, v2 = k.clone(), v.clone()
    B = len(lens)
    kn = rand_rows((B, H, D), "bf16", 172, dev)
    vn = rand_rows((B, H, D), "bf16", 173, dev)
    q = rand_rows((B, 4 * H, D), "bf16", 174, dev)
    lens_t = torch.tensor(lens, dtype=torch.int32, device=dev)
    out = _step(pkv.Pool(k, v, H, D), w, q, kn, vn, lens_t, dev)
    bt, _, offs, _ = dev_batch(w.batch, dev)
    pool2 = pkv.Pool(k2, v2, H, D)
    seq = torch.arange(B, dtype=torch.int32, device=dev)
    pkv.append_tokens(pool2, w.layer, bt, offs, seq, lens_t - 1, kn, vn, None)
    out2 = torch.empty_like(q)
    ws = torch.empty(pkv.decode_workspace_size(B, q.shape[1], D, dev), dtype=torch.uint8,
                     device=dev)
    pkv.decode_attention(pool2, w.layer, q, w.scale, bt, lens_t, offs, out2, ws)
    torch.cuda.synchronize()
    assert torch.equal(k, k2) and torch.equal(v, v2)
    assert torch.equal(out.view(torch.int16), out2.view(torch.int16))
