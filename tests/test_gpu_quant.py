"""GPU parity for int8 KV pools against ``oracle.quant``:

* the quantising scatter is bit-exact (codes, scales, untouched padding and
  untouched rows), including zero heads, ties, subnormal and huge values;
* decode over int8 pools matches the dequantised fp64 oracle within the bf16
  output tolerance, for every supported head layout, block size, split count,
  first-block offsets, empty and one-token sequences, and at the full decode
  workload size on sampled (sequence, head) pairs;
* scatter then decode on the GPU equals the oracle's scatter then decode;
* block copy, swap and gather move int8 byte rows bit-exactly.

All inputs are drawn by ``workloads`` (or written here from closed forms);
nothing the CUDA path computes is fed to the oracle."""

import zlib

import numpy as np
import pytest
import torch

import oracle
from oracle import quant as Q
import paged_kv_cache_blk_gb300 as pkv
from workloads import PoolSpec, fill_pool_i8, make_workload, rand_rows, to_numpy_bits
from workloads.gen import Batch, FreeList, _pack

from gpu_util import BF16_TOL, dev_batch, gpu_decode, host_layer, max_abs, need_gpu, widen_out

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def dev():
    d = need_gpu()
    pkv.set_validate(False)
    pkv.set_decode_ctas(0)
    pkv.device_error(clear=True)
    return d


def _pools(dev, spec, seed):
    k = torch.zeros(spec.shape, dtype=torch.uint8, device=dev)
    v = torch.zeros_like(k)
    for layer in range(spec.num_layers):
        fill_pool_i8(k, v, spec, layer, seed + 101 * layer)
    return k, v, pkv.Pool(k, v, spec.num_kv_heads, spec.head_dim)


def _bits(t):
    return to_numpy_bits(t)


def _new_rows(dev, n, H, D, seed):
    """bf16 rows with magnitudes spread over 10^-3 .. 10^3 per (token, head),
    plus hand-made heads: zeros, exact ties, a lone value, subnormals, huge."""
    x = rand_rows((n, H, D), "f32", seed, dev)
    g = torch.Generator(device=dev)
    g.manual_seed(seed + 7)
    mag = torch.pow(10.0, torch.rand((n, H, 1), generator=g, device=dev) * 6 - 3)
    x = (x * mag)
    if n >= 5:
        x[0, 0] = 0.0                                            # zero head: scale 0
        ties = torch.zeros(D, device=dev)
        ties[0] = 127.0                                          # scale exactly 1
        ties[1:9] = torch.tensor([0.5, 1.5, 2.5, -2.5, 3.5, -0.5, 126.5, -126.5])
        x[1, 0] = ties
        x[2, 0] = 0.0
        x[2, 0, D // 2] = -3.0                                   # lone value
        x[3, 0] = torch.linspace(-1, 1, D, device=dev) * 1e-39   # subnormal bf16
        x[4, 0] = torch.linspace(-1, 1, D, device=dev) * 3e38    # near the top of range
    return x.to(torch.bfloat16)


@pytest.mark.parametrize("H,D", [(8, 128), (2, 64), (4, 32), (1, 256), (3, 128)])
def test_quantising_scatter_bit_exact(dev, H, D):
    spec = PoolSpec(40, 2, 16, H, D, "i8")
    k, v, pool = _pools(dev, spec, 11 + H + D)
    kh, vh = _bits(k), _bits(v)
    rng = np.random.default_rng(H * 1000 + D)
    n = 150
    slots = rng.permutation(spec.num_blocks * spec.block_size)[:n].astype(np.int64)
    slots[rng.random(n) < 0.1] = -1
    kn = _new_rows(dev, n, H, D, 5 + D)
    vn = _new_rows(dev, n, H, D, 9 + D)
    for layer in (1, 0):
        pkv.write_slots(pool, layer, kn, vn, torch.from_numpy(slots).to(dev))
        Q.write_slots_i8(kh, vh, layer, _bits(kn), _bits(vn), slots, H, D)
        assert np.array_equal(_bits(k), kh)
        assert np.array_equal(_bits(v), vh)
    assert pkv.device_error() == "PKV_OK"


def test_quantising_scatter_bad_slots(dev):
    spec = PoolSpec(8, 1, 16, 2, 64, "i8")
    k, v, pool = _pools(dev, spec, 3)
    kh, vh = _bits(k), _bits(v)
    kn = _new_rows(dev, 3, 2, 64, 1)
    slots = np.array([5, 8 * 16, -3], np.int64)            # good, past the pool, bad negative
    pkv.write_slots(pool, 0, kn, kn, torch.from_numpy(slots).to(dev))
    assert pkv.device_error() == "PKV_ERR_INDEX"
    Q.write_slots_i8(kh, vh, 0, _bits(kn)[:1], _bits(kn)[:1], slots[:1], 2, 64)
    assert np.array_equal(_bits(k), kh) and np.array_equal(_bits(v), vh)


def _case(dev, seed, lens, G, H=8, D=128, bs=16, offsets=True):
    rng = np.random.default_rng(seed)
    lens = np.asarray(lens, np.int64)
    B = len(lens)
    offs = rng.integers(0, bs, size=B) if offsets else np.zeros(B, np.int64)
    need = [-(-(int(o) + int(L)) // bs) for o, L in zip(offs, lens)]
    N = max(16, sum(need) + 8)
    spec = PoolSpec(N, 2, bs, H, D, "i8")
    free = FreeList(rng.permutation(N))
    tables = [free.pop(n) for n in need]
    batch = _pack(tables, lens, offs)
    k, v, pool = _pools(dev, spec, seed)
    q = rand_rows((B, H * G, D), "bf16", seed + 3, dev)
    return spec, batch, k, v, pool, q


def _decode_vs_oracle(dev, spec, batch, k, v, pool, q, layer=1, scale=None):
    D = spec.head_dim
    scale = D ** -0.5 if scale is None else scale
    out = gpu_decode(pool, layer, q, scale, batch, dev)
    torch.cuda.synchronize()
    ref = Q.decode_attention_i8(host_layer(k, layer), host_layer(v, layer), 0, _bits(q),
                                batch.block_tables, batch.seq_lens, batch.offsets, scale)
    return out, ref


DECODE_CASES = [
    # G, H, D, bs, lens
    (4, 8, 128, 16, [1, 17, 300, 1000]),
    (1, 8, 128, 16, [64, 129]),
    (8, 4, 128, 16, [250, 3]),
    (2, 2, 64, 32, [500, 77]),
    (4, 1, 128, 8, [333]),
    (4, 8, 64, 64, [129, 700]),
    (8, 8, 128, 1, [40, 9]),
    (4, 8, 128, 128, [1025, 1]),
]


@pytest.mark.parametrize("G,H,D,bs,lens", DECODE_CASES,
                         ids=[f"G{c[0]}-H{c[1]}-D{c[2]}-bs{c[3]}-{c[4]}" for c in DECODE_CASES])
def test_decode_int8_matches_oracle(dev, G, H, D, bs, lens):
    seed = zlib.crc32(repr((G, H, D, bs, lens)).encode()) % 10000
    spec, batch, k, v, pool, q = _case(dev, seed, lens, G, H, D, bs)
    out, ref = _decode_vs_oracle(dev, spec, batch, k, v, pool, q)
    assert torch.isfinite(out.float()).all()
    assert max_abs(widen_out(out), ref) <= BF16_TOL
    assert pkv.device_error() == "PKV_OK"


@pytest.mark.parametrize("ctas", [1, 7, 300, 0])
def test_decode_int8_split_counts(dev, ctas):
    """One CTA (no split), a few, more CTAs than blocks of some sequences, and
    the default grid: the split-K combine must not change the result."""
    spec, batch, k, v, pool, q = _case(dev, 21, [3000, 1, 0, 450, 16], 4)
    pkv.set_decode_ctas(ctas)
    try:
        out, ref = _decode_vs_oracle(dev, spec, batch, k, v, pool, q)
    finally:
        pkv.set_decode_ctas(0)
    assert max_abs(widen_out(out), ref) <= BF16_TOL
    assert torch.count_nonzero(out[2]) == 0        # empty sequence: zeros


def test_decode_int8_extreme_query_scales(dev):
    """Queries of very different magnitudes per head (the power-of-two fp16
    scaling of q) and a zero query head (uniform weights)."""
    spec, batch, k, v, pool, q = _case(dev, 31, [200, 90], 4)
    f = torch.tensor([1e-20, 1e-3, 1.0, 30.0] * 8, device=dev).view(1, 32, 1)
    q = (q.float() * f).to(torch.bfloat16)
    q[1, 5] = 0
    out, ref = _decode_vs_oracle(dev, spec, batch, k, v, pool, q, scale=0.05)
    assert max_abs(widen_out(out), ref) <= BF16_TOL


def test_decode_int8_full_size_sampled(dev):
    """The decode workload at full size (64 sequences of 1024..8192 tokens,
    Hq 32 / Hkv 8, 32-layer pool) over an int8 pool, in the configuration the
    benchmark times; checked on sampled (sequence, head) pairs."""
    w = make_workload("decode_gqa")
    bp = w.pool
    spec = PoolSpec(bp.num_blocks, bp.num_layers, bp.block_size, bp.num_kv_heads, bp.head_dim,
                    "i8")
    k = torch.empty(spec.shape, dtype=torch.uint8, device=dev)
    v = torch.empty_like(k)
    fill_pool_i8(k, v, spec, w.layer, w.seed)
    pool = pkv.Pool(k, v, spec.num_kv_heads, spec.head_dim)
    q = rand_rows((w.batch.batch, w.num_q_heads, spec.head_dim), "bf16", w.seed + 1, dev)
    out = gpu_decode(pool, w.layer, q, w.scale, w.batch, dev)
    torch.cuda.synchronize()
    kh, vh = host_layer(k, w.layer), host_layer(v, w.layer)
    del k, v
    rng = np.random.default_rng(5)
    pairs = [(int(b), int(h)) for b, h in zip(rng.integers(0, w.batch.batch, 24),
                                              rng.integers(0, w.num_q_heads, 24))]
    ref = Q.decode_attention_i8_pairs(kh, vh, 0, _bits(q), w.batch.block_tables,
                                      w.batch.seq_lens, w.batch.offsets, w.scale, pairs)
    got = widen_out(out)
    for b, h in pairs:
        assert max_abs(got[b, h], ref[(b, h)]) <= BF16_TOL, (b, h)
    assert pkv.device_error() == "PKV_OK"


def test_scatter_then_decode(dev):
    """A decode step on int8 pools, all on the GPU: append one token per
    sequence through the quantising scatter, then decode; the oracle runs its
    own scatter and decode from the same pools and inputs."""
    G, H, D = 4, 8, 128
    spec, batch, k, v, pool, q = _case(dev, 41, [100, 33, 512, 2], G)
    layer = 1
    kh, vh = _bits(k), _bits(v)
    B = batch.batch
    tok_seq = torch.arange(B, dtype=torch.int32, device=dev)
    tok_pos = torch.from_numpy((batch.seq_lens - 1).astype(np.int32)).to(dev)
    bt, lens, offs, _ = dev_batch(batch, dev)
    sm = torch.empty(B, dtype=torch.int64, device=dev)
    pkv.build_slot_mapping(pool, bt, offs, tok_seq, tok_pos, sm)
    # N(0,1) rows like the decode workload's (the wide-range rows of the
    # scatter tests would make bf16 output rounding alone exceed the tolerance)
    kn = rand_rows((B, H, D), "bf16", 77, dev)
    vn = rand_rows((B, H, D), "bf16", 78, dev)
    pkv.write_slots(pool, layer, kn, vn, sm)
    out = gpu_decode(pool, layer, q, D ** -0.5, batch, dev)
    torch.cuda.synchronize()
    slots = oracle.build_slot_mapping(batch.block_tables, batch.offsets,
                                      np.arange(B, dtype=np.int32),
                                      (batch.seq_lens - 1).astype(np.int32), spec.block_size)
    Q.write_slots_i8(kh, vh, layer, _bits(kn), _bits(vn), slots, H, D)
    assert np.array_equal(_bits(k), kh) and np.array_equal(_bits(v), vh)
    ref = Q.decode_attention_i8(kh, vh, layer, _bits(q), batch.block_tables, batch.seq_lens,
                                batch.offsets, D ** -0.5)
    assert max_abs(widen_out(out), ref) <= BF16_TOL


def test_int8_graph_replay(dev):
    """Scatter + decode on int8 pools captured in a CUDA graph and replayed
    with new inputs copied into the captured buffers."""
    G, H, D = 4, 8, 128
    spec, batch, k, v, pool, q = _case(dev, 51, [300, 41, 1200], G)
    layer = 0
    B = batch.batch
    bt, lens, offs, _ = dev_batch(batch, dev)
    slots = oracle.build_slot_mapping(batch.block_tables, batch.offsets,
                                      np.arange(B, dtype=np.int32),
                                      (batch.seq_lens - 1).astype(np.int32), spec.block_size)
    sm = torch.empty(B, dtype=torch.int64, device=dev)
    pkv.build_slot_mapping(pool, bt, offs, torch.arange(B, dtype=torch.int32, device=dev),
                           torch.from_numpy((batch.seq_lens - 1).astype(np.int32)).to(dev), sm)
    assert np.array_equal(sm.cpu().numpy(), slots)
    kn = torch.zeros((B, H, D), dtype=torch.bfloat16, device=dev)
    vn = torch.zeros_like(kn)
    qb = torch.zeros_like(q)
    out = torch.empty_like(q)
    ws = torch.empty(pkv.decode_workspace_size(B, H * G, D, dev), dtype=torch.uint8, device=dev)
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        pkv.write_slots(pool, layer, kn, vn, sm)
        pkv.decode_attention(pool, layer, qb, D ** -0.5, bt, lens, offs, out, ws)
    torch.cuda.current_stream().wait_stream(s)
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        pkv.write_slots(pool, layer, kn, vn, sm)
        pkv.decode_attention(pool, layer, qb, D ** -0.5, bt, lens, offs, out, ws)
    for step in range(3):
        kh, vh = _bits(k), _bits(v)
        nk = rand_rows((B, H, D), "bf16", 300 + step, dev)
        nv = rand_rows((B, H, D), "bf16", 400 + step, dev)
        nq = rand_rows(q.shape, "bf16", 500 + step, dev)
        kn.copy_(nk), vn.copy_(nv), qb.copy_(nq)
        graph.replay()
        torch.cuda.synchronize()
        Q.write_slots_i8(kh, vh, layer, _bits(nk), _bits(nv), slots, H, D)
        assert np.array_equal(_bits(k), kh) and np.array_equal(_bits(v), vh)
        ref = Q.decode_attention_i8(kh, vh, layer, _bits(nq), batch.block_tables,
                                    batch.seq_lens, batch.offsets, D ** -0.5)
        assert max_abs(widen_out(out), ref) <= BF16_TOL, step


def test_int8_block_moves_and_gather(dev):
    spec = PoolSpec(48, 3, 16, 8, 128, "i8")
    k, v, pool = _pools(dev, spec, 61)
    kh, vh = _bits(k), _bits(v)
    rng = np.random.default_rng(62)
    ids = rng.permutation(48)
    src, dst = ids[:6], ids[6:12]
    pkv.copy_blocks(pool, -1, torch.from_numpy(src.astype(np.int32)).to(dev),
                    torch.from_numpy(dst.astype(np.int32)).to(dev))
    oracle.copy_blocks(kh, vh, -1, src, dst)
    assert np.array_equal(_bits(k), kh) and np.array_equal(_bits(v), vh)
    out_ids = ids[12:20]
    hk = torch.empty((8, 3, 16, spec.row_bytes), dtype=torch.uint8, pin_memory=True)
    hv = torch.empty_like(hk, pin_memory=True)
    pkv.swap_out(pool, -1, torch.from_numpy(out_ids.astype(np.int32)).to(dev), hk, hv)
    torch.cuda.synchronize()
    rk, rv = oracle.swap_out(kh, vh, -1, out_ids)
    assert np.array_equal(hk.numpy(), rk) and np.array_equal(hv.numpy(), rv)
    in_ids = ids[20:28]
    pkv.swap_in(pool, -1, torch.from_numpy(in_ids.astype(np.int32)).to(dev), hk, hv)
    torch.cuda.synchronize()
    oracle.swap_in(kh, vh, -1, in_ids, rk, rv)
    assert np.array_equal(_bits(k), kh) and np.array_equal(_bits(v), vh)
    # gather returns the stored byte rows
    tables = [list(ids[28:33]), list(ids[33:36])]
    batch = _pack(tables, np.array([70, 33]), np.array([3, 0]))
    bt, lens, offs, cu = dev_batch(batch, dev)
    ko = torch.empty((batch.total_tokens, spec.row_bytes), dtype=torch.uint8, device=dev)
    vo = torch.empty_like(ko)
    pkv.gather(pool, 2, bt, lens, offs, cu, ko, vo)
    rk, rv = oracle.gather_batch(kh, vh, 2, batch.block_tables, batch.seq_lens, batch.offsets)
    assert np.array_equal(_bits(ko), rk) and np.array_equal(_bits(vo), rv)
