"""Oracle parity of the benchmarked decode step at its full size.

``bench.py`` times ``pkv_decode_step`` on the decode-GQA workload (64
sequences, lengths U[1024, 8192], Hq 32 over Hkv 8, D 128, layer 7 of a
16384 x 32 x 16 x 8 x 128 pool) with the library's default grid.  These tests
run that same call on the same seeded inputs, for the bf16 pool and for the
int8 pool of the same geometry, and check:

  * the whole accessed layer after the step, bit for bit, against the oracle's
    slot mapping and scatter (quantising scatter for int8) of each sequence's
    new row at position seq_len - 1 into a host copy of the layer taken
    before the step;
  * every one of the 64 x 32 outputs against the oracle's fp64 decode
    attention over that layer, within max-abs 2e-2.
"""

import numpy as np
import pytest
import torch

import oracle
import paged_kv_cache_blk_gb300 as pkv
from workloads import (PoolSpec, fill_pool, fill_pool_i8, make_workload, new_pool, rand_rows,
                       to_numpy_bits)

from gpu_util import dev_batch, host_layer, max_abs, need_gpu, widen_out

pytestmark = pytest.mark.gpu

TOL = 2e-2


@pytest.fixture(scope="module")
def dev():
    d = need_gpu()
    pkv.set_validate(False)
    pkv.set_decode_ctas(0)          # the default grid: one CTA per SM, as benchmarked
    pkv.device_error(clear=True)
    yield d
    torch.cuda.empty_cache()


def _bench_inputs(w, dev):
    """q and the new K / V rows exactly as the benchmark draws them."""
    B, hq, D = w.batch.batch, w.num_q_heads, w.pool.head_dim
    T = w.tokens.num_tokens
    row = (w.pool.num_kv_heads, D)
    q = rand_rows((B, hq, D), "bf16", 1000, dev)
    kn = rand_rows((T,) + row, "bf16", 1001, dev)
    vn = rand_rows((T,) + row, "bf16", 1002, dev)
    return q, kn, vn


def _step(pool, w, q, kn, vn, dev):
    bt, lens, offs, _ = dev_batch(w.batch, dev)
    B, hq, D = q.shape
    out = torch.full_like(q, float("nan"))
    ws = torch.empty(pkv.decode_workspace_size(B, hq, D, dev), dtype=torch.uint8, device=dev)
    pkv.decode_step(pool, w.layer, q, w.scale, bt, lens, offs, kn, vn, out, ws)
    torch.cuda.synchronize()
    return out


def _new_token_slots(w):
    # the step's new token of sequence b sits at position seq_len - 1
    seqs = np.arange(w.batch.batch, dtype=np.int32)
    pos = (w.batch.seq_lens - 1).astype(np.int32)
    assert np.array_equal(w.tokens.token_seq, seqs) and np.array_equal(w.tokens.token_pos, pos)
    return oracle.build_slot_mapping(w.batch.block_tables, w.batch.offsets, seqs, pos,
                                     w.pool.block_size)


def test_decode_step_full_size_bf16(dev):
    w = make_workload("decode_gqa")
    k, v = new_pool(w.pool, dev)
    fill_pool(k, v, w.pool, w.layer, w.seed)
    q, kn, vn = _bench_inputs(w, dev)
    kh, vh = host_layer(k, w.layer), host_layer(v, w.layer)
    out = _step(pkv.Pool(k, v), w, q, kn, vn, dev)
    oracle.write_slots(kh, vh, 0, to_numpy_bits(kn), to_numpy_bits(vn), _new_token_slots(w))
    assert np.array_equal(host_layer(k, w.layer), kh), "K layer differs after the step"
    assert np.array_equal(host_layer(v, w.layer), vh), "V layer differs after the step"
    ref = oracle.decode_attention(kh, vh, 0, to_numpy_bits(q), w.batch.block_tables,
                                  w.batch.seq_lens, w.batch.offsets, w.scale)
    got = widen_out(out)
    assert got.shape == (64, 32, 128) and np.isfinite(got).all()
    assert max_abs(got, ref) <= TOL
    assert pkv.device_error(clear=True) == "PKV_OK"
    del k, v
    torch.cuda.empty_cache()


def test_decode_step_full_size_int8(dev):
    from oracle import quant as Q
    w = make_workload("decode_gqa")
    sp = w.pool
    spec = PoolSpec(sp.num_blocks, sp.num_layers, sp.block_size, sp.num_kv_heads, sp.head_dim,
                    "i8")
    k = torch.empty(spec.shape, dtype=torch.uint8, device=dev)
    v = torch.empty_like(k)
    fill_pool_i8(k, v, spec, w.layer, w.seed)
    q, kn, vn = _bench_inputs(w, dev)
    kh, vh = host_layer(k, w.layer), host_layer(v, w.layer)
    out = _step(pkv.Pool(k, v, spec.num_kv_heads, spec.head_dim), w, q, kn, vn, dev)
    Q.write_slots_i8(kh, vh, 0, to_numpy_bits(kn), to_numpy_bits(vn), _new_token_slots(w),
                     spec.num_kv_heads, spec.head_dim)
    assert np.array_equal(host_layer(k, w.layer), kh), "K layer differs after the step"
    assert np.array_equal(host_layer(v, w.layer), vh), "V layer differs after the step"
    ref = Q.decode_attention_i8(kh, vh, 0, to_numpy_bits(q), w.batch.block_tables,
                                w.batch.seq_lens, w.batch.offsets, w.scale)
    got = widen_out(out)
    assert got.shape == (64, 32, 128) and np.isfinite(got).all()
    assert max_abs(got, ref) <= TOL
    assert pkv.device_error(clear=True) == "PKV_OK"
    del k, v
    torch.cuda.empty_cache()
