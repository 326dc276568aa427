"""The allocation-free decode entry point (pkv_decode_attention_static).

Callers that cannot allocate device memory where they run decode attention
(serving processes whose memory manager owns all device memory, plugin
runtimes whose execute step must not allocate, plain C programs without a
device allocator) pass no workspace: the library keeps the scratch in its own
fixed device array.  This checks, through the C ABI, that two calls in a row
give the oracle's results and the same results as pkv_decode_attention with a
caller workspace, and that a shape too large for the array is refused.

The file is named to be collected last, so a run that stops at the first
failure has run every other test first; it also passes on its own in a fresh
process."""

import ctypes

import numpy as np
import pytest
import torch

import oracle
import paged_kv_cache_blk_gb300 as pkv
from paged_kv_cache_blk_gb300 import _binding as B
from workloads import rand_rows, small_workload, to_numpy_bits

from gpu_util import dev_batch, gpu_decode, host_layer, make_pools, max_abs, need_gpu, widen_out

pytestmark = pytest.mark.gpu

TOL = 2e-2  # bf16 decode tolerance used by every decode parity test


@pytest.fixture(scope="module")
def dev():
    d = need_gpu()
    pkv.set_decode_ctas(0)
    pkv.set_validate(False)
    return d


def _static_call(pool, layer, q, scale, bt, lens, offs, out):
    lib = pkv.load()
    st = lib.pkv_decode_attention_static(
        pool.ref, layer, q.data_ptr(), q.shape[1], float(scale), bt.data_ptr(), bt.shape[1],
        lens.data_ptr(), offs.data_ptr(), lens.numel(), out.data_ptr(),
        torch.cuda.current_stream(q.device).cuda_stream)
    return st


def test_static_scratch_matches_workspace_entry(dev):
    w = small_workload(seed=81, num_blocks=512, num_layers=2, block_size=16, num_kv_heads=8,
                       head_dim=128, dtype="bf16", batch=12, min_len=1, max_len=1500,
                       num_q_heads=32, shared_prefix=2)
    k, v = make_pools(w, dev)
    pool = pkv.Pool(k, v)
    bt, lens, offs, _ = dev_batch(w.batch, dev)
    kh, vh = host_layer(k, w.layer), host_layer(v, w.layer)
    for call, seed in enumerate((83, 84)):          # two calls in a row
        q = rand_rows((12, 32, 128), "bf16", seed, dev)
        ref = gpu_decode(pool, w.layer, q, w.scale, w.batch, dev)
        out = torch.full_like(q, float("nan"))
        assert _static_call(pool, w.layer, q, w.scale, bt, lens, offs, out) == 0, call
        torch.cuda.synchronize()
        assert torch.isfinite(out.float()).all(), call
        err = (out.double() - ref.double()).abs().max().item()
        assert err <= TOL, (call, err)
        want = oracle.decode_attention(kh, vh, 0, to_numpy_bits(q), w.batch.block_tables,
                                       w.batch.seq_lens, w.batch.offsets, w.scale)
        assert max_abs(widen_out(out), want) <= TOL, call


def test_static_scratch_binding_and_fp32(dev):
    w = small_workload(seed=85, num_blocks=128, num_layers=1, block_size=16, num_kv_heads=4,
                       head_dim=64, dtype="f32", batch=5, min_len=0, max_len=300, layer=0,
                       num_q_heads=4)
    k, v = make_pools(w, dev)
    pool = pkv.Pool(k, v)
    bt, lens, offs, _ = dev_batch(w.batch, dev)
    kh, vh = host_layer(k, 0), host_layer(v, 0)
    for seed in (86, 87):
        q = rand_rows((5, 4, 64), "f32", seed, dev)
        ref = gpu_decode(pool, 0, q, w.scale, w.batch, dev)
        out = torch.empty_like(q)
        pkv.decode_attention_static(pool, 0, q, w.scale, bt, lens, offs, out)
        torch.cuda.synchronize()
        assert (out.double() - ref.double()).abs().max().item() <= 1e-5
        want = oracle.decode_attention(kh, vh, 0, to_numpy_bits(q), w.batch.block_tables,
                                       w.batch.seq_lens, w.batch.offsets, w.scale)
        assert max_abs(widen_out(out), want) <= 1e-5


def test_static_scratch_refuses_oversized_shape(dev):
    w = small_workload(seed=88, num_blocks=64, num_layers=1, block_size=16, num_kv_heads=8,
                       head_dim=128, dtype="bf16", batch=3, min_len=1, max_len=40, layer=0,
                       num_q_heads=32)
    k, v = make_pools(w, dev)
    pool = pkv.Pool(k, v)
    # a batch whose scratch exceeds the fixed array (checked on the host)
    B_big = 2000
    assert pkv.decode_workspace_size(B_big, 64, 128, dev) > (16 << 20)
    q = torch.zeros((B_big, 64, 128), dtype=torch.bfloat16, device=dev)
    out = torch.zeros_like(q)
    bt = torch.zeros((B_big, 1), dtype=torch.int32, device=dev)
    lens = torch.zeros(B_big, dtype=torch.int32, device=dev)
    offs = torch.zeros(B_big, dtype=torch.int32, device=dev)
    pool8 = pkv.Pool(k, v)
    st = _static_call(pool8, 0, q, 0.1, bt, lens, offs, out)
    assert st == B.STATUS_CODES["PKV_ERR_WORKSPACE"]
    assert torch.count_nonzero(out) == 0             # nothing was enqueued
