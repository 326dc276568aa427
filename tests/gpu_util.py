"""Helpers for the GPU parity tests: put a workload on the device, run the
library through its binding, and run the oracle on the same seeded inputs.

The oracle only ever sees values drawn by ``workloads`` (copied from the
device where the generator drew them); nothing the CUDA path computes is fed
to it."""

from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle
import paged_kv_cache_blk_gb300 as pkv
from workloads import fill_pool, new_pool, rand_rows, to_numpy_bits

BF16_TOL = 2e-2
F32_TOL = 1e-5


def need_gpu():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    pkv.build()
    pkv.load()
    return torch.device("cuda", 0)


def tol(dtype: str) -> float:
    return F32_TOL if dtype == "f32" else BF16_TOL


def dev_batch(batch, dev):
    t = lambda a, dt: torch.from_numpy(np.ascontiguousarray(a)).to(dev, dt)
    return (t(batch.block_tables, torch.int32), t(batch.seq_lens, torch.int32),
            t(batch.offsets, torch.int32), t(batch.cu_seqlens, torch.int64))


def make_pools(w, dev, fill=True):
    k, v = new_pool(w.pool, dev)
    if fill:
        fill_pool(k, v, w.pool, w.layer, w.seed, w.k_boost_frac, w.k_boost)
    return k, v


def host_layer(t: torch.Tensor, layer: int) -> np.ndarray:
    """Host copy of one layer of a pool as a 1-layer oracle pool."""
    return to_numpy_bits(t[:, layer:layer + 1])


def gpu_slots(pool, batch, tokens, dev):
    bt, _, offs, _ = dev_batch(batch, dev)
    seq = torch.from_numpy(tokens.token_seq).to(dev)
    pos = torch.from_numpy(tokens.token_pos).to(dev)
    sm = torch.empty(tokens.num_tokens, dtype=torch.int64, device=dev)
    pkv.build_slot_mapping(pool, bt, offs, seq, pos, sm)
    return sm


def oracle_slots(w, batch, tokens):
    return oracle.build_slot_mapping(batch.block_tables, batch.offsets, tokens.token_seq,
                                     tokens.token_pos, w.pool.block_size)


def gpu_gather(pool, layer, batch, dev):
    bt, lens, offs, cu = dev_batch(batch, dev)
    n = batch.total_tokens
    shape = (n, pool.num_kv_heads, pool.head_dim)
    ko = torch.empty(shape, dtype=pool.dtype, device=dev)
    vo = torch.empty(shape, dtype=pool.dtype, device=dev)
    pkv.gather(pool, layer, bt, lens, offs, cu, ko, vo)
    return ko, vo


def gpu_decode(pool, layer, q, scale, batch, dev):
    bt, lens, offs, _ = dev_batch(batch, dev)
    B, hq, D = q.shape
    out = torch.empty_like(q)
    ws = torch.empty(pkv.decode_workspace_size(B, hq, D, dev), dtype=torch.uint8, device=dev)
    pkv.decode_attention(pool, layer, q, scale, bt, lens, offs, out, ws)
    return out


def widen_out(t: torch.Tensor) -> np.ndarray:
    return t.detach().cpu().double().numpy()


def max_abs(a: np.ndarray, b: np.ndarray) -> float:
    if a.size == 0:
        return 0.0
    return float(np.max(np.abs(a - b)))
