"""The split-K merge of paged decode attention (partial pass + combine).

A sequence cut by the CTA ranges leaves one partial softmax state per CTA it
spans; the combine pass merges them with the log-sum-exp rule.  These tests
check the merged outputs against the fp64 oracle where a sequence is cut into
many states (more than a warp's width of them), where empty sequences sit
between cut ones, and where one workspace serves many calls of different
shapes."""

import pytest
import torch

import oracle
import paged_kv_cache_blk_gb300 as pkv
from workloads import rand_rows, small_workload, to_numpy_bits

from gpu_util import dev_batch, host_layer, make_pools, max_abs, need_gpu, tol, widen_out

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def dev():
    d = need_gpu()
    pkv.set_decode_ctas(0)
    pkv.set_validate(False)
    pkv.device_error(clear=True)
    yield d
    pkv.set_decode_ctas(0)
    pkv.set_validate(False)
    torch.cuda.empty_cache()


def _case(seed, lens, dev, dtype="bf16", G=4, hkv=8, D=128, num_blocks=2048):
    w = small_workload(seed=seed, num_blocks=num_blocks, num_layers=1, block_size=16,
                       num_kv_heads=hkv, head_dim=D, dtype=dtype, lens=lens, layer=0,
                       num_q_heads=hkv * G)
    k, v = make_pools(w, dev)
    pool = pkv.Pool(k, v)
    q = rand_rows((len(lens), hkv * G, D), dtype, seed + 7, dev)
    ref = oracle.decode_attention(host_layer(k, 0), host_layer(v, 0), 0, to_numpy_bits(q),
                                  w.batch.block_tables, w.batch.seq_lens, w.batch.offsets,
                                  w.scale)
    return w, pool, q, ref


@pytest.mark.parametrize("ctas", [0, 7, 152, 3000])
def test_one_workspace_many_calls(dev, ctas):
    """One workspace reused by calls of different batches and lengths, never
    cleared between them: every result matches the oracle."""
    pkv.set_decode_ctas(ctas)  # the workspace size depends on the grid
    try:
        ws = torch.empty(pkv.decode_workspace_size(64, 32, 128, dev), dtype=torch.uint8,
                         device=dev)
        for i, lens in enumerate([[900, 17, 2000, 1], [1, 2, 3], [3000] * 5,
                                  list(range(0, 640, 10)), [4095]]):
            w, pool, q, ref = _case(100 + i, lens, dev)
            bt, sl, offs, _ = dev_batch(w.batch, dev)
            out = torch.empty_like(q)
            pkv.decode_attention(pool, 0, q, w.scale, bt, sl, offs, out, ws)
            assert max_abs(widen_out(out), ref) <= tol("bf16"), (ctas, i)
    finally:
        pkv.set_decode_ctas(0)
    assert pkv.device_error(clear=True) == "PKV_OK"


@pytest.mark.parametrize("dtype,G,hkv,D", [("bf16", 4, 8, 128), ("bf16", 8, 1, 64),
                                           ("f32", 2, 4, 128), ("f32", 1, 2, 64)])
def test_single_sequence_over_every_cta(dev, dtype, G, hkv, D):
    """One long sequence split over the whole grid: up to one partial state
    per CTA (150 of them at most here) merged into one output row."""
    w, pool, q, ref = _case(200, [2400], dev, dtype=dtype, G=G, hkv=hkv, D=D)
    bt, sl, offs, _ = dev_batch(w.batch, dev)
    for ctas in (0, 40, 150):
        pkv.set_decode_ctas(ctas)
        try:
            out = torch.empty_like(q)
            ws = torch.empty(pkv.decode_workspace_size(1, hkv * G, D, dev), dtype=torch.uint8,
                             device=dev)
            pkv.decode_attention(pool, 0, q, w.scale, bt, sl, offs, out, ws)
        finally:
            pkv.set_decode_ctas(0)
        assert max_abs(widen_out(out), ref) <= tol(dtype), ctas


@pytest.mark.parametrize("ctas", [1, 3, 5, 152])
def test_empty_sequences_between_cut_ones(dev, ctas):
    """Empty sequences at the ends and between cut sequences: zero rows, and
    the other sequences' states still merge into the right rows."""
    lens = [0, 500, 0, 0, 700, 0, 1, 0, 1300, 0]
    w, pool, q, ref = _case(300, lens, dev)
    bt, sl, offs, _ = dev_batch(w.batch, dev)
    out = torch.full_like(q, float("nan"))
    pkv.set_decode_ctas(ctas)
    try:
        ws = torch.empty(pkv.decode_workspace_size(len(lens), 32, 128, dev),
                         dtype=torch.uint8, device=dev)
        pkv.decode_attention(pool, 0, q, w.scale, bt, sl, offs, out, ws)
    finally:
        pkv.set_decode_ctas(0)
    assert max_abs(widen_out(out), ref) <= tol("bf16")
    for b, n in enumerate(lens):
        if n == 0:
            assert int(torch.count_nonzero(out[b])) == 0, b
