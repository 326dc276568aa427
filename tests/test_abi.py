"""The C ABI library without a GPU: it builds for sm_103a, loads, exports
every entry point include/pkv.h declares, and its host-side argument checks
return the documented status before touching the device."""

import ctypes
import os
import re
import subprocess

import pytest

import paged_kv_cache_blk_gb300 as pkv
from paged_kv_cache_blk_gb300 import _binding as B

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "pkv.h")


def declared_symbols():
    text = open(HEADER).read()
    return re.findall(r"^PKV_API\s+[\w\s\*]+?\b(pkv_\w+)\s*\(", text, flags=re.M)


@pytest.fixture(scope="module")
def lib():
    pkv.build()
    return pkv.load()


def test_header_declares_the_hot_path():
    names = set(declared_symbols())
    for n in ("pkv_build_slot_mapping", "pkv_write_slots", "pkv_gather",
              "pkv_decode_attention", "pkv_decode_workspace_size"):
        assert n in names


def test_every_declared_symbol_is_exported(lib):
    names = declared_symbols()
    assert len(names) >= 12
    out = subprocess.run(["nm", "-D", "--defined-only", pkv.library_path()],
                         capture_output=True, text=True, check=True).stdout
    exported = {line.split()[-1] for line in out.splitlines() if " T " in line}
    for n in names:
        assert n in exported, n
        assert hasattr(lib, n)
    # nothing but the C ABI is exported
    assert exported == set(names)


def test_binding_covers_every_symbol():
    assert set(declared_symbols()) == set(B._SIGS)


def _pool(**kw):
    base = dict(k_cache=16, v_cache=32, num_blocks=8, num_layers=2, block_size=16,
                num_kv_heads=2, head_dim=64, dtype=1)
    base.update(kw)
    return B._PoolStruct(base["k_cache"], base["v_cache"], base["num_blocks"], base["num_layers"],
                         base["block_size"], base["num_kv_heads"], base["head_dim"], base["dtype"])


S = B.STATUS_CODES


def test_host_checks_pool(lib):
    assert lib.pkv_write_slots(None, 0, 16, 16, 8, 1, None) == S["PKV_ERR_INVALID_ARG"]
    for bad, want in [(dict(dtype=7), "PKV_ERR_UNSUPPORTED"),
                      (dict(block_size=3), "PKV_ERR_INVALID_ARG"),
                      (dict(block_size=2048), "PKV_ERR_INVALID_ARG"),
                      (dict(num_blocks=0), "PKV_ERR_INVALID_ARG"),
                      (dict(num_layers=0), "PKV_ERR_INVALID_ARG"),
                      (dict(k_cache=0), "PKV_ERR_INVALID_ARG"),
                      (dict(v_cache=8), "PKV_ERR_INVALID_ARG"),
                      (dict(num_kv_heads=1, head_dim=4), "PKV_ERR_UNSUPPORTED")]:
        p = _pool(**bad)
        assert lib.pkv_write_slots(ctypes.byref(p), 0, 16, 16, 8, 1, None) == S[want], bad


def test_host_checks_scatter(lib):
    p = ctypes.byref(_pool())
    assert lib.pkv_write_slots(p, 2, 16, 16, 8, 1, None) == S["PKV_ERR_INVALID_ARG"]   # layer
    assert lib.pkv_write_slots(p, -1, 16, 16, 8, 1, None) == S["PKV_ERR_INVALID_ARG"]
    assert lib.pkv_write_slots(p, 0, 16, 16, 8, -1, None) == S["PKV_ERR_INVALID_ARG"]
    assert lib.pkv_write_slots(p, 0, 16, 16, 8, 0, None) == S["PKV_OK"]                # empty
    assert lib.pkv_write_slots(p, 0, 0, 16, 8, 1, None) == S["PKV_ERR_INVALID_ARG"]
    assert lib.pkv_write_slots(p, 0, 24, 16, 8, 1, None) == S["PKV_ERR_INVALID_ARG"]   # align
    assert lib.pkv_write_slots(p, 0, 16, 16, 4, 1, None) == S["PKV_ERR_INVALID_ARG"]


def test_host_checks_gather(lib):
    p = ctypes.byref(_pool())
    assert lib.pkv_gather(p, 0, 16, 4, 16, 16, 0, 16, 0, 16, 16, None) == S["PKV_OK"]
    assert lib.pkv_gather(p, 0, 16, 4, 16, 16, 0, 16, 5, 16, 16, None) == S["PKV_ERR_INVALID_ARG"]
    assert lib.pkv_gather(p, 0, 16, 0, 16, 16, 2, 16, 5, 16, 16, None) == S["PKV_ERR_INVALID_ARG"]
    assert lib.pkv_gather(p, 0, 16, 4, 16, 16, 2, None, 5, 16, 16, None) == S["PKV_ERR_INVALID_ARG"]
    assert lib.pkv_gather(p, 0, 16, 4, 16, 16, 2, 16, 5, 17, 16, None) == S["PKV_ERR_INVALID_ARG"]
    assert lib.pkv_gather(p, 5, 16, 4, 16, 16, 2, 16, 5, 16, 16, None) == S["PKV_ERR_INVALID_ARG"]


def test_host_checks_slot_mapping(lib):
    p = ctypes.byref(_pool(k_cache=0, v_cache=0))    # geometry only: no tensors needed
    assert lib.pkv_build_slot_mapping(p, 16, 4, None, 2, 16, 16, 0, 16, None) == S["PKV_OK"]
    assert lib.pkv_build_slot_mapping(p, 16, 4, None, 2, 16, 16, -1, 16, None) == S["PKV_ERR_INVALID_ARG"]
    assert lib.pkv_build_slot_mapping(p, None, 4, None, 2, 16, 16, 3, 16, None) == S["PKV_ERR_INVALID_ARG"]
    assert lib.pkv_build_slot_mapping(p, 16, 4, None, 2, 16, 16, 3, 12, None) == S["PKV_ERR_INVALID_ARG"]


def test_host_checks_decode(lib):
    p = ctypes.byref(_pool())
    args = lambda **kw: [kw.get("layer", 0), kw.get("q", 16), kw.get("hq", 8), 0.1, 16, 4, 16, None,
                         kw.get("batch", 2), kw.get("out", 16), kw.get("ws", 16), 1 << 20, None]
    assert lib.pkv_decode_attention(p, *args(hq=7)) == S["PKV_ERR_INVALID_ARG"]
    assert lib.pkv_decode_attention(p, *args(hq=0)) == S["PKV_ERR_INVALID_ARG"]
    assert lib.pkv_decode_attention(p, *args(hq=2 * 16)) == S["PKV_ERR_UNSUPPORTED"]   # group 16
    assert lib.pkv_decode_attention(p, *args(layer=9)) == S["PKV_ERR_INVALID_ARG"]
    assert lib.pkv_decode_attention(p, *args(batch=0)) == S["PKV_OK"]
    assert lib.pkv_decode_attention(p, *args(q=8)) == S["PKV_ERR_INVALID_ARG"]
    assert lib.pkv_decode_attention(p, *args(ws=0)) == S["PKV_ERR_WORKSPACE"]
    p96 = ctypes.byref(_pool(head_dim=96))
    assert lib.pkv_decode_attention(p96, *args()) == S["PKV_ERR_UNSUPPORTED"]
    nan = [0, 16, 8, float("nan"), 16, 4, 16, None, 2, 16, 16, 1 << 20, None]
    assert lib.pkv_decode_attention(p, *nan) == S["PKV_ERR_INVALID_ARG"]


def test_host_checks_append(lib):
    p = ctypes.byref(_pool())
    args = lambda **kw: [kw.get("layer", 0), kw.get("bt", 16), 4, None, kw.get("batch", 2),
                         kw.get("seq", 16), kw.get("pos", 16), kw.get("n", 3),
                         kw.get("k", 16), kw.get("v", 16), kw.get("sm", None), None]
    assert lib.pkv_append_tokens(p, *args(n=0)) == S["PKV_OK"]
    assert lib.pkv_append_tokens(p, *args(layer=2)) == S["PKV_ERR_INVALID_ARG"]
    assert lib.pkv_append_tokens(p, *args(n=-1)) == S["PKV_ERR_INVALID_ARG"]
    assert lib.pkv_append_tokens(p, *args(k=24)) == S["PKV_ERR_INVALID_ARG"]   # align
    assert lib.pkv_append_tokens(p, *args(seq=0)) == S["PKV_ERR_INVALID_ARG"]
    assert lib.pkv_append_tokens(p, *args(sm=12)) == S["PKV_ERR_INVALID_ARG"]  # slot align
    assert lib.pkv_append_tokens(p, *args(bt=0)) == S["PKV_ERR_INVALID_ARG"]


def test_host_checks_int8_pools(lib):
    # int8 pools: codes must fill 16-byte multiples, the quantising scatter
    # takes head sizes 32..256 (powers of two), prefill takes bf16 pools only
    p8 = ctypes.byref(_pool(dtype=2, num_kv_heads=1, head_dim=8))
    assert lib.pkv_write_slots(p8, 0, 16, 16, 8, 1, None) == S["PKV_ERR_UNSUPPORTED"]
    p96 = ctypes.byref(_pool(dtype=2, num_kv_heads=2, head_dim=96))
    assert lib.pkv_write_slots(p96, 0, 16, 16, 8, 1, None) == S["PKV_ERR_UNSUPPORTED"]
    p = ctypes.byref(_pool(dtype=2))
    assert lib.pkv_write_slots(p, 0, 16, 16, 8, 0, None) == S["PKV_OK"]
    assert lib.pkv_write_slots(p, 0, 24, 16, 8, 1, None) == S["PKV_ERR_INVALID_ARG"]
    dec = [0, 16, 8, 0.1, 16, 4, 16, None, 2, 16, 16, 1 << 20, None]
    assert lib.pkv_decode_attention(p96, *dec) == S["PKV_ERR_UNSUPPORTED"]
    pre = [0, 16, 8, 0.1, 16, 4, 16, None, 16, 2, 4, 4, 16, None]
    assert lib.pkv_prefill_attention(p, *pre) == S["PKV_ERR_UNSUPPORTED"]
    assert B.int8_row_bytes(8, 128) == 1056 and B.int8_row_bytes(3, 32) == 112


def test_host_checks_decode_step(lib):
    # the fused decode step: new rows required and 16-byte aligned (int8
    # pools too: they quantise the new rows)
    p = ctypes.byref(_pool())
    head = [0, 16, 8, 0.1, 16, 4, 16, None, 2]
    tail = [16, 16, 1 << 20, None]
    assert lib.pkv_decode_step(p, *head[:-1], 0, None, None, *tail) == S["PKV_OK"]
    assert lib.pkv_decode_step(p, *head, None, 16, *tail) == S["PKV_ERR_INVALID_ARG"]
    assert lib.pkv_decode_step(p, *head, 16, None, *tail) == S["PKV_ERR_INVALID_ARG"]
    assert lib.pkv_decode_step(p, *head, 24, 16, *tail) == S["PKV_ERR_INVALID_ARG"]
    p8 = ctypes.byref(_pool(dtype=2))
    assert lib.pkv_decode_step(p8, *head, 24, 16, *tail) == S["PKV_ERR_INVALID_ARG"]
    p96 = ctypes.byref(_pool(dtype=2, num_kv_heads=2, head_dim=96))
    assert lib.pkv_decode_step(p96, *head, 16, 16, *tail) == S["PKV_ERR_UNSUPPORTED"]
    assert lib.pkv_decode_step(p, 3, *head[1:], 16, 16, *tail) == S["PKV_ERR_INVALID_ARG"]


def test_options_and_strings(lib):
    assert lib.pkv_set_decode_ctas(-1) == S["PKV_ERR_INVALID_ARG"]
    assert lib.pkv_set_decode_ctas(0) == S["PKV_OK"]
    assert lib.pkv_set_validate(1) == 0 and lib.pkv_get_validate() == 1
    assert lib.pkv_set_validate(0) == 0 and lib.pkv_get_validate() == 0
    assert lib.pkv_set_decode_events(None, None) == 0
    assert lib.pkv_version() == 100
    for code in range(8):
        assert lib.pkv_status_string(code)
    assert b"unknown" in lib.pkv_status_string(99)
    assert lib.pkv_device_error(None, 0) == S["PKV_ERR_INVALID_ARG"]


def test_binding_fails_loudly_without_library(tmp_path):
    with pytest.raises(RuntimeError, match="not built"):
        B.load(str(tmp_path / "missing.so"))


def test_host_checks_block_moves(lib):
    p = ctypes.byref(_pool())
    assert lib.pkv_copy_blocks(p, 0, 16, 16, 0, None) == S["PKV_OK"]
    assert lib.pkv_copy_blocks(p, 2, 16, 16, 1, None) == S["PKV_ERR_INVALID_ARG"]    # layer
    assert lib.pkv_copy_blocks(p, -2, 16, 16, 1, None) == S["PKV_ERR_INVALID_ARG"]
    assert lib.pkv_copy_blocks(p, -1, None, 16, 1, None) == S["PKV_ERR_INVALID_ARG"]
    assert lib.pkv_copy_blocks(None, 0, 16, 16, 1, None) == S["PKV_ERR_INVALID_ARG"]
    # host buffers too small for n blocks: refused before any device call
    run = 16 * 2 * 64 * 2 * 2                                  # all layers: L*bs*Hkv*D*e
    assert lib.pkv_swap_out(p, -1, 16, 3, 16, 16, 3 * run - 16, None) == S["PKV_ERR_INVALID_ARG"]
    assert lib.pkv_swap_in(p, 0, 16, 3, 16, 16, 3 * run // 2 - 1, None) == S["PKV_ERR_INVALID_ARG"]
    assert lib.pkv_swap_out(p, 0, 16, 0, None, None, 0, None) == S["PKV_OK"]
    assert lib.pkv_swap_out(p, 0, 16, 2, 8, 16, 1 << 20, None) == S["PKV_ERR_INVALID_ARG"]
