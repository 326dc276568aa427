"""ctypes binding of libpkv: argument marshalling only.

Each function has the name of the C call without the ``pkv_`` prefix, takes
torch tensors, passes their device pointers and the current torch stream to
the library, and raises :class:`PkvError` on any status other than
``PKV_OK``.  Every step of the path runs in the library's CUDA kernels; there
is no Python or CPU fallback, and a missing library is an error.
"""

from __future__ import annotations

import ctypes
import os
from typing import List, Optional, Sequence, Tuple

import numpy as np
import torch

from . import build as _build

_STATUS = {
    0: "PKV_OK", 1: "PKV_ERR_INVALID_ARG", 2: "PKV_ERR_CAPACITY", 3: "PKV_ERR_UNSUPPORTED",
    4: "PKV_ERR_WORKSPACE", 5: "PKV_ERR_INDEX", 6: "PKV_ERR_CUDA", 7: "PKV_ERR_TIMEOUT",
    8: "PKV_ERR_NO_BLOCKS",
}
STATUS_CODES = {v: k for k, v in _STATUS.items()}
_DTYPE = {torch.float32: 0, torch.bfloat16: 1, torch.uint8: 2}


class PkvError(RuntimeError):
    def __init__(self, status: int, where: str, message: str):
        self.status = status
        self.name = _STATUS.get(status, str(status))
        super().__init__(f"{where}: {self.name} ({message})")


class _PoolStruct(ctypes.Structure):
    _fields_ = [
        ("k_cache", ctypes.c_void_p),
        ("v_cache", ctypes.c_void_p),
        ("num_blocks", ctypes.c_int64),
        ("num_layers", ctypes.c_int32),
        ("block_size", ctypes.c_int32),
        ("num_kv_heads", ctypes.c_int32),
        ("head_dim", ctypes.c_int32),
        ("dtype", ctypes.c_int32),
    ]


_lib = None
_P, _I32, _I64, _F32, _SZ = (ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_float,
                             ctypes.c_size_t)
_SIGS = {
    "pkv_build_slot_mapping": (_I32, [_P, _P, _I32, _P, _I32, _P, _P, _I64, _P, _P]),
    "pkv_write_slots": (_I32, [_P, _I32, _P, _P, _P, _I64, _P]),
    "pkv_append_tokens": (_I32, [_P, _I32, _P, _I32, _P, _I32, _P, _P, _I64, _P, _P, _P, _P]),
    "pkv_gather": (_I32, [_P, _I32, _P, _I32, _P, _P, _I32, _P, _I64, _P, _P, _P]),
    "pkv_decode_workspace_size": (_SZ, [_I32, _I32, _I32]),
    "pkv_decode_attention": (_I32, [_P, _I32, _P, _I32, _F32, _P, _I32, _P, _P, _I32, _P, _P,
                                    _SZ, _P]),
    "pkv_decode_attention_static": (_I32, [_P, _I32, _P, _I32, _F32, _P, _I32, _P, _P, _I32,
                                           _P, _P]),
    "pkv_decode_shared_prefix_workspace_size": (_SZ, [_P, _I32, _I32, _I32]),
    "pkv_decode_attention_shared_prefix": (_I32, [_P, _I32, _P, _I32, _F32, _P, _I32, _P, _P,
                                                  _I32, _I32, _P, _P, _SZ, _P]),
    "pkv_decode_step": (_I32, [_P, _I32, _P, _I32, _F32, _P, _I32, _P, _P, _I32, _P, _P, _P, _P,
                               _SZ, _P]),
    "pkv_copy_blocks": (_I32, [_P, _I32, _P, _P, _I32, _P]),
    "pkv_swap_out": (_I32, [_P, _I32, _P, _I32, _P, _P, _SZ, _P]),
    "pkv_swap_in": (_I32, [_P, _I32, _P, _I32, _P, _P, _SZ, _P]),
    "pkv_prefill_attention": (_I32, [_P, _I32, _P, _I32, _F32, _P, _I32, _P, _P, _P, _I32, _I64,
                                      _I32, _P, _P]),
    "pkv_set_decode_ctas": (_I32, [_I32]),
    "pkv_set_decode_events": (_I32, [_P, _P]),
    "pkv_set_validate": (_I32, [_I32]),
    "pkv_set_wait_limit_ns": (_I32, [ctypes.c_uint64]),
    "pkv_get_wait_limit_ns": (ctypes.c_uint64, []),
    "pkv_set_debug_skip_fill": (_I32, [_I32]),
    "pkv_get_validate": (_I32, []),
    "pkv_device_error": (_I32, [ctypes.POINTER(ctypes.c_int32), _I32]),
    "pkv_alloc_create": (_I32, [_I64, _I32, _P, ctypes.POINTER(ctypes.c_void_p)]),
    "pkv_alloc_destroy": (_I32, [_P]),
    "pkv_alloc_num_free": (_I64, [_P]),
    "pkv_alloc_ref_count": (_I32, [_P, _I64]),
    "pkv_alloc_blocks": (_I32, [_P, _I64, _P]),
    "pkv_alloc_inc_ref": (_I32, [_P, _I32]),
    "pkv_alloc_dec_ref": (_I32, [_P, _I32]),
    "pkv_seq_new": (_I32, [_P, _I64, _I32]),
    "pkv_seq_share": (_I32, [_P, _I64, _P, _I32, _I64]),
    "pkv_seq_append": (_I32, [_P, _I64, _I64, _P, _P, _P, _P]),
    "pkv_seq_append_batch": (_I32, [_P, _P, _I32, _P, _P, _P, _P, _P]),
    "pkv_seq_fork": (_I32, [_P, _I64, _I64]),
    "pkv_seq_free": (_I32, [_P, _I64]),
    "pkv_seq_info": (_I32, [_P, _I64, _P, _P, _P]),
    "pkv_seq_tables": (_I32, [_P, _P, _I32, _I32, _P, _P, _P]),
    "pkv_alloc_stats": (_I32, [_P, _P, _P, _P]),
    "pkv_status_string": (ctypes.c_char_p, [_I32]),
    "pkv_version": (_I32, []),
}


def library_path() -> str:
    return _build.LIB


def load(path: Optional[str] = None) -> ctypes.CDLL:
    """Load libpkv.so (built by ``build()``); raises if it is missing."""
    global _lib
    if _lib is not None and path is None:
        return _lib
    p = path or _build.LIB
    if not os.path.exists(p):
        raise RuntimeError(f"libpkv is not built ({p} missing): run __graft_entry__.build() "
                           "or python -m paged_kv_cache_blk_gb300.build")
    lib = ctypes.CDLL(p)
    for name, (res, args) in _SIGS.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    if path is None:
        _lib = lib
    return lib


def _check(status: int, where: str) -> None:
    if status != 0:
        msg = load().pkv_status_string(status).decode()
        raise PkvError(status, where, msg)


def _ptr(t: Optional[torch.Tensor]) -> Optional[int]:
    return None if t is None else t.data_ptr()


def _stream(dev: torch.device) -> int:
    return torch.cuda.current_stream(dev).cuda_stream


def int8_row_bytes(num_kv_heads: int, head_dim: int) -> int:
    """Bytes of one token row of an int8 pool (PKV_I8 in include/pkv.h)."""
    return num_kv_heads * head_dim + (4 * num_kv_heads + 15) // 16 * 16


class Pool:
    """K and V block pools ``[num_blocks, num_layers, block_size, num_kv_heads,
    head_dim]`` on one CUDA device, as the library's pool descriptor.  An int8
    pool is a pair of uint8 tensors ``[num_blocks, num_layers, block_size, R]``
    (R = :func:`int8_row_bytes`) with ``num_kv_heads`` and ``head_dim`` given."""

    def __init__(self, k_cache: torch.Tensor, v_cache: torch.Tensor,
                 num_kv_heads: Optional[int] = None, head_dim: Optional[int] = None):
        if k_cache.shape != v_cache.shape or k_cache.dtype != v_cache.dtype:
            raise ValueError("k_cache and v_cache must have the same shape and dtype")
        if not k_cache.is_contiguous() or not v_cache.is_contiguous():
            raise ValueError("pools must be contiguous tensors")
        if k_cache.dtype not in _DTYPE:
            raise ValueError(f"unsupported pool dtype {k_cache.dtype}")
        if k_cache.dtype == torch.uint8:
            if k_cache.dim() != 4 or num_kv_heads is None or head_dim is None:
                raise ValueError("int8 pools are [N, L, bs, R] uint8 tensors with "
                                 "num_kv_heads and head_dim given")
            if k_cache.shape[3] != int8_row_bytes(num_kv_heads, head_dim):
                raise ValueError("int8 pool rows do not match num_kv_heads and head_dim")
            N, L, bs = k_cache.shape[:3]
            H, D = num_kv_heads, head_dim
        else:
            if k_cache.dim() != 5:
                raise ValueError("pools must be contiguous [N, L, bs, Hkv, D] tensors")
            N, L, bs, H, D = k_cache.shape
        self.k_cache, self.v_cache = k_cache, v_cache
        self.struct = _PoolStruct(k_cache.data_ptr(), v_cache.data_ptr(), N, L, bs, H, D,
                                  _DTYPE[k_cache.dtype])
        self.device = k_cache.device
        self.num_blocks, self.num_layers, self.block_size = N, L, bs
        self.num_kv_heads, self.head_dim = H, D
        self.dtype = k_cache.dtype

    @property
    def ref(self):
        return ctypes.byref(self.struct)


class _NoSwitch:
    def __enter__(self):
        return self

    def __exit__(self, *exc):
        return False


_NO_SWITCH = _NoSwitch()


def _dev(pool: Pool):
    """Make the pool's device current for the call (no-op when it already is)."""
    idx = pool.device.index
    if idx is None or idx == torch.cuda.current_device():
        return _NO_SWITCH
    return torch.cuda.device(pool.device)


def build_slot_mapping(pool: Pool, block_tables: torch.Tensor, offsets: Optional[torch.Tensor],
                       token_seq: torch.Tensor, token_pos: torch.Tensor,
                       slot_mapping: torch.Tensor) -> torch.Tensor:
    """Fill ``slot_mapping`` (int64 [T]) from (sequence, position) pairs."""
    lib = load()
    B = block_tables.shape[0]
    with _dev(pool):
        st = lib.pkv_build_slot_mapping(pool.ref, _ptr(block_tables), block_tables.shape[1],
                                        _ptr(offsets), B, _ptr(token_seq), _ptr(token_pos),
                                        token_seq.numel(), _ptr(slot_mapping),
                                        _stream(pool.device))
    _check(st, "pkv_build_slot_mapping")
    return slot_mapping


def write_slots(pool: Pool, layer: int, k_new: torch.Tensor, v_new: torch.Tensor,
                slot_mapping: torch.Tensor) -> None:
    """Scatter ``k_new``/``v_new`` ([T, Hkv, D]) into the pools at the slots."""
    lib = load()
    with _dev(pool):
        st = lib.pkv_write_slots(pool.ref, layer, _ptr(k_new), _ptr(v_new), _ptr(slot_mapping),
                                 slot_mapping.numel(), _stream(pool.device))
    _check(st, "pkv_write_slots")


def append_tokens(pool: Pool, layer: int, block_tables: torch.Tensor,
                  offsets: Optional[torch.Tensor], token_seq: torch.Tensor,
                  token_pos: torch.Tensor, k_new: torch.Tensor, v_new: torch.Tensor,
                  slot_mapping: Optional[torch.Tensor] = None) -> None:
    """Slot mapping and scatter in one call: rows of ``k_new``/``v_new``
    ([T, Hkv, D]) go to the slots of (token_seq, token_pos); the slots are
    also written to ``slot_mapping`` (int64 [T]) when given."""
    lib = load()
    with _dev(pool):
        st = lib.pkv_append_tokens(pool.ref, layer, _ptr(block_tables), block_tables.shape[1],
                                   _ptr(offsets), block_tables.shape[0], _ptr(token_seq),
                                   _ptr(token_pos), token_seq.numel(), _ptr(k_new), _ptr(v_new),
                                   _ptr(slot_mapping), _stream(pool.device))
    _check(st, "pkv_append_tokens")


def gather(pool: Pool, layer: int, block_tables: torch.Tensor, seq_lens: torch.Tensor,
           offsets: Optional[torch.Tensor], cu_seqlens: torch.Tensor, k_out: torch.Tensor,
           v_out: torch.Tensor) -> None:
    """Gather every sequence to packed contiguous ``k_out``/``v_out``."""
    lib = load()
    with _dev(pool):
        st = lib.pkv_gather(pool.ref, layer, _ptr(block_tables), block_tables.shape[1],
                            _ptr(seq_lens), _ptr(offsets), seq_lens.numel(), _ptr(cu_seqlens),
                            k_out.shape[0], _ptr(k_out), _ptr(v_out), _stream(pool.device))
    _check(st, "pkv_gather")


def decode_workspace_size(batch: int, num_q_heads: int, head_dim: int,
                          device: Optional[torch.device] = None) -> int:
    lib = load()
    with torch.cuda.device(device if device is not None else torch.cuda.current_device()):
        n = lib.pkv_decode_workspace_size(batch, num_q_heads, head_dim)
    if n == 0:
        raise PkvError(1, "pkv_decode_workspace_size", "bad shape or no CUDA device")
    return n


def decode_attention(pool: Pool, layer: int, q: torch.Tensor, scale: float,
                     block_tables: torch.Tensor, seq_lens: torch.Tensor,
                     offsets: Optional[torch.Tensor], out: torch.Tensor,
                     workspace: torch.Tensor) -> None:
    """Paged decode attention of ``q`` [B, Hq, D] into ``out`` [B, Hq, D]."""
    lib = load()
    with _dev(pool):
        st = lib.pkv_decode_attention(pool.ref, layer, _ptr(q), q.shape[1], float(scale),
                                      _ptr(block_tables), block_tables.shape[1], _ptr(seq_lens),
                                      _ptr(offsets), seq_lens.numel(), _ptr(out),
                                      _ptr(workspace), workspace.numel() * workspace.element_size(),
                                      _stream(pool.device))
    _check(st, "pkv_decode_attention")


def decode_shared_prefix_workspace_size(pool: Pool, batch: int, num_q_heads: int,
                                        num_prefix_blocks: int) -> int:
    with _dev(pool):
        return int(load().pkv_decode_shared_prefix_workspace_size(pool.ref, batch, num_q_heads,
                                                                  num_prefix_blocks))


def decode_attention_shared_prefix(pool: Pool, layer: int, q: torch.Tensor, scale: float,
                                   block_tables: torch.Tensor, seq_lens: torch.Tensor,
                                   offsets: Optional[torch.Tensor], num_prefix_blocks: int,
                                   out: torch.Tensor, workspace: torch.Tensor) -> None:
    """Paged decode attention of ``q`` [B, Hq, D] whose sequences share their
    first ``num_prefix_blocks`` table entries: the prefix is read once."""
    lib = load()
    with _dev(pool):
        st = lib.pkv_decode_attention_shared_prefix(
            pool.ref, layer, _ptr(q), q.shape[1], float(scale), _ptr(block_tables),
            block_tables.shape[1], _ptr(seq_lens), _ptr(offsets), seq_lens.numel(),
            int(num_prefix_blocks), _ptr(out), _ptr(workspace),
            workspace.numel() * workspace.element_size(), _stream(pool.device))
    _check(st, "pkv_decode_attention_shared_prefix")


def decode_step(pool: Pool, layer: int, q: torch.Tensor, scale: float,
                block_tables: torch.Tensor, seq_lens: torch.Tensor,
                offsets: Optional[torch.Tensor], k_new: torch.Tensor, v_new: torch.Tensor,
                out: torch.Tensor, workspace: torch.Tensor) -> None:
    """One decode step: store each sequence's new K/V row (``k_new``,
    ``v_new`` [B, Hkv, D]) at its last position, then paged decode attention
    of ``q`` [B, Hq, D] into ``out``, in one pass over the pool."""
    lib = load()
    with _dev(pool):
        st = lib.pkv_decode_step(pool.ref, layer, _ptr(q), q.shape[1], float(scale),
                                 _ptr(block_tables), block_tables.shape[1], _ptr(seq_lens),
                                 _ptr(offsets), seq_lens.numel(), _ptr(k_new), _ptr(v_new),
                                 _ptr(out), _ptr(workspace),
                                 workspace.numel() * workspace.element_size(),
                                 _stream(pool.device))
    _check(st, "pkv_decode_step")


def decode_attention_static(pool: Pool, layer: int, q: torch.Tensor, scale: float,
                            block_tables: torch.Tensor, seq_lens: torch.Tensor,
                            offsets: Optional[torch.Tensor], out: torch.Tensor) -> None:
    """Paged decode attention without a workspace argument: the library keeps
    the scratch in its own fixed device array (for callers that cannot
    allocate device memory where they run; shapes beyond the array's size
    raise PKV_ERR_WORKSPACE, and calls that overlap on the GPU race)."""
    lib = load()
    with _dev(pool):
        st = lib.pkv_decode_attention_static(pool.ref, layer, _ptr(q), q.shape[1], float(scale),
                                             _ptr(block_tables), block_tables.shape[1],
                                             _ptr(seq_lens), _ptr(offsets), seq_lens.numel(),
                                             _ptr(out), _stream(pool.device))
    _check(st, "pkv_decode_attention_static")


def copy_blocks(pool: Pool, layer: int, src_blocks: torch.Tensor,
                dst_blocks: torch.Tensor) -> None:
    """Block dst[i] <- block src[i] (K and V), one layer or every layer (-1)."""
    lib = load()
    with _dev(pool):
        st = lib.pkv_copy_blocks(pool.ref, layer, _ptr(src_blocks), _ptr(dst_blocks),
                                 src_blocks.numel(), _stream(pool.device))
    _check(st, "pkv_copy_blocks")


def swap_out(pool: Pool, layer: int, blocks: torch.Tensor, host_k: torch.Tensor,
             host_v: torch.Tensor) -> None:
    """Listed blocks -> page-locked host tensors [n, layers, bs, Hkv, D]."""
    lib = load()
    nbytes = min(host_k.numel(), host_v.numel()) * host_k.element_size()
    with _dev(pool):
        st = lib.pkv_swap_out(pool.ref, layer, _ptr(blocks), blocks.numel(), _ptr(host_k),
                              _ptr(host_v), nbytes, _stream(pool.device))
    _check(st, "pkv_swap_out")


def swap_in(pool: Pool, layer: int, blocks: torch.Tensor, host_k: torch.Tensor,
            host_v: torch.Tensor) -> None:
    """Page-locked host tensors [n, layers, bs, Hkv, D] -> listed blocks."""
    lib = load()
    nbytes = min(host_k.numel(), host_v.numel()) * host_k.element_size()
    with _dev(pool):
        st = lib.pkv_swap_in(pool.ref, layer, _ptr(blocks), blocks.numel(), _ptr(host_k),
                             _ptr(host_v), nbytes, _stream(pool.device))
    _check(st, "pkv_swap_in")


def prefill_attention(pool: Pool, layer: int, q: torch.Tensor, scale: float,
                      block_tables: torch.Tensor, seq_lens: torch.Tensor,
                      offsets: Optional[torch.Tensor], cu_q: torch.Tensor, max_q_len: int,
                      out: torch.Tensor) -> None:
    """Causal prefill attention of q [T, Hq, D] (the last cu_q[b+1]-cu_q[b]
    tokens of each sequence) over the paged cache into out [T, Hq, D]."""
    lib = load()
    with _dev(pool):
        st = lib.pkv_prefill_attention(pool.ref, layer, _ptr(q), q.shape[1], float(scale),
                                       _ptr(block_tables), block_tables.shape[1], _ptr(seq_lens),
                                       _ptr(offsets), _ptr(cu_q), seq_lens.numel(), q.shape[0],
                                       max_q_len, _ptr(out), _stream(pool.device))
    _check(st, "pkv_prefill_attention")


def set_decode_ctas(n: int) -> None:
    _check(load().pkv_set_decode_ctas(n), "pkv_set_decode_ctas")


def set_decode_events(start: Optional[torch.cuda.Event], stop: Optional[torch.cuda.Event]) -> None:
    """Have later decode calls record ``start``/``stop`` around the partial
    pass kernel (``None`` stops it).  The events must have been recorded once
    so that torch has created them."""
    a = start.cuda_event if start is not None else None
    b = stop.cuda_event if stop is not None else None
    _check(load().pkv_set_decode_events(a, b), "pkv_set_decode_events")


def set_validate(on: bool) -> None:
    _check(load().pkv_set_validate(1 if on else 0), "pkv_set_validate")


def set_wait_limit_ns(ns: int) -> None:
    """Bound of every device-side wait in nanoseconds (0 = the default)."""
    _check(load().pkv_set_wait_limit_ns(int(ns)), "pkv_set_wait_limit_ns")


def get_wait_limit_ns() -> int:
    return int(load().pkv_get_wait_limit_ns())


def set_debug_skip_fill(mode: int) -> None:
    """Test hook: with 1 the first CTA, with 2 every CTA, of each decode /
    prefill launch leaves its first stage unfilled, so a wait there can only
    give up; 0 turns it off."""
    _check(load().pkv_set_debug_skip_fill(int(mode)), "pkv_set_debug_skip_fill")


def get_validate() -> bool:
    return bool(load().pkv_get_validate())


def device_error(clear: bool = True) -> str:
    """Status name of the sticky device error word (synchronises the device)."""
    s = ctypes.c_int32(0)
    _check(load().pkv_device_error(ctypes.byref(s), 1 if clear else 0), "pkv_device_error")
    return _STATUS[s.value]


def status_string(status: int) -> str:
    return load().pkv_status_string(status).decode()


def version() -> int:
    return load().pkv_version()


class Allocator:
    """Host block allocator of the library (the allocator section of
    include/pkv.h): FIFO free deque, reference counts, per-sequence block
    tables with a first-block offset, copy-on-write on shared blocks."""

    def __init__(self, num_blocks: int, block_size: int,
                 free_order: Optional[Sequence[int]] = None):
        lib = load()
        h = ctypes.c_void_p()
        order = None
        if free_order is not None:
            order = np.ascontiguousarray(np.asarray(free_order, dtype=np.int32))
        _check(lib.pkv_alloc_create(num_blocks, block_size,
                                    None if order is None else order.ctypes.data,
                                    ctypes.byref(h)), "pkv_alloc_create")
        self._h = h
        self._lib = lib
        self.num_blocks, self.block_size = num_blocks, block_size

    def close(self) -> None:
        if self._h:
            self._lib.pkv_alloc_destroy(self._h)
            self._h = ctypes.c_void_p()

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def num_free(self) -> int:
        return self._lib.pkv_alloc_num_free(self._h)

    def ref_count(self, block: int) -> int:
        return self._lib.pkv_alloc_ref_count(self._h, block)

    def allocate_blocks(self, n: int) -> List[int]:
        out = np.empty(max(n, 1), dtype=np.int32)
        _check(self._lib.pkv_alloc_blocks(self._h, n, out.ctypes.data), "pkv_alloc_blocks")
        return out[:n].tolist()

    def inc_ref(self, block: int) -> None:
        _check(self._lib.pkv_alloc_inc_ref(self._h, block), "pkv_alloc_inc_ref")

    def dec_ref(self, block: int) -> None:
        _check(self._lib.pkv_alloc_dec_ref(self._h, block), "pkv_alloc_dec_ref")

    def seq_new(self, sid: int, offset: int = 0) -> None:
        _check(self._lib.pkv_seq_new(self._h, sid, offset), "pkv_seq_new")

    def seq_share(self, sid: int, blocks: Sequence[int], num_tokens: int) -> None:
        arr = np.ascontiguousarray(np.asarray(blocks, dtype=np.int32))
        _check(self._lib.pkv_seq_share(self._h, sid, arr.ctypes.data if len(arr) else None,
                                       len(arr), num_tokens), "pkv_seq_share")

    def seq_append(self, sid: int, num_tokens: int) -> Tuple[np.ndarray, List[Tuple[int, int]]]:
        slots = np.empty(max(num_tokens, 1), dtype=np.int64)
        src, dst, n = ctypes.c_int32(), ctypes.c_int32(), ctypes.c_int32()
        _check(self._lib.pkv_seq_append(self._h, sid, num_tokens, slots.ctypes.data,
                                        ctypes.byref(src), ctypes.byref(dst), ctypes.byref(n)),
               "pkv_seq_append")
        return slots[:num_tokens], ([(src.value, dst.value)] if n.value else [])

    def seq_append_batch(self, sids: Sequence[int], counts: Optional[Sequence[int]] = None):
        ids = np.ascontiguousarray(np.asarray(sids, dtype=np.int64))
        n = len(ids)
        cnt = None if counts is None else np.ascontiguousarray(np.asarray(counts, dtype=np.int64))
        total = n if cnt is None else int(cnt.sum())
        slots = np.empty(max(total, 1), dtype=np.int64)
        src = np.empty(max(n, 1), dtype=np.int32)
        dst = np.empty(max(n, 1), dtype=np.int32)
        nc = ctypes.c_int32()
        _check(self._lib.pkv_seq_append_batch(self._h, ids.ctypes.data if n else None, n,
                                              None if cnt is None else cnt.ctypes.data,
                                              slots.ctypes.data, src.ctypes.data, dst.ctypes.data,
                                              ctypes.byref(nc)), "pkv_seq_append_batch")
        return slots[:total], list(zip(src[:nc.value].tolist(), dst[:nc.value].tolist()))

    def seq_fork(self, src: int, dst: int) -> None:
        _check(self._lib.pkv_seq_fork(self._h, src, dst), "pkv_seq_fork")

    def seq_free(self, sid: int) -> None:
        _check(self._lib.pkv_seq_free(self._h, sid), "pkv_seq_free")

    def seq_info(self, sid: int) -> Tuple[int, int, int]:
        n, off, nb = ctypes.c_int64(), ctypes.c_int32(), ctypes.c_int32()
        _check(self._lib.pkv_seq_info(self._h, sid, ctypes.byref(n), ctypes.byref(off),
                                      ctypes.byref(nb)), "pkv_seq_info")
        return n.value, off.value, nb.value

    def seq_tables(self, sids: Sequence[int], max_blocks: int):
        ids = np.ascontiguousarray(np.asarray(sids, dtype=np.int64))
        B = len(ids)
        tables = np.empty((max(B, 1), max_blocks), dtype=np.int32)
        lens = np.empty(max(B, 1), dtype=np.int32)
        offs = np.empty(max(B, 1), dtype=np.int32)
        _check(self._lib.pkv_seq_tables(self._h, ids.ctypes.data if B else None, B, max_blocks,
                                        tables.ctypes.data, lens.ctypes.data, offs.ctypes.data),
               "pkv_seq_tables")
        return tables[:B], lens[:B], offs[:B]

    def stats(self) -> Tuple[int, int, float]:
        a, u, f = ctypes.c_int64(), ctypes.c_int64(), ctypes.c_double()
        _check(self._lib.pkv_alloc_stats(self._h, ctypes.byref(a), ctypes.byref(u),
                                         ctypes.byref(f)), "pkv_alloc_stats")
        return a.value, u.value, f.value
