"""Oracle for the quantised (int8) KV pool: a plain, slow CPU restatement.

TEST INFRASTRUCTURE ONLY, like the rest of ``oracle/``: only ``tests/``,
``__graft_entry__.smoke()`` and the CPU-baseline leg of ``bench.py`` may
import it.  It imports nothing from the CUDA library.

What the pages fix.  "mini-runtime ch.12 Paged KV Cache", §6 Evolution, names
quantised KV (int8 / int4) as the step that follows paged KV: the same block
pool holding fewer bytes per token.  The pages give no scheme.  The readings
taken here are the plainest ones that keep every other step unchanged:

* Granularity: one scale per (token, kv head), so that a token row is written
  once by the scatter and never rewritten, and a block copy or swap still
  moves whole rows.
* Symmetric absmax quantisation in fp32: with ``x`` the head's D values
  (bf16, widened exactly to fp32), ``scale = absmax(x) / 127`` and
  ``code = round(x / scale)``, both divisions IEEE fp32 round-to-nearest and
  the rounding to integer half-to-even, codes clamped to [-127, 127].  A row
  of zeros has scale 0 and codes 0.  Dequantised value: ``code * scale``.
* Row format: a pool is bytes ``[num_blocks, num_layers, block_size, R]``
  with ``R = Hkv * D + pad16(4 * Hkv)``; a token row holds the Hkv * D codes
  (head-major, each stored offset binary as the byte ``code + 128``, so the
  kernels turn a byte into a number without a sign fix-up) followed by the
  Hkv scales (fp32, little-endian) and padding up to a multiple of 16 bytes.  The scatter leaves the padding
  bytes untouched; nothing reads them.
* Attention over an int8 pool is attention over the dequantised K and V, in
  fp64, with the bf16 query (the decode definition of ``oracle.oracle``).

Parity pins: ``tests/test_quant_pins.py`` checks every function here against
closed forms (exact rational arithmetic for the fp32 divisions, worked
half-way cases, exactness on representable inputs) and plants mistakes.
"""

from __future__ import annotations

from typing import Iterable, Sequence

import numpy as np

from .oracle import attention_fp64, gather_loop, widen

__all__ = [
    "QMAX", "row_bytes", "code_bytes", "quantize_head", "quantize_rows", "write_slots_i8",
    "unpack_rows", "dequantize_rows", "decode_attention_i8", "decode_attention_i8_pairs",
]

QMAX = 127


def row_bytes(num_kv_heads: int, head_dim: int) -> int:
    """Bytes of one token row of an int8 pool: codes, scales, padding to 16."""
    scale_bytes = 4 * num_kv_heads
    return num_kv_heads * head_dim + (scale_bytes + 15) // 16 * 16


def _bf16_to_f32(bits: np.ndarray) -> np.ndarray:
    """bf16 bit patterns as the fp32 numbers they encode (exact)."""
    return (np.asarray(bits).astype(np.uint32) << 16).view(np.float32)


def quantize_head(x: np.ndarray):
    """Codes and scale of one head's values ``x`` (fp32 ``[D]``).

    absmax in fp32, ``scale = absmax / 127`` as one fp32 division, then each
    code is the fp32 quotient ``x / scale`` rounded half-to-even and clamped.
    """
    x = np.asarray(x, dtype=np.float32)
    absmax = np.float32(np.max(np.abs(x))) if x.size else np.float32(0)
    scale = np.float32(absmax) / np.float32(QMAX)
    if scale == 0:
        return np.zeros(x.shape, dtype=np.int8), np.float32(0)
    q = np.rint(x / scale)  # float32 / float32: one IEEE division per element
    return np.clip(q, -QMAX, QMAX).astype(np.int8), np.float32(scale)


def quantize_rows(x_bits: np.ndarray):
    """``[n, Hkv, D]`` bf16 bits -> codes int8 ``[n, Hkv, D]``, scales fp32
    ``[n, Hkv]``, one (token, head) at a time."""
    x = _bf16_to_f32(x_bits)
    n, H, D = x.shape
    codes = np.zeros((n, H, D), dtype=np.int8)
    scales = np.zeros((n, H), dtype=np.float32)
    for t in range(n):
        for g in range(H):
            codes[t, g], scales[t, g] = quantize_head(x[t, g])
    return codes, scales


def code_bytes(codes: np.ndarray) -> np.ndarray:
    """The stored byte of each code: offset binary, ``code + 128`` (codes in
    [-127, 127] become bytes 1..255)."""
    return (np.asarray(codes).astype(np.int16) + 128).astype(np.uint8)


def _store_row(row: np.ndarray, codes: np.ndarray, scales: np.ndarray) -> None:
    """Write one token's codes ``[Hkv, D]`` and scales ``[Hkv]`` into its byte
    row, leaving the padding bytes as they were."""
    H, D = codes.shape
    row[:H * D] = code_bytes(codes).reshape(-1)
    row[H * D:H * D + 4 * H] = np.asarray(scales, dtype="<f4").view(np.uint8)


def write_slots_i8(k_cache: np.ndarray, v_cache: np.ndarray, layer: int,
                   k_new: np.ndarray, v_new: np.ndarray, slot_mapping: np.ndarray,
                   num_kv_heads: int, head_dim: int) -> None:
    """The slot_mapping scatter ("vLLM PagedAttention source notes" §2.2) into
    int8 pools: each new bf16 row is quantised, then stored at its slot; ``-1``
    entries are padding and are skipped; any other bad slot is rejected."""
    N, L, bs, R = k_cache.shape
    if R != row_bytes(num_kv_heads, head_dim):
        raise ValueError("pool rows do not match the int8 row format")
    seen = set()
    for t in range(len(slot_mapping)):
        s = int(slot_mapping[t])
        if s == -1:
            continue
        if s < 0 or s >= N * bs:
            raise IndexError(f"slot {s} outside the pool")
        if s in seen:
            raise ValueError(f"slot {s} written twice")
        seen.add(s)
        blk, j = divmod(s, bs)
        for pool, new in ((k_cache, k_new), (v_cache, v_new)):
            codes, scales = quantize_rows(np.asarray(new[t:t + 1]))
            _store_row(pool[blk, layer, j], codes[0], scales[0])


def unpack_rows(rows: np.ndarray, num_kv_heads: int, head_dim: int):
    """Byte rows ``[n, R]`` -> codes int8 ``[n, Hkv, D]``, scales fp32 ``[n, Hkv]``."""
    rows = np.ascontiguousarray(rows, dtype=np.uint8)
    n = rows.shape[0]
    H, D = num_kv_heads, head_dim
    codes = (rows[:, :H * D].astype(np.int16) - 128).astype(np.int8).reshape(n, H, D)
    scales = rows[:, H * D:H * D + 4 * H].copy().view("<f4").reshape(n, H).astype(np.float32)
    return codes, scales


def dequantize_rows(rows: np.ndarray, num_kv_heads: int, head_dim: int) -> np.ndarray:
    """Byte rows ``[n, R]`` -> fp64 ``[n, Hkv, D]``: code * scale, exactly."""
    codes, scales = unpack_rows(rows, num_kv_heads, head_dim)
    return codes.astype(np.float64) * scales.astype(np.float64)[:, :, None]


def decode_attention_i8(k_cache: np.ndarray, v_cache: np.ndarray, layer: int,
                        q: np.ndarray, block_tables: np.ndarray, seq_lens: np.ndarray,
                        offsets: np.ndarray, scale: float) -> np.ndarray:
    """Decode attention over int8 pools, ``[B, Hq, D]`` fp64: gather each
    sequence's byte rows through its block table (first-block offset as in
    ch.12 §2.2), dequantise, then standard attention per query head with the
    GQA head map ``h -> h // (Hq // Hkv)``."""
    B, Hq, D = q.shape
    H = _heads(k_cache.shape[3], D)
    group = Hq // H
    qd = widen(q)
    out = np.zeros((B, Hq, D), dtype=np.float64)
    for b in range(B):
        kb = dequantize_rows(gather_loop(k_cache, layer, block_tables[b], int(seq_lens[b]),
                                         int(offsets[b])), H, D)
        vb = dequantize_rows(gather_loop(v_cache, layer, block_tables[b], int(seq_lens[b]),
                                         int(offsets[b])), H, D)
        for h in range(Hq):
            g = h // group
            out[b, h] = attention_fp64(qd[b, h], kb[:, g, :], vb[:, g, :], scale)
    return out


def decode_attention_i8_pairs(k_cache: np.ndarray, v_cache: np.ndarray, layer: int,
                              q: np.ndarray, block_tables: np.ndarray, seq_lens: np.ndarray,
                              offsets: np.ndarray, scale: float, pairs: Iterable) -> dict:
    """:func:`decode_attention_i8` for selected ``(b, h)`` pairs only."""
    Hq, D = q.shape[1], q.shape[2]
    H = _heads(k_cache.shape[3], D)
    group = Hq // H
    out = {}
    for b, h in pairs:
        g = h // group
        kb = dequantize_rows(gather_loop(k_cache, layer, block_tables[b], int(seq_lens[b]),
                                         int(offsets[b])), H, D)
        vb = dequantize_rows(gather_loop(v_cache, layer, block_tables[b], int(seq_lens[b]),
                                         int(offsets[b])), H, D)
        out[(b, h)] = attention_fp64(widen(q[b, h]), kb[:, g, :], vb[:, g, :], scale)
    return out


def _heads(R: int, D: int) -> int:
    """Kv heads of an int8 row of R bytes and head size D."""
    for H in range(1, R // D + 1):
        if row_bytes(H, D) == R:
            return H
    raise ValueError(f"{R}-byte rows are not int8 rows of head size {D}")
