"""Pins for the int8 KV oracle (``oracle.quant``): what the arithmetic fixes,
independent of the oracle's own code.

* Quantisation decisions are recomputed with exact rational arithmetic
  (``fractions.Fraction``) and a round-to-nearest-even fp32 rounding written
  here, so the fp32 divisions of the oracle are checked against their
  definition, on every bf16 value of a range.
* Worked half-way cases, the all-zero row, per-head independence and the
  dequantisation error bound are closed forms.
* On rows whose values are already code * scale (integer multiples of a power
  of two with absmax 127 * scale) quantisation is exact, so decode over the
  int8 pool must equal the pinned bf16 decode oracle.

Each check takes the implementation as arguments; ``test_quant_pins_catch_
planted_mistakes`` runs the same checks against broken copies.
"""

import struct
from fractions import Fraction

import numpy as np
import pytest

import oracle
from oracle import quant as Q


# ---------------------------------------------------------------------------
# exact fp32 model
# ---------------------------------------------------------------------------

def f32_round(r: Fraction) -> Fraction:
    """Nearest fp32 number to the rational r (ties to even), subnormals
    included; r must be inside the fp32 range."""
    if r == 0:
        return Fraction(0)
    sign = -1 if r < 0 else 1
    a = abs(r)
    e = a.numerator.bit_length() - a.denominator.bit_length()
    while Fraction(2) ** e > a:
        e -= 1
    while Fraction(2) ** (e + 1) <= a:
        e += 1
    e = max(e, -126)
    ulp = Fraction(2) ** (e - 23)
    return sign * round(a / ulp) * ulp   # round() on a Fraction ties to even


def bf16(bits) -> np.ndarray:
    return (np.asarray(bits, dtype=np.uint32) << 16).view(np.float32)


def f32_to_bf16_bits(x) -> np.ndarray:
    """fp32 values that are exactly bf16 -> their bit patterns."""
    b = np.asarray(x, dtype=np.float32).view(np.uint32)
    assert np.all(b & 0xFFFF == 0), "value is not a bf16 number"
    return (b >> 16).astype(np.uint16)


def exact_codes(x: np.ndarray):
    """The reading's quantisation, decided in exact arithmetic: fp32 absmax,
    fp32 quotient absmax/127, fp32 quotients x/scale, ties-to-even rounding."""
    xs = [Fraction(float(v)) for v in x]
    absmax = max(abs(v) for v in xs)
    scale = f32_round(absmax / 127)
    if scale == 0:
        return [0] * len(xs), scale
    return [max(-127, min(127, round(f32_round(v / scale)))) for v in xs], scale


# ---------------------------------------------------------------------------
# reusable checks
# ---------------------------------------------------------------------------

def check_half_way_cases(quantize_head):
    # absmax 127 gives scale exactly 1, so every quotient is x itself
    x = np.array([127, 2.5, 3.5, -2.5, 0.5, 1.5, -0.5, -1.5, 126.5, 0], np.float32)
    codes, scale = quantize_head(x)
    assert float(scale) == 1.0
    assert codes.tolist() == [127, 2, 4, -2, 0, 2, 0, -2, 126, 0]
    codes, scale = quantize_head(-x)
    assert codes.tolist() == [-127, -2, -4, 2, 0, -2, 0, 2, -126, 0]
    codes, scale = quantize_head(np.zeros(8, np.float32))
    assert float(scale) == 0.0 and not np.any(codes)
    codes, scale = quantize_head(np.array([0, 0, -3.0, 0], np.float32))
    assert codes.tolist() == [0, 0, -127, 0]


@pytest.mark.parametrize("absmax_bits", [0x3F80, 0x3F8F, 0x3F90])
def test_fp32_decisions_every_bf16(absmax_bits):
    check_fp32_decisions(Q.quantize_head, absmax_bits)


def check_fp32_decisions(quantize_head, absmax_bits=0x3F90):
    """Every bf16 x with 2^-31 <= |x| <= absmax, quantised together with the
    absmax itself, against the exact model.  absmax 1.125 is a value where
    exact scaling x*127/absmax and multiplying by a reciprocal both round some
    codes differently from two fp32 divisions."""
    am = bf16([absmax_bits])[0]
    pos = bf16(np.arange(0x3000, 0x4400))
    pos = pos[pos <= am]
    x = np.concatenate([[am], pos, -pos]).astype(np.float32)
    codes, scale = quantize_head(x)
    want, want_scale = exact_codes(x)
    assert Fraction(float(scale)) == want_scale
    assert codes.astype(int).tolist() == want


def check_dequant_bound(quantize_rows):
    rng = np.random.default_rng(5)
    x = (rng.standard_normal((40, 4, 64)) * rng.uniform(0.01, 50, (40, 4, 1))).astype(np.float32)
    xb = f32_to_bf16_bits(bf16(x.view(np.uint32) >> 16))
    xf = bf16(xb)
    codes, scales = quantize_rows(xb)
    assert codes.dtype == np.int8 and scales.dtype == np.float32
    assert np.all(np.abs(codes.astype(int)) <= 127)
    # absmax maps to +-127 in each (token, head)
    assert np.all(np.abs(codes).max(axis=2) == 127)
    s = scales.astype(np.float64)[:, :, None]
    err = np.abs(codes * s - xf.astype(np.float64))
    assert np.all(err <= 0.5 * s + np.abs(xf) * 2.0 ** -22)


def check_per_head_scale(quantize_rows):
    x = np.zeros((1, 3, 16), np.float32)
    x[0, 0, 3] = 0.25
    x[0, 1, 7] = -64.0
    x[0, 2, :] = 1.0
    codes, scales = quantize_rows(f32_to_bf16_bits(x))
    assert scales[0].tolist() == [float(np.float32(0.25) / np.float32(127)),
                                  float(np.float32(64.0) / np.float32(127)),
                                  float(np.float32(1.0) / np.float32(127))]
    assert codes[0, 0, 3] == 127 and codes[0, 1, 7] == -127
    assert np.all(codes[0, 2] == 127)


def check_row_format(write_slots_i8, unpack_rows):
    H, D, bs = 3, 32, 4
    R = Q.row_bytes(H, D)
    assert R == 96 + 16   # 12 bytes of scales, padded to 16
    assert Q.row_bytes(8, 128) == 1056 and Q.row_bytes(1, 64) == 80
    rng = np.random.default_rng(9)
    k = rng.integers(0, 256, (6, 2, bs, R), dtype=np.uint8)
    v = rng.integers(0, 256, (6, 2, bs, R), dtype=np.uint8)
    k0, v0 = k.copy(), v.copy()
    xk = np.zeros((3, H, D), np.float32)
    xv = np.zeros((3, H, D), np.float32)
    for t in range(3):
        for g in range(H):
            xk[t, g, (t + g) % D] = 2.0 ** (g - t)          # absmax 2^(g-t), code 127 there
            xk[t, g, (t + g + 1) % D] = -(2.0 ** (g - t - 1))
            xv[t, g, g] = -(g + 1.0)
    slots = np.array([5, -1, 13], np.int64)                # block 1 row 1, pad, block 3 row 1
    write_slots_i8(k, v, 1, f32_to_bf16_bits(xk), f32_to_bf16_bits(xv), slots, H, D)
    changed = [(1, 1, 1), (3, 1, 1)]
    for (blk, layer, row), t in zip(changed, (0, 2)):
        rk, rv = k[blk, layer, row], v[blk, layer, row]
        for g in range(H):
            sk = struct.unpack("<f", rk[H * D + 4 * g:H * D + 4 * g + 4].tobytes())[0]
            assert sk == float(np.float32(2.0 ** (g - t)) / np.float32(127))
            ck = rk[g * D:(g + 1) * D].astype(np.int16) - 128       # offset-binary bytes
            assert ck[(t + g) % D] == 127
            # -absmax/2: the fp32 quotient is exactly -63.5, which ties to -64
            assert ck[(t + g + 1) % D] == -64
            assert np.count_nonzero(ck) == 2
            sv = struct.unpack("<f", rv[H * D + 4 * g:H * D + 4 * g + 4].tobytes())[0]
            assert sv == float(np.float32(g + 1.0) / np.float32(127))
            cv = rv[g * D:(g + 1) * D].astype(np.int16) - 128
            assert cv[g] == -127 and np.count_nonzero(cv) == 1
        # padding untouched
        assert np.array_equal(rk[H * D + 4 * H:], k0[blk, layer, row, H * D + 4 * H:])
        assert np.array_equal(rv[H * D + 4 * H:], v0[blk, layer, row, H * D + 4 * H:])
    mask = np.ones(k.shape[:3], bool)
    for c in changed:
        mask[c] = False
    assert np.array_equal(k[mask], k0[mask]) and np.array_equal(v[mask], v0[mask])
    codes, scales = unpack_rows(k[1, 1, 1:2], H, D)
    assert codes.shape == (1, H, D) and scales.shape == (1, H)
    assert scales[0, 2] == np.float32(4.0) / np.float32(127)
    # the byte of code c is c + 128: 0 -> 128, 127 -> 255, -64 -> 64, -127 -> 1
    rk = k[1, 1, 1]
    assert rk[(0 + 0) % D] == 255 and rk[(0 + 1) % D] == 64 and rk[5] == 128
    assert v[1, 1, 1, 0] == 1


def check_dequant_formula(dequantize_rows):
    H, D = 2, 16
    R = Q.row_bytes(H, D)
    row = np.zeros((1, R), np.uint8)
    codes = np.arange(-16, 16, dtype=np.int8).reshape(H, D)
    row[0, :H * D] = (codes.reshape(-1).astype(np.int16) + 128).astype(np.uint8)
    row[0, H * D:H * D + 8] = np.frombuffer(struct.pack("<ff", 0.5, -3.0), np.uint8)
    got = dequantize_rows(row, H, D)
    want = np.stack([codes[0] * 0.5, codes[1] * -3.0])[None].astype(np.float64)
    assert np.array_equal(got, want)


def _representable_case(seed, lens, H=2, G=2, D=32, bs=8):
    """bf16 K/V whose heads are integer multiples of a power of two with one
    element of magnitude 127 * 2^e, so quantisation reproduces them exactly."""
    rng = np.random.default_rng(seed)
    B = len(lens)
    offs = rng.integers(0, bs, B)
    need = [-(-(int(o) + L) // bs) for o, L in zip(offs, lens)]
    N = sum(need) + 3
    perm = rng.permutation(N)
    tables = np.full((B, max(need)), -1, np.int32)
    at = 0
    for b, n in enumerate(need):
        tables[b, :n] = perm[at:at + n]
        at += n
    L = 2
    rows = N * L * bs
    def draw():
        c = rng.integers(-127, 128, (rows, H, D)).astype(np.float32)
        c[:, :, 0] = np.where(rng.random((rows, H)) < 0.5, 127.0, -127.0)
        e = rng.integers(-8, 2, (rows, H, 1)).astype(np.float32)
        return (c * np.float32(2.0) ** e).astype(np.float32)
    xk, xv = draw(), draw()
    k16 = f32_to_bf16_bits(xk).reshape(N, L, bs, H, D)
    v16 = f32_to_bf16_bits(xv).reshape(N, L, bs, H, D)
    q = (rng.standard_normal((B, H * G, D)).astype(np.float32).view(np.uint32) >> 16
         ).astype(np.uint16)
    return k16, v16, q, tables, np.asarray(lens, np.int32), offs.astype(np.int32), bs


def check_representable_exact(write_slots_i8, decode_attention_i8):
    k16, v16, q, bt, lens, offs, bs = _representable_case(3, [1, 17, 40])
    N, L, _, H, D = k16.shape
    R = Q.row_bytes(H, D)
    k8 = np.zeros((N, L, bs, R), np.uint8)
    v8 = np.zeros((N, L, bs, R), np.uint8)
    for layer in range(L):
        slots = np.arange(N * bs, dtype=np.int64)
        write_slots_i8(k8, v8, layer, k16[:, layer].reshape(-1, H, D),
                       v16[:, layer].reshape(-1, H, D), slots, H, D)
    scale = D ** -0.5
    want = oracle.decode_attention(k16, v16, 1, q, bt, lens, offs, scale)
    got = decode_attention_i8(k8, v8, 1, q, bt, lens, offs, scale)
    assert np.allclose(got, want, rtol=0, atol=1e-12)


# ---------------------------------------------------------------------------
# the pins
# ---------------------------------------------------------------------------

def test_half_way_cases():
    check_half_way_cases(Q.quantize_head)


def test_dequant_bound():
    check_dequant_bound(Q.quantize_rows)


def test_per_head_scale():
    check_per_head_scale(Q.quantize_rows)


def test_row_format():
    check_row_format(Q.write_slots_i8, Q.unpack_rows)


def test_dequant_formula():
    check_dequant_formula(Q.dequantize_rows)


def test_representable_rows_decode_exactly():
    check_representable_exact(Q.write_slots_i8, Q.decode_attention_i8)


def test_pairs_match_full():
    k16, v16, q, bt, lens, offs, bs = _representable_case(4, [5, 30])
    N, L, _, H, D = k16.shape
    R = Q.row_bytes(H, D)
    rng = np.random.default_rng(1)
    k8 = rng.integers(0, 256, (N, L, bs, R), dtype=np.uint8)
    v8 = rng.integers(0, 256, (N, L, bs, R), dtype=np.uint8)
    # random codes with sane scales
    for p in (k8, v8):
        p[..., H * D:H * D + 4 * H] = rng.uniform(0.01, 0.05, (N, L, bs, H)).astype(
            "<f4").view(np.uint8).reshape(N, L, bs, 4 * H)
    full = Q.decode_attention_i8(k8, v8, 0, q, bt, lens, offs, 0.2)
    pairs = [(0, 0), (1, 3), (1, 2)]
    part = Q.decode_attention_i8_pairs(k8, v8, 0, q, bt, lens, offs, 0.2, pairs)
    for b, h in pairs:
        assert np.array_equal(part[(b, h)], full[b, h])


# ---------------------------------------------------------------------------
# planted mistakes
# ---------------------------------------------------------------------------

def _qh_div128(x):
    x = np.asarray(x, np.float32)
    s = np.float32(np.max(np.abs(x))) / np.float32(128)
    return (np.zeros(x.shape, np.int8), s) if s == 0 else (
        np.clip(np.rint(x / s), -127, 127).astype(np.int8), s)


def _qh_round_away(x):
    c, s = Q.quantize_head(x)
    if s == 0:
        return c, s
    q = np.asarray(x, np.float32) / s
    return np.clip(np.sign(q) * np.floor(np.abs(q) + 0.5), -127, 127).astype(np.int8), s


def _qh_floor(x):
    c, s = Q.quantize_head(x)
    if s == 0:
        return c, s
    return np.clip(np.floor(np.asarray(x, np.float32) / s), -127, 127).astype(np.int8), s


def _qh_reciprocal(x):
    c, s = Q.quantize_head(x)
    if s == 0:
        return c, s
    inv = np.float32(1) / s
    return np.clip(np.rint(np.asarray(x, np.float32) * inv), -127, 127).astype(np.int8), s


def _qh_exact_scaling(x):
    x = np.asarray(x, np.float32)
    am = np.float64(np.max(np.abs(x)))
    s = np.float32(am) / np.float32(127)
    if am == 0:
        return np.zeros(x.shape, np.int8), np.float32(0)
    return np.clip(np.rint(x.astype(np.float64) * 127 / am), -127, 127).astype(np.int8), s


def _qr_per_token(x_bits):
    x = bf16(x_bits)
    n, H, D = x.shape
    codes = np.zeros((n, H, D), np.int8)
    scales = np.zeros((n, H), np.float32)
    for t in range(n):
        c, s = Q.quantize_head(x[t].reshape(-1))
        codes[t] = c.reshape(H, D)
        scales[t] = s
    return codes, scales


def _write_big_endian(k, v, layer, kn, vn, sm, H, D):
    Q.write_slots_i8(k, v, layer, kn, vn, sm, H, D)
    bs = k.shape[2]
    for s in sm:
        if s < 0:
            continue
        for pool in (k, v):
            r = pool[s // bs, layer, s % bs]
            for g in range(H):
                seg = r[H * D + 4 * g:H * D + 4 * g + 4]
                seg[:] = seg[::-1].copy()


def _write_scales_first(k, v, layer, kn, vn, sm, H, D):
    bs = k.shape[2]
    for t, s in enumerate(sm):
        if s < 0:
            continue
        for pool, new in ((k, kn), (v, vn)):
            codes, scales = Q.quantize_rows(np.asarray(new[t:t + 1]))
            r = pool[s // bs, layer, s % bs]
            r[:4 * H] = scales[0].astype("<f4").view(np.uint8)
            r[4 * H:4 * H + H * D] = Q.code_bytes(codes[0]).reshape(-1)


def _write_twos_complement(k, v, layer, kn, vn, sm, H, D):
    """Codes stored as two's-complement bytes instead of offset binary."""
    Q.write_slots_i8(k, v, layer, kn, vn, sm, H, D)
    bs = k.shape[2]
    for s in sm:
        if s < 0:
            continue
        for pool in (k, v):
            r = pool[s // bs, layer, s % bs]
            r[:H * D] = (r[:H * D].astype(np.int16) - 128).astype(np.int8).view(np.uint8)


def _deq_divides(rows, H, D):
    codes, scales = Q.unpack_rows(rows, H, D)
    return codes.astype(np.float64) / scales.astype(np.float64)[:, :, None]


def _decode_i8_kv_swapped(k, v, layer, q, bt, lens, offs, scale):
    return Q.decode_attention_i8(v, k, layer, q, bt, lens, offs, scale)


def _decode_i8_codes_only(k, v, layer, q, bt, lens, offs, scale):
    B, Hq, D = q.shape
    H = Q._heads(k.shape[3], D)
    out = np.zeros((B, Hq, D))
    for b in range(B):
        kb, _ = Q.unpack_rows(oracle.gather_loop(k, layer, bt[b], int(lens[b]), int(offs[b])), H, D)
        vb = Q.dequantize_rows(oracle.gather_loop(v, layer, bt[b], int(lens[b]), int(offs[b])),
                               H, D)
        for h in range(Hq):
            g = h // (Hq // H)
            out[b, h] = oracle.attention_fp64(oracle.widen(q[b, h]), kb[:, g].astype(np.float64),
                                              vb[:, g], scale)
    return out


PLANTED = [
    ("scale absmax/128", lambda: check_half_way_cases(_qh_div128)),
    ("round half away from zero", lambda: check_half_way_cases(_qh_round_away)),
    ("floor instead of round", lambda: check_half_way_cases(_qh_floor)),
    ("multiply by reciprocal", lambda: check_fp32_decisions(_qh_reciprocal)),
    ("exact fp64 scaling", lambda: check_fp32_decisions(_qh_exact_scaling)),
    ("one scale per token", lambda: check_per_head_scale(_qr_per_token)),
    ("scales big-endian", lambda: check_row_format(_write_big_endian, Q.unpack_rows)),
    ("scales before codes", lambda: check_row_format(_write_scales_first, Q.unpack_rows)),
    ("codes two's complement", lambda: check_row_format(_write_twos_complement, Q.unpack_rows)),
    ("dequant divides", lambda: check_dequant_formula(_deq_divides)),
    ("decode reads V for K", lambda: check_representable_exact(Q.write_slots_i8,
                                                               _decode_i8_kv_swapped)),
    ("decode ignores K scales", lambda: check_representable_exact(Q.write_slots_i8,
                                                                  _decode_i8_codes_only)),
]


@pytest.mark.parametrize("name,run", PLANTED, ids=[p[0] for p in PLANTED])
def test_quant_pins_catch_planted_mistakes(name, run):
    with pytest.raises(AssertionError):
        run()
