"""Pins for the oracle: what the pages and the mathematics fix, independent of
the oracle's own code.

Each ``check_*`` helper takes the implementation under test as arguments so
that ``test_pins_catch_planted_mistakes`` can run the same checks against
deliberately broken copies of the oracle (on the CPU) and show that each
plausible mistake fails at least one pin.
"""

import math
import os

import numpy as np
import pytest
import torch

import oracle
from oracle import oracle as O

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _rows(path):
    out = []
    with open(path) as f:
        for line in f:
            line = line.strip()
            if line and not line.startswith("#"):
                out.append(line.split())
    return out


def _tagged_pool(N, L, bs, H, D, dtype=np.float32):
    """Pool whose every element encodes (block, layer, row, head, d), so a
    gathered row tells where it came from."""
    idx = np.arange(N * L * bs * H * D, dtype=np.int64).reshape(N, L, bs, H, D)
    if dtype == np.uint16:
        return (idx % 65521).astype(np.uint16)
    return idx.astype(np.float32)


# ---------------------------------------------------------------------------
# reusable checks
# ---------------------------------------------------------------------------

def check_block_table_example(slot_of, build_slot_mapping, gather_loop):
    rows = _rows(os.path.join(GOLDEN, "block_table_7_3_12.txt"))
    table = [7, 3, 12]
    for tok, blk, row, slot in ((int(a), int(b), int(c), int(d)) for a, b, c, d in rows):
        assert slot_of(table, 0, tok, 16) == slot
        assert slot // 16 == blk and slot % 16 == row
    sm = build_slot_mapping(np.array([table], np.int32), np.array([0], np.int32),
                            np.zeros(48, np.int32), np.arange(48, dtype=np.int32), 16)
    assert sm.tolist() == [int(r[3]) for r in rows]
    pool = _tagged_pool(16, 1, 16, 1, 1)
    got = gather_loop(pool, 0, table, 48, 0)[:, 0, 0]
    want = np.array([pool[int(r[1]), 0, int(r[2]), 0, 0] for r in rows])
    assert np.array_equal(got, want)


def check_slot_walk(slot_of):
    """Brute force: enumerate a table's rows in storage order (first block
    from the offset, later blocks from row 0) and number the tokens; every
    token's slot must match."""
    rng = np.random.default_rng(5)
    for bs in (1, 2, 4, 16):
        for _ in range(20):
            N = 40
            nblk = int(rng.integers(1, 6))
            table = rng.permutation(N)[:nblk]
            off = int(rng.integers(0, bs))
            tok = 0
            for k, blk in enumerate(table):
                for r in range(off if k == 0 else 0, bs):
                    assert slot_of(table, off, tok, bs) == int(blk) * bs + r
                    tok += 1


def check_gather_forms(gather_loop, gather_indexed):
    rng = np.random.default_rng(6)
    for bs in (1, 4, 16):
        pool = _tagged_pool(32, 3, bs, 2, 4)
        for _ in range(15):
            nblk = int(rng.integers(1, 6))
            table = rng.permutation(32)[:nblk]
            off = int(rng.integers(0, bs))
            n = int(rng.integers(0, nblk * bs - off + 1))
            layer = int(rng.integers(0, 3))
            a = gather_loop(pool, layer, table, n, off)
            b = gather_indexed(pool, layer, table, n, off)
            assert a.shape == (n, 2, 4)
            assert np.array_equal(a, b)


def check_identity_table(gather_loop):
    """Table 0,1,2,... : the sequence is a contiguous run of the layer."""
    N, L, bs = 12, 2, 4
    pool = _tagged_pool(N, L, bs, 3, 2)
    for layer in range(L):
        flat = pool[:, layer].reshape(N * bs, 3, 2)
        for off in range(bs):
            for n in (0, 1, 5, N * bs - off):
                got = gather_loop(pool, layer, list(range(N)), n, off)
                assert np.array_equal(got, flat[off:off + n])


def check_scatter_round_trip(build_slot_mapping, write_slots, gather_loop):
    rng = np.random.default_rng(7)
    N, L, bs, H, D = 24, 2, 4, 2, 3
    for _ in range(10):
        k = rng.standard_normal((N, L, bs, H, D)).astype(np.float32)
        v = rng.standard_normal((N, L, bs, H, D)).astype(np.float32)
        k0, v0 = k.copy(), v.copy()
        nblk = int(rng.integers(1, 6))
        table = rng.permutation(N)[:nblk]
        off = int(rng.integers(0, bs))
        n = int(rng.integers(1, nblk * bs - off + 1))
        layer = int(rng.integers(0, L))
        seq = np.zeros(n, np.int32)
        pad = rng.random(n) < 0.3
        seq[pad] = -1
        pos = np.arange(n, dtype=np.int32)
        sm = build_slot_mapping(np.array([table], np.int32), np.array([off], np.int32),
                                seq, pos, bs)
        assert np.all(sm[pad] == -1) and np.all(sm[~pad] >= 0)
        kn = rng.standard_normal((n, H, D)).astype(np.float32)
        vn = rng.standard_normal((n, H, D)).astype(np.float32)
        write_slots(k, v, layer, kn, vn, sm)
        gk = gather_loop(k, layer, table, n, off)
        gv = gather_loop(v, layer, table, n, off)
        # written rows come back; padded rows keep the old contents
        assert np.array_equal(gk[~pad], kn[~pad])
        assert np.array_equal(gv[~pad], vn[~pad])
        assert np.array_equal(gk[pad], gather_loop(k0, layer, table, n, off)[pad])
        # nothing outside the written rows changed
        touched = np.zeros((N, L, bs), bool)
        for s in sm[sm >= 0]:
            touched[s // bs, layer, s % bs] = True
        assert np.array_equal(k[~touched], k0[~touched])
        assert np.array_equal(v[~touched], v0[~touched])


def check_identity_scatter(build_slot_mapping, write_slots):
    """With the identity table, a scatter lays tokens out in pool order."""
    N, L, bs, H, D = 6, 1, 4, 1, 2
    k = np.zeros((N, L, bs, H, D), np.float32)
    v = np.zeros((N, L, bs, H, D), np.float32)
    n = N * bs - 1
    kn = np.arange(n * H * D, dtype=np.float32).reshape(n, H, D) + 1
    sm = build_slot_mapping(np.array([list(range(N))], np.int32), np.array([1], np.int32),
                            np.zeros(n, np.int32), np.arange(n, dtype=np.int32), bs)
    write_slots(k, v, 0, kn, -kn, sm)
    flat = k[:, 0].reshape(N * bs, H, D)
    assert np.array_equal(flat[1:], kn) and np.all(flat[0] == 0)


def _rand_case(rng, N=20, L=2, bs=4, Hkv=2, group=2, D=8, B=3, maxlen=30):
    k = rng.standard_normal((N, L, bs, Hkv, D)).astype(np.float32)
    v = rng.standard_normal((N, L, bs, Hkv, D)).astype(np.float32)
    q = rng.standard_normal((B, Hkv * group, D)).astype(np.float32)
    lens = rng.integers(0, maxlen + 1, size=B).astype(np.int32)
    offs = rng.integers(0, bs, size=B).astype(np.int32)
    mb = max(1, max(O.blocks_needed(int(n), bs, int(o)) for n, o in zip(lens, offs)))
    bt = np.full((B, mb), -1, np.int32)
    for b in range(B):
        nb = O.blocks_needed(int(lens[b]), bs, int(offs[b]))
        bt[b, :nb] = rng.choice(N, size=nb, replace=False)
    return k, v, q, bt, lens, offs


def check_attention_vs_sdpa(decode_attention):
    """Library cross-check: torch's scaled_dot_product_attention in fp64 on
    the gathered K/V, with kv heads repeated for grouped queries."""
    rng = np.random.default_rng(8)
    for group in (1, 2, 4):
        k, v, q, bt, lens, offs = _rand_case(rng, group=group)
        scale = 0.37
        got = decode_attention(k, v, 1, q, bt, lens, offs, scale)
        for b in range(len(lens)):
            kb = O.gather_indexed(k, 1, bt[b], int(lens[b]), int(offs[b])).astype(np.float64)
            vb = O.gather_indexed(v, 1, bt[b], int(lens[b]), int(offs[b])).astype(np.float64)
            if lens[b] == 0:
                assert np.all(got[b] == 0)
                continue
            qt = torch.from_numpy(q[b].astype(np.float64))[:, None, :]          # [Hq,1,D]
            kt = torch.from_numpy(kb).permute(1, 0, 2).repeat_interleave(group, 0)
            vt = torch.from_numpy(vb).permute(1, 0, 2).repeat_interleave(group, 0)
            ref = torch.nn.functional.scaled_dot_product_attention(
                qt, kt, vt, scale=scale)[:, 0, :].numpy()
            np.testing.assert_allclose(got[b], ref, rtol=0, atol=1e-12)


def check_attention_closed_forms(attention_fp64):
    rng = np.random.default_rng(9)
    D = 6
    q = rng.standard_normal(D)
    v = rng.standard_normal((5, D))
    # one token: softmax of a single logit is 1
    assert np.array_equal(attention_fp64(q, rng.standard_normal((1, D)), v[:1], 0.5), v[0])
    # equal keys: uniform weights, the output is the mean of V
    k_eq = np.tile(rng.standard_normal(D), (5, 1))
    np.testing.assert_allclose(attention_fp64(q, k_eq, v, 0.5), v.mean(0), atol=1e-14)
    # one key aligned with q far above the rest: the output is that V row
    k = rng.standard_normal((5, D)) * 0.01
    k[3] = q * 1e3
    np.testing.assert_allclose(attention_fp64(q, k, v, 1.0), v[3], atol=1e-12)
    # two tokens: logistic weights in closed form
    k2 = rng.standard_normal((2, D))
    s = 0.7 * (k2 @ q)
    w1 = 1.0 / (1.0 + math.exp(s[0] - s[1]))
    np.testing.assert_allclose(attention_fp64(q, k2, v[:2], 0.7),
                               (1 - w1) * v[0] + w1 * v[1], atol=1e-14)
    # no tokens: zeros
    assert np.array_equal(attention_fp64(q, np.zeros((0, D)), np.zeros((0, D)), 1.0),
                          np.zeros(D))


def check_block_permutation_invariance(decode_attention):
    """Moving blocks to other physical ids and relabelling the tables to
    match must not change the result (logical order is all that counts)."""
    rng = np.random.default_rng(10)
    k, v, q, bt, lens, offs = _rand_case(rng)
    a = decode_attention(k, v, 0, q, bt, lens, offs, 0.3)
    perm = rng.permutation(k.shape[0])          # new id of old block i
    k2 = np.empty_like(k); v2 = np.empty_like(v)
    k2[perm] = k; v2[perm] = v
    bt2 = np.where(bt >= 0, perm[np.maximum(bt, 0)], -1).astype(np.int32)
    b = decode_attention(k2, v2, 0, q, bt2, lens, offs, 0.3)
    np.testing.assert_allclose(a, b, atol=1e-13)


# ---------------------------------------------------------------------------
# the pins, against the real oracle
# ---------------------------------------------------------------------------

def test_block_table_example():
    check_block_table_example(O.slot_of, O.build_slot_mapping, O.gather_loop)


def test_exercise_30_tokens():
    for n, bs, blocks, slots, last, util, frag in _rows(
            os.path.join(GOLDEN, "exercise_30_tokens.txt")):
        n, bs, blocks, slots, last = int(n), int(bs), int(blocks), int(slots), int(last)
        assert oracle.blocks_needed(n, bs) == blocks
        assert oracle.capacity(blocks, bs, 0) == slots
        assert oracle.last_block_fill(n, bs) == last
        assert oracle.last_block_fill(n, bs) / bs == float(util)
        assert oracle.fragmentation_ratio(blocks, bs, n) == float(frag)


def test_waste_example():
    (req, bs, per_req, kb, wasted, wasted_kb), = _rows(os.path.join(GOLDEN, "waste_example.txt"))
    req, bs, per_req = int(req), int(bs), int(per_req)
    # each request uses one block, half filled: allocated slots minus used tokens
    frag = oracle.fragmentation_ratio(req, bs, req * (bs - per_req))
    assert frag * req * bs == int(wasted)
    assert int(wasted) * int(kb) == int(wasted_kb)
    assert abs(int(wasted_kb) * 1024 / 1e6 - 74) < 2      # the page's "about 74 MB"


def test_capacity_and_offsets():
    assert oracle.capacity(3, 16, 5) == 43
    assert oracle.blocks_needed(43, 16, 5) == 3
    assert oracle.blocks_needed(44, 16, 5) == 4
    assert oracle.blocks_needed(0, 16, 5) == 0
    assert oracle.last_block_fill(43, 16, 5) == 16
    pool = _tagged_pool(8, 1, 16, 1, 1)
    assert oracle.gather_loop(pool, 0, [1, 2, 3], 43, 5).shape[0] == 43
    with pytest.raises(IndexError):
        oracle.gather_loop(pool, 0, [1, 2, 3], 44, 5)


def test_slot_walk():
    check_slot_walk(O.slot_of)


def test_gather_forms_agree():
    check_gather_forms(O.gather_loop, O.gather_indexed)


def test_identity_table_is_contiguous():
    check_identity_table(O.gather_loop)


def test_scatter_round_trip_and_canaries():
    check_scatter_round_trip(O.build_slot_mapping, O.write_slots, O.gather_loop)


def test_identity_scatter():
    check_identity_scatter(O.build_slot_mapping, O.write_slots)


def test_scatter_rejects_bad_slots():
    k = np.zeros((4, 1, 4, 1, 1), np.float32)
    v = k.copy()
    row = np.ones((1, 1, 1), np.float32)
    with pytest.raises(IndexError):
        oracle.write_slots(k, v, 0, row, row, np.array([-2]))
    with pytest.raises(IndexError):
        oracle.write_slots(k, v, 0, row, row, np.array([16]))
    with pytest.raises(ValueError):
        oracle.write_slots(k, v, 0, np.ones((2, 1, 1), np.float32),
                           np.ones((2, 1, 1), np.float32), np.array([3, 3]))
    k[:] = 0
    v[:] = 0
    oracle.write_slots(k, v, 0, row, row, np.array([-1]))
    assert not k.any() and not v.any()


def test_attention_vs_sdpa():
    check_attention_vs_sdpa(O.decode_attention)


def test_attention_closed_forms():
    check_attention_closed_forms(O.attention_fp64)


def test_block_permutation_invariance():
    check_block_permutation_invariance(O.decode_attention)


def test_decode_pairs_match_full():
    rng = np.random.default_rng(11)
    k, v, q, bt, lens, offs = _rand_case(rng, group=4)
    full = O.decode_attention(k, v, 1, q, bt, lens, offs, 0.25)
    pairs = [(b, h) for b in range(len(lens)) for h in range(q.shape[1])]
    sel = O.decode_attention_pairs(k, v, 1, q, bt, lens, offs, 0.25, pairs)
    for (b, h), x in sel.items():
        np.testing.assert_allclose(x, full[b, h], atol=1e-13)


def check_split_combine(combine):
    """Any split of the tokens, merged, equals direct attention."""
    rng = np.random.default_rng(12)
    D = 16
    for n in (1, 2, 17, 100):
        q = rng.standard_normal(D)
        k = rng.standard_normal((n, D)) * 2
        v = rng.standard_normal((n, D))
        direct = O.attention_fp64(q, k, v, 0.9)
        for nsplit in (1, 2, 3, 7, n):
            cuts = sorted(set([0, n] + list(rng.integers(0, n + 1, size=nsplit - 1))))
            got = combine(O.split_partials(q, k, v, 0.9, cuts), D)
            np.testing.assert_allclose(got, direct, atol=1e-13)
    assert np.array_equal(combine([], 4), np.zeros(4))


def test_split_combine_equals_direct():
    check_split_combine(O.combine_partials)


def test_widen_bf16_bits():
    bits = np.array([0x3F80, 0xC000, 0x3E20, 0x0000, 0x8000, 0x7F7F], np.uint16)
    want = np.array([1.0, -2.0, 0.15625, 0.0, -0.0, 3.3895313892515355e38])
    got = O.widen(bits)
    assert np.array_equal(got, want)
    assert np.signbit(got[4])
    # torch agrees on the bit meaning of bf16
    t = torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16).double().numpy()
    assert np.array_equal(t, want)


# ---------------------------------------------------------------------------
# planted mistakes: each broken copy of the oracle must fail some pin
# ---------------------------------------------------------------------------

def _slot_no_offset(table, offset, i, bs):
    return int(table[i // bs]) * bs + i % bs


def _slot_swapped(table, offset, i, bs):
    p = offset + i
    return int(table[p % bs if p % bs < len(table) else 0]) * bs + p // bs


def _gather_loop_ignores_offset(pool, layer, table, n, offset=0):
    return O.gather_loop(pool, layer, table, n, 0)


def _gather_loop_one_short(pool, layer, table, n, offset=0):
    out = O.gather_loop(pool, layer, table, n, offset)
    if n > 1:
        out = out.copy()
        out[-1] = out[-2]
    return out


def _build_sm_with(slot_fn):
    def f(bt, offs, seq, pos, bs):
        return np.array([-1 if s < 0 else slot_fn(bt[s], int(offs[s]), int(p), bs)
                         for s, p in zip(seq, pos)], dtype=np.int64)
    return f


def _write_writes_padding(k, v, layer, kn, vn, sm):
    bs = k.shape[2]
    for t, s in enumerate(sm):
        s = int(s) if s >= 0 else 0
        k[s // bs, layer, s % bs] = kn[t]
        v[s // bs, layer, s % bs] = vn[t]


def _attn_no_scale(q, k, v, scale):
    return O.attention_fp64(q, k, v, 1.0)


def _attn_wrong_sign(q, k, v, scale):
    return O.attention_fp64(q, k, v, -scale)


def _attn_unnormalised(q, k, v, scale):
    if k.shape[0] == 0:
        return np.zeros(v.shape[1])
    s = scale * (k @ q)
    return np.exp(s - s.max()) @ v


def _attn_keys_for_values(q, k, v, scale):
    return O.attention_fp64(q, k, k, scale)


def _decode_with(attn=None, gqa_mod=False):
    def f(k_cache, v_cache, layer, q, bt, lens, offs, scale):
        B, Hq, D = q.shape
        Hkv = k_cache.shape[3]
        out = np.zeros((B, Hq, D))
        for b in range(B):
            kb = O.widen(O.gather_loop(k_cache, layer, bt[b], int(lens[b]), int(offs[b])))
            vb = O.widen(O.gather_loop(v_cache, layer, bt[b], int(lens[b]), int(offs[b])))
            for h in range(Hq):
                g = h % Hkv if gqa_mod else h // (Hq // Hkv)
                out[b, h] = (attn or O.attention_fp64)(O.widen(q[b, h]), kb[:, g], vb[:, g], scale)
        return out
    return f


def _prefill_with(extra_keys=0, first_positions=False, gqa_mod=False):
    """A copy of the prefill oracle with one mistake planted."""
    def f(k_cache, v_cache, layer, q, bt, lens, offs, cu, scale):
        T, Hq, D = q.shape
        Hkv = k_cache.shape[3]
        out = np.zeros((T, Hq, D))
        for b in range(len(lens)):
            n, L = int(cu[b + 1] - cu[b]), int(lens[b])
            if n == 0:
                continue
            kb = O.widen(O.gather_loop(k_cache, layer, bt[b], L, int(offs[b])))
            vb = O.widen(O.gather_loop(v_cache, layer, bt[b], L, int(offs[b])))
            for i in range(n):
                P = i if first_positions else L - n + i
                hi = min(L, P + 1 + extra_keys)
                for h in range(Hq):
                    g = h % Hkv if gqa_mod else h // (Hq // Hkv)
                    out[cu[b] + i, h] = O.attention_fp64(O.widen(q[cu[b] + i, h]), kb[:hi, g],
                                                         vb[:hi, g], scale)
        return out
    return f


def _combine_unweighted(parts, head_dim):
    if not parts:
        return np.zeros(head_dim)
    return sum(acc for _, _, acc in parts) / sum(l for _, l, _ in parts)


def _combine_weight_sign(parts, head_dim):
    if not parts:
        return np.zeros(head_dim)
    M = max(m for m, _, _ in parts)
    num = sum(math.exp(M - m) * acc for m, _, acc in parts)
    den = sum(math.exp(M - m) * l for m, l, _ in parts)
    return num / den


# ---------------------------------------------------------------------------
# gather_batch: the batch form every GPU gather test checks against
# ---------------------------------------------------------------------------

# Hand-enumerated (block, row) pairs of three sequences at block_size 4, found
# by walking each table in storage order from its first-block offset, the way
# the ch.12 §2.1 figure walks the table [7, 3, 12]:
#   seq 0: table [5, 2],    offset 1, 6 tokens -> rows 1..3 of block 5, 0..2 of block 2
#   seq 1: table [7],       offset 3, 0 tokens -> nothing
#   seq 2: table [0, 3, 6], offset 2, 7 tokens -> rows 2..3 of 0, 0..3 of 3, 0 of 6
#   seq 3: table [4],       offset 0, 1 token  -> row 0 of block 4
GATHER_BATCH_EXAMPLE = dict(
    bs=4,
    tables=[[5, 2, -1], [7, -1, -1], [0, 3, 6], [4, -1, -1]],
    offsets=[1, 3, 2, 0],
    lens=[6, 0, 7, 1],
    rows=[(5, 1), (5, 2), (5, 3), (2, 0), (2, 1), (2, 2),
          (0, 2), (0, 3), (3, 0), (3, 1), (3, 2), (3, 3), (6, 0),
          (4, 0)],
)


def _tagged_pools(N, L, bs, H, D):
    """K and V pools whose every element names its own coordinates (V
    negated), so a misplaced, mixed-up or dropped row is visible."""
    idx = np.indices((N, L, bs, H, D)).astype(np.int64)
    tag = (((idx[0] * L + idx[1]) * bs + idx[2]) * H + idx[3]) * D + idx[4] + 1
    return tag, -tag


def check_gather_batch(gather_batch):
    ex = GATHER_BATCH_EXAMPLE
    bs, layer = ex["bs"], 1
    k, v = _tagged_pools(8, 2, bs, 2, 3)
    bt = np.array(ex["tables"], np.int32)
    lens = np.array(ex["lens"], np.int32)
    offs = np.array(ex["offsets"], np.int32)
    ko, vo = gather_batch(k, v, layer, bt, lens, offs)
    want_k = np.stack([k[blk, layer, row] for blk, row in ex["rows"]])
    want_v = np.stack([v[blk, layer, row] for blk, row in ex["rows"]])
    assert ko.shape == want_k.shape and vo.shape == want_v.shape
    assert np.array_equal(ko, want_k) and np.array_equal(vo, want_v)
    # per sequence it is the flat-index gather of step14_2 "Solution", in order
    rng = np.random.default_rng(41)
    N, bs2 = 40, 8
    k2, v2 = _tagged_pools(N, 1, bs2, 1, 2)
    lens2 = rng.integers(0, 30, size=6).astype(np.int32)
    offs2 = rng.integers(0, bs2, size=6).astype(np.int32)
    perm = rng.permutation(N)
    tables, used = np.full((6, 6), -1, np.int32), 0
    for b in range(6):
        nb = O.blocks_needed(int(lens2[b]), bs2, int(offs2[b])) if lens2[b] else 0
        tables[b, :nb] = perm[used:used + nb]
        used += nb
    ko2, vo2 = gather_batch(k2, v2, 0, tables, lens2, offs2)
    parts_k = [O.gather_indexed(k2, 0, tables[b], int(lens2[b]), int(offs2[b])) for b in range(6)]
    parts_v = [O.gather_indexed(v2, 0, tables[b], int(lens2[b]), int(offs2[b])) for b in range(6)]
    assert np.array_equal(ko2, np.concatenate(parts_k)) and np.array_equal(vo2, np.concatenate(parts_v))


def test_gather_batch_hand_example():
    check_gather_batch(O.gather_batch)


def _gather_batch_first_offset(k, v, layer, bt, lens, offs):
    return O.gather_batch(k, v, layer, bt, lens, np.full_like(offs, offs[0]))


def _gather_batch_reversed(k, v, layer, bt, lens, offs):
    ko, vo = O.gather_batch(k, v, layer, bt[::-1], lens[::-1], offs[::-1])
    return ko, vo


def _gather_batch_kv_swapped(k, v, layer, bt, lens, offs):
    ko, vo = O.gather_batch(k, v, layer, bt, lens, offs)
    return vo, ko


def _gather_batch_v_from_k(k, v, layer, bt, lens, offs):
    ko, _ = O.gather_batch(k, v, layer, bt, lens, offs)
    return ko, O.gather_batch(k, k, layer, bt, lens, offs)[1]


PLANTED = [
    ("slot ignores offset", lambda: check_slot_walk(_slot_no_offset)),
    ("slot quotient/remainder swapped", lambda: check_slot_walk(_slot_swapped)),
    ("example with swapped slot", lambda: check_block_table_example(
        _slot_swapped, _build_sm_with(_slot_swapped), O.gather_loop)),
    ("gather ignores offset", lambda: check_identity_table(_gather_loop_ignores_offset)),
    ("gather drops last row", lambda: check_gather_forms(_gather_loop_one_short, O.gather_indexed)),
    ("scatter writes padding", lambda: check_scatter_round_trip(
        O.build_slot_mapping, _write_writes_padding, O.gather_loop)),
    ("scatter slots ignore offset", lambda: check_identity_scatter(
        _build_sm_with(_slot_no_offset), O.write_slots)),
    ("attention without scale", lambda: check_attention_vs_sdpa(_decode_with(_attn_no_scale))),
    ("attention with sign flipped", lambda: check_attention_vs_sdpa(_decode_with(_attn_wrong_sign))),
    ("attention unnormalised", lambda: check_attention_closed_forms(_attn_unnormalised)),
    ("attention reads K for V", lambda: check_attention_closed_forms(_attn_keys_for_values)),
    ("GQA head map h % Hkv", lambda: check_attention_vs_sdpa(_decode_with(gqa_mod=True))),
    ("prefill mask admits the next key", lambda: check_prefill_vs_sdpa(_prefill_with(extra_keys=1))),
    ("prefill queries at the first positions",
     lambda: check_prefill_vs_sdpa(_prefill_with(first_positions=True))),
    ("prefill GQA head map h % Hkv", lambda: check_prefill_vs_sdpa(_prefill_with(gqa_mod=True))),
    ("combine without the max weights", lambda: check_split_combine(_combine_unweighted)),
    ("combine weights with the sign flipped", lambda: check_split_combine(_combine_weight_sign)),
    ("batch gather takes the first offset for all",
     lambda: check_gather_batch(_gather_batch_first_offset)),
    ("batch gather in reverse order", lambda: check_gather_batch(_gather_batch_reversed)),
    ("batch gather with K and V swapped", lambda: check_gather_batch(_gather_batch_kv_swapped)),
    ("batch gather reads V from K", lambda: check_gather_batch(_gather_batch_v_from_k)),
]


@pytest.mark.parametrize("name,run", PLANTED, ids=[p[0] for p in PLANTED])
def test_pins_catch_planted_mistakes(name, run):
    with pytest.raises((AssertionError, IndexError)):
        run()


# ---------------------------------------------------------------------------
# block copy and swap (copy-on-write and preemption by swapping)
# ---------------------------------------------------------------------------

def test_swap_round_trip_and_copy():
    rng = np.random.default_rng(13)
    N, L, bs, H, D = 10, 3, 4, 2, 2
    k = rng.standard_normal((N, L, bs, H, D)).astype(np.float32)
    v = rng.standard_normal((N, L, bs, H, D)).astype(np.float32)
    k0, v0 = k.copy(), v.copy()
    for layer in (-1, 1):
        hk, hv = O.swap_out(k, v, layer, [7, 2, 5])
        assert hk.shape == ((3, L) if layer < 0 else (3, 1)) + (bs, H, D)
        assert np.array_equal(hk[1], k[2] if layer < 0 else k[2, 1:2])
        # bring them back into other blocks: those blocks now hold the data
        O.swap_in(k, v, layer, [0, 1, 3], hk, hv)
        ls = slice(None) if layer < 0 else slice(1, 2)
        for src, dst in ((7, 0), (2, 1), (5, 3)):
            assert np.array_equal(k[dst, ls], k0[src, ls]) and np.array_equal(v[dst, ls], v0[src, ls])
        k[:], v[:] = k0, v0
    O.copy_blocks(k, v, 2, [4], [9])
    assert np.array_equal(k[9, 2], k0[4, 2]) and np.array_equal(k[9, :2], k0[9, :2])
    O.copy_blocks(k, v, -1, [1, 2], [6, 8])
    assert np.array_equal(v[6], v0[1]) and np.array_equal(v[8], v0[2])


def test_copy_on_write_keeps_shared_prefix():
    """Fork a sequence, append to the fork: the allocator reports a
    (shared, fresh) pair; after copying it, the fork reads the same prefix as
    the original and each writes its new token into its own block."""
    from oracle import allocator as OA
    bs, N = 4, 12
    m = OA.KVCacheManager(N, bs)
    rng = np.random.default_rng(14)
    k = np.zeros((N, 1, bs, 1, 2), np.float32)
    v = np.zeros_like(k)
    m.seq_new(1, offset=1)
    slots, _ = m.seq_append(1, 6)
    kn = rng.standard_normal((6, 1, 2)).astype(np.float32)
    O.write_slots(k, v, 0, kn, -kn, np.array(slots))
    m.seq_fork(1, 2)
    s2, cow = m.seq_append(2, 1)
    assert len(cow) == 1
    O.copy_blocks(k, v, -1, [c[0] for c in cow], [c[1] for c in cow])
    new2 = rng.standard_normal((1, 1, 2)).astype(np.float32)
    O.write_slots(k, v, 0, new2, -new2, np.array(s2))
    s1, cow1 = m.seq_append(1, 1)
    assert cow1 == []
    new1 = rng.standard_normal((1, 1, 2)).astype(np.float32)
    O.write_slots(k, v, 0, new1, -new1, np.array(s1))
    t1, t2 = m.seq_table(1), m.seq_table(2)
    g1 = O.gather_loop(k, 0, t1.block_ids, t1.num_tokens, t1.offset)
    g2 = O.gather_loop(k, 0, t2.block_ids, t2.num_tokens, t2.offset)
    assert np.array_equal(g1[:6], kn) and np.array_equal(g2[:6], kn)
    assert np.array_equal(g1[6], new1[0]) and np.array_equal(g2[6], new2[0])


# ---------------------------------------------------------------------------
# prefill attention
# ---------------------------------------------------------------------------

def _prefill_case(rng, group=2, B=3, maxlen=40):
    k, v, _, bt, lens, offs = _rand_case(rng, group=group, B=B, maxlen=maxlen)
    n = np.array([rng.integers(0, L + 1) for L in lens], np.int64)
    cu = np.concatenate([[0], np.cumsum(n)]).astype(np.int64)
    q = rng.standard_normal((int(cu[-1]), k.shape[3] * group, k.shape[4])).astype(np.float32)
    return k, v, q, bt, lens, offs, cu


def check_prefill_vs_sdpa(prefill):
    """Prefill equals SDPA with a bottom-right aligned causal mask."""
    rng = np.random.default_rng(15)
    for group in (1, 2, 4):
        k, v, q, bt, lens, offs, cu = _prefill_case(rng, group=group)
        got = prefill(k, v, 1, q, bt, lens, offs, cu, 0.31)
        for b in range(len(lens)):
            n, L = int(cu[b + 1] - cu[b]), int(lens[b])
            if n == 0:
                continue
            kb = O.gather_indexed(k, 1, bt[b], L, int(offs[b])).astype(np.float64)
            vb = O.gather_indexed(v, 1, bt[b], L, int(offs[b])).astype(np.float64)
            qt = torch.from_numpy(q[cu[b]:cu[b + 1]].astype(np.float64)).permute(1, 0, 2)
            kt = torch.from_numpy(kb).permute(1, 0, 2).repeat_interleave(group, 0)
            vt = torch.from_numpy(vb).permute(1, 0, 2).repeat_interleave(group, 0)
            # query i (position L-n+i) sees keys 0..L-n+i: a bottom-right aligned mask
            mask = torch.arange(L)[None, :] <= (L - n + torch.arange(n))[:, None]
            ref = torch.nn.functional.scaled_dot_product_attention(
                qt, kt, vt, attn_mask=mask, scale=0.31).permute(1, 0, 2).numpy()
            np.testing.assert_allclose(got[cu[b]:cu[b + 1]], ref, rtol=0, atol=1e-12)


def test_prefill_vs_sdpa_with_explicit_causal_mask():
    check_prefill_vs_sdpa(O.prefill_attention)


def test_prefill_rows_vs_sdpa():
    """The sampled-rows form, checked row by row against SDPA with the
    bottom-right causal mask (including sequences with no queries)."""
    rng = np.random.default_rng(17)
    for group in (1, 4):
        k, v, q, bt, lens, offs, cu = _prefill_case(rng, group=group, B=4)
        Hq = q.shape[1]
        rows = [(t, h) for t in range(int(cu[-1])) for h in range(Hq)]
        got = O.prefill_attention_rows(k, v, 1, q, bt, lens, offs, cu, 0.27, rows)
        for b in range(len(lens)):
            n, L = int(cu[b + 1] - cu[b]), int(lens[b])
            if n == 0:
                continue
            kb = O.gather_indexed(k, 1, bt[b], L, int(offs[b])).astype(np.float64)
            vb = O.gather_indexed(v, 1, bt[b], L, int(offs[b])).astype(np.float64)
            qt = torch.from_numpy(q[cu[b]:cu[b + 1]].astype(np.float64)).permute(1, 0, 2)
            kt = torch.from_numpy(kb).permute(1, 0, 2).repeat_interleave(group, 0)
            vt = torch.from_numpy(vb).permute(1, 0, 2).repeat_interleave(group, 0)
            mask = torch.arange(L)[None, :] <= (L - n + torch.arange(n))[:, None]
            ref = torch.nn.functional.scaled_dot_product_attention(
                qt, kt, vt, attn_mask=mask, scale=0.27).permute(1, 0, 2).numpy()
            for i in range(n):
                for h in range(Hq):
                    np.testing.assert_allclose(got[(int(cu[b]) + i, h)], ref[i, h], rtol=0,
                                               atol=1e-12)


def test_prefill_whole_prompt_is_plain_causal_and_last_row_is_decode():
    rng = np.random.default_rng(16)
    k, v, _, bt, lens, offs = _rand_case(rng, group=2, B=2, maxlen=30)
    lens = np.maximum(lens, 1).astype(np.int32)
    for b in range(2):
        nb = O.blocks_needed(int(lens[b]), 4, int(offs[b]))
        bt[b, :nb] = np.arange(b * 10, b * 10 + nb)
    cu = np.concatenate([[0], np.cumsum(lens)]).astype(np.int64)
    q = rng.standard_normal((int(cu[-1]), 4, 8)).astype(np.float32)
    got = O.prefill_attention(k, v, 0, q, bt, lens, offs, cu, 0.5)
    for b in range(2):
        L = int(lens[b])
        kb = O.gather_indexed(k, 0, bt[b], L, int(offs[b])).astype(np.float64)
        vb = O.gather_indexed(v, 0, bt[b], L, int(offs[b])).astype(np.float64)
        qt = torch.from_numpy(q[cu[b]:cu[b + 1]].astype(np.float64)).permute(1, 0, 2)
        kt = torch.from_numpy(kb).permute(1, 0, 2).repeat_interleave(2, 0)
        vt = torch.from_numpy(vb).permute(1, 0, 2).repeat_interleave(2, 0)
        ref = torch.nn.functional.scaled_dot_product_attention(
            qt, kt, vt, is_causal=True, scale=0.5).permute(1, 0, 2).numpy()
        np.testing.assert_allclose(got[cu[b]:cu[b + 1]], ref, atol=1e-12)
        # the last prompt token attends to the whole sequence: a decode step
        dec = O.decode_attention(k, v, 0, q[cu[b + 1] - 1][None], bt[b:b + 1], lens[b:b + 1],
                                 offs[b:b + 1], 0.5)
        np.testing.assert_allclose(got[cu[b + 1] - 1], dec[0], atol=1e-12)
        # the first token attends only to itself: its V row
        np.testing.assert_allclose(got[cu[b]], np.repeat(vb[0], 2, axis=0), atol=1e-14)
