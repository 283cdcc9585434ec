"""Pins of the oracle's ternary formats and MMVQ (no GPU).

Page: "三值量化模型的无损压缩" -- section 2 (the PTQ1_0 block and the PTQ1_1
superblock that packs eight of them), section 3 (the MMVQ product
d[r,c] = sum_k W[r,k] x[c,k]), 3.1 (x as block_q8_1 in the PT layout) and
3.2 (where each trit of a PTQ1_0 block sits).  The sizes, counts and the
worked placement example are the page's (tests/golden/p4_ternary_formats.txt);
the products are checked against numpy matmuls of the dequantised operands.
"""
import math

import numpy as np
import pytest

import oracle
import synth
from helpers import bf16_bits, load_golden

G = load_golden("p4_ternary_formats.txt")


def _block(trits, d=0x3C00):
    """One PTQ1_0 block (28 bytes) of the given 128 trits."""
    t = np.asarray(trits, dtype=np.int8).reshape(1, 128)
    return oracle.ptq1_0_pack(t, np.array([[d]], np.uint16))[0, 0]


def _changed_bytes(e):
    """Bytes of a block that change when weight e goes from -1 to +1 (the
    others at -1), with the change in value of each."""
    base = np.full(128, -1, np.int8)
    b0 = _block(base).astype(np.int64)
    t = base.copy()
    t[e] = 0
    b1 = _block(t).astype(np.int64)
    return {int(i): int(b1[i] - b0[i]) for i in np.nonzero(b1 != b0)[0]}


def _pt_dequant(pt, K):
    """x as the PT bytes hold it: qs * d per element (numpy's float16 for d)."""
    pt = np.atleast_2d(pt)
    bpr = K // 128
    out = np.zeros((pt.shape[0], K))
    for c in range(pt.shape[0]):
        v = pt[c]
        for i in range(bpr):
            for j in range(4):
                o = 16 * (8 * bpr + i) + 4 * j
                d = float(np.frombuffer(bytes(v[o:o + 2]), np.float16)[0])
                for t in range(32):
                    e = 32 * j + t
                    out[c, 128 * i + e] = float(v[16 * ((e // 16) * bpr + i) + e % 16].astype(np.int8)) * d
    return out


def _dense_weights(trits, d_bits):
    """W[r, k] = d[r, k/128] * t[r, k] with numpy's float16 for d."""
    d = np.asarray(d_bits, np.uint16).view(np.float16).astype(np.float64)
    return trits.astype(np.float64) * np.repeat(d, 128, axis=1)


def _inputs(N, K, C, seed, outliers=0.0):
    ti = synth.ternary_inputs(N, K, C, seed=seed, outlier_fraction=outliers)
    return ti.trits.numpy(), synth.np_bits(ti.d), synth.np_bits(ti.x)


# ---------------------------------------------------------------------------
# PTQ1_0
# ---------------------------------------------------------------------------

def test_ptq1_0_sizes_match_page():
    blk = _block(np.zeros(128))
    assert blk.size == G["ptq1_0_block_bytes"][0] == 28 and 8 * blk.size == G["ptq1_0_block_bits"][0]
    assert G["ptq1_0_qs_bytes"][0] * G["qs_trits_per_byte"][0] == G["ptq1_0_qs_trits"][0]
    assert G["ptq1_0_qh_bytes"][0] * 8 // G["qh_bits_per_trit"][0] == G["ptq1_0_qh_trits"][0]
    assert G["ptq1_0_qs_trits"][0] + G["ptq1_0_qh_trits"][0] == 128
    assert G["head_trits"][0] + G["middle_trits"][0] + G["tail_trits"][0] == 128
    assert G["ptq1_0_qs_bytes"][0] + G["ptq1_0_qh_bytes"][0] + 2 == G["ptq1_0_block_bytes"][0]
    assert G["d_sign_bits"][0] + G["d_exponent_bits"][0] + G["d_mantissa_bits"][0] == 16
    # five trits fit a byte (3^5 = 243 <= 256), six do not
    assert 3 ** G["qs_trits_per_byte"][0] <= 256 < 3 ** (G["qs_trits_per_byte"][0] + 1)


def test_ptq1_0_places_each_weight_where_the_page_says():
    """First 80 weights: byte e & 15, trit e >> 4 (so byte 0 holds 0, 16, 32,
    48, 64 -- the page's example); next 40: byte e & 7 of the eight bytes
    after them, trit e >> 3; last 8: 2-bit fields of qh."""
    place = {e: _changed_bytes(e) for e in range(128)}
    assert all(len(v) == 1 for v in place.values())
    byte_of = {e: next(iter(v)) for e, v in place.items()}
    delta = {e: next(iter(v.values())) for e, v in place.items()}
    first = sorted((e for e in range(128) if byte_of[e] == 0), key=lambda e: delta[e])
    assert first == G["first_byte_elements"]
    for e in range(G["head_trits"][0]):
        assert byte_of[e] == (e & 15)
    for f in range(G["middle_trits"][0]):
        assert byte_of[80 + f] == 16 + (f & 7)
    for j in range(G["tail_trits"][0]):
        assert byte_of[120 + j] in (24, 25)
    # positions increase with e >> 4 (head) and e >> 3 (middle): within a
    # byte, the later element is the higher position
    for b in range(24):
        members = sorted(e for e in range(120) if byte_of[e] == b)
        assert len(members) == 5
        assert [delta[e] for e in members] == sorted(delta[e] for e in members)


def test_trit_digits_and_qh_fields_follow_the_stated_reading():
    """The reading the page leaves open: digit u = t + 1, a byte is sum u_p 3^p
    over positions p, and qh's tail trit j is the 2-bit field j of the
    little-endian 16-bit word."""
    for p, e in enumerate(G["first_byte_elements"]):
        assert _changed_bytes(e) == {0: 3 ** p}       # -1 -> 0 raises digit p by one
    for j in range(8):
        d = _changed_bytes(120 + j)
        assert d == {24 + j // 4: 1 << (2 * (j % 4))}


def test_five_trits_per_byte_is_a_bijection():
    """All 243 combinations of byte 0's five trits give 243 distinct bytes
    below 243, and decode back."""
    seen = {}
    for combo in range(243):
        t = np.zeros(128, np.int8)
        for p, e in enumerate(G["first_byte_elements"]):
            t[e] = (combo // 3 ** p) % 3 - 1
        blk = _block(t)
        seen[int(blk[0])] = combo
        back, _ = oracle.ptq1_0_unpack(blk.reshape(1, 1, 28))
        assert np.array_equal(back[0], t)
    assert sorted(seen) == list(range(243))


def test_ptq1_0_round_trip_and_rejects_non_trits():
    rng = np.random.default_rng(3)
    t = rng.integers(-1, 2, (7, 640)).astype(np.int8)
    d = rng.integers(0, 2 ** 16, (7, 5)).astype(np.uint16)      # any half pattern, sign included
    t2, d2 = oracle.ptq1_0_unpack(oracle.ptq1_0_pack(t, d))
    assert np.array_equal(t, t2) and np.array_equal(d, d2)
    bad = t.copy()
    bad[3, 100] = 2
    with pytest.raises(ValueError):
        oracle.ptq1_0_pack(bad, d)


# ---------------------------------------------------------------------------
# PTQ1_1
# ---------------------------------------------------------------------------

def test_ptq1_1_sizes_match_page():
    t, d, _ = _inputs(4, 1024, 1, 5)
    w = oracle.ptq1_1_encode(oracle.ptq1_0_pack(t, d))
    sb = w.sblocks.shape[-1]
    parts = [G["ptq1_1_qs_bytes"][0], G["ptq1_1_qh_bytes"][0],
             G["ptq1_1_mantissas"][0] * G["ptq1_1_mantissa_bits"][0] // 8, G["ptq1_1_exponent_bytes"][0]]
    assert sb == sum(parts) == 216
    assert parts[0] + parts[1] == G["ptq1_1_trit_bytes"][0]
    assert G["ptq1_1_blocks"][0] * (G["ptq1_0_qs_bytes"][0] + G["ptq1_0_qh_bytes"][0]) == G["ptq1_0_trit_bytes_for_1024"][0]
    assert parts[2] + parts[3] == G["ptq1_1_float_bytes"][0]
    assert G["ptq1_1_blocks"][0] * 2 == G["ptq1_0_float_bytes_for_8"][0]
    assert G["ptq1_1_blocks"][0] * G["ptq1_0_block_bytes"][0] - sb == G["saved_bytes"][0]
    assert G["ptq1_1_blocks"][0] * G["ptq1_0_block_bytes"][0] // G["saved_bytes"][0] == G["shrink_denominator"][0]
    assert G["ptq1_1_qh_bytes"][0] * G["qs_trits_per_byte"][0] == G["ptq1_1_qh_capacity_trits"][0]
    assert G["ptq1_1_qh_capacity_trits"][0] - G["ptq1_1_qh_trits"][0] == 1          # one free trit
    assert 256 ** G["ptq1_1_exponent_bytes"][0] * 3 == G["pattern_cases"][0]
    assert G["escape_index"][0] == G["pattern_cases"][0] - 1
    bits = 128 * math.log2(3) + G["exponent_entropy_centibits"][0] / 100 + G["d_mantissa_bits"][0]
    assert math.floor(100 * bits) == G["information_centibits"][0]     # printed cut to two decimals
    assert math.ceil(bits / 8) * 8 == G["rounded_bits"][0] and G["rounded_bits"][0] // 8 == G["rounded_bytes"][0]
    assert sb // G["ptq1_1_blocks"][0] == G["rounded_bytes"][0]


def test_ptq1_1_keeps_each_blocks_qs_bytes():
    """The MMVQ listing reads sub-block `sub`'s qs straight from the
    superblock as a PTQ1_0 qs array: the 24 bytes are carried over as they are."""
    t, d, _ = _inputs(6, 2048, 1, 6)
    blocks = oracle.ptq1_0_pack(t, d)
    w = oracle.ptq1_1_encode(blocks)
    for r in range(6):
        for b in range(16):
            sb, s = divmod(b, 8)
            assert np.array_equal(w.sblocks[r, sb, 24 * s:24 * s + 24], blocks[r, b, :24])


def _pattern_index(sblock):
    """exponents + 256 * (the free trit: position 4 of qh's last byte)."""
    return int(sblock[215]) + 256 * ((int(sblock[192 + 12]) // 81) % 3)


def test_ptq1_1_is_lossless_with_escapes():
    """Half the rows draw wild exponents, so the tensor has more than 767
    patterns: the codebook fills, indices past 255 and 511 use the free trit,
    the rest escape to 767; every trit and every d decodes as PTQ1_0 holds it."""
    t, d, _ = _inputs(2048, 1024, 1, 7, outliers=0.5)
    blocks = oracle.ptq1_0_pack(t, d)
    w = oracle.ptq1_1_encode(blocks)
    assert w.codebook.shape == (767, 8) and len(w.esc_idx) > 0
    t2, d2 = oracle.ptq1_1_unpack(w)
    assert np.array_equal(t2, t) and np.array_equal(d2, d)
    idx = np.array([_pattern_index(w.sblocks[r, 0]) for r in range(2048)])
    assert idx.max() == 767 and (idx < 768).all()
    assert np.array_equal(np.nonzero(idx == 767)[0], w.esc_idx)
    assert ((idx >= 256) & (idx < 512)).any() and ((idx >= 512) & (idx < 767)).any()
    for i, g in enumerate(w.esc_idx):
        assert np.array_equal(w.esc_patt[i], (d[g] >> 10) & 31)


def test_ptq1_1_codebook_orders_by_frequency():
    """Most frequent pattern first; equal counts in ascending order of the
    pattern (block 0's exponent most significant)."""
    pats = {"A": [9] * 8, "B": [10] * 8, "C": [8] * 7 + [12], "D": [11, 9, 9, 9, 9, 9, 9, 9]}
    rows = ["A"] * 5 + ["C"] * 3 + ["B"] * 3 + ["D"]
    d = np.array([[(e << 10) | 5 for e in pats[name]] for name in rows], np.uint16)
    t = np.zeros((len(rows), 1024), np.int8)
    w = oracle.ptq1_1_encode(oracle.ptq1_0_pack(t, d))
    assert [list(p) for p in w.codebook] == [pats["A"], pats["C"], pats["B"], pats["D"]]
    assert len(w.esc_idx) == 0


def test_ptq1_1_rejects_negative_scale():
    t = np.zeros((1, 1024), np.int8)
    d = np.full((1, 8), 0x3C00, np.uint16)
    d[0, 3] = 0xBC00       # -1.0: PTQ1_1 stores no sign bit
    with pytest.raises(ValueError):
        oracle.ptq1_1_encode(oracle.ptq1_0_pack(t, d))


@pytest.mark.parametrize("K", [1152, 5120, 17280])
def test_ptq1_1_pads_the_last_superblock(K):
    """K/128 blocks take ceil(K/1024) superblocks; the pad blocks hold zero
    trits and d = +0 and decode to nothing past K."""
    N = 3
    t, d, _ = _inputs(N, K, 1, 8)
    w = oracle.ptq1_1_encode(oracle.ptq1_0_pack(t, d))
    bpr, sbpr = K // 128, -(-K // 1024)
    assert w.sblocks.shape == (N, sbpr, 216)
    t2, d2 = oracle.ptq1_1_unpack(w)
    assert np.array_equal(t2, t) and np.array_equal(d2, d)
    pad = 8 * sbpr - bpr
    if pad:
        for r in range(N):
            p = w.codebook[_pattern_index(w.sblocks[r, -1])] if _pattern_index(w.sblocks[r, -1]) < 767 else None
            if p is not None:
                assert (p[8 - pad:] == 0).all()
            # zero trits are digit 1 at every position
            assert (w.sblocks[r, -1, 24 * (8 - pad):192] == 1 + 3 + 9 + 27 + 81).all()


# ---------------------------------------------------------------------------
# MMVQ
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("N,K,C", [(24, 1152, 3), (9, 5120, 1)])
def test_mmvq_matches_dense_matmul(N, K, C):
    t, d, x = _inputs(N, K, C, 9)
    pt = oracle.quantize_q8_1_pt(x)
    got, ref_abs = oracle.mmvq_ptq1_0(oracle.ptq1_0_pack(t, d), pt)
    want = _pt_dequant(pt, K) @ _dense_weights(t, d).T
    assert np.all(np.abs(got - want) <= 1e-12 * ref_abs)
    assert np.allclose(ref_abs, np.abs(_pt_dequant(pt, K)) @ np.abs(_dense_weights(t, d)).T, rtol=1e-12)


def test_mmvq_exact_on_integer_activations():
    """x integer with a 127 in every 32-block (d_x = 1): the product is W x
    exactly."""
    N, K, C = 16, 2048, 2
    t, d, _ = _inputs(N, K, C, 10)
    rng = np.random.default_rng(10)
    x = rng.integers(-15, 16, (C, K)).astype(np.float64)
    x[:, ::32] = 127
    got, _ = oracle.mmvq_ptq1_0(oracle.ptq1_0_pack(t, d), oracle.quantize_q8_1_pt(bf16_bits(x)))
    assert np.array_equal(got, x @ _dense_weights(t, d).T)


def test_mmvq_one_hot_picks_a_single_weight():
    N, K = 5, 1024
    t, d, _ = _inputs(N, K, 1, 11)
    blocks = oracle.ptq1_0_pack(t, d)
    W = _dense_weights(t, d)
    for k in (0, 15, 16, 79, 80, 119, 120, 127, 128, 1023):
        x = np.zeros((1, K))
        x[0, k] = 127.0
        got, _ = oracle.mmvq_ptq1_0(blocks, oracle.quantize_q8_1_pt(bf16_bits(x)))
        assert np.array_equal(got[0], 127.0 * W[:, k])


def test_mmvq_sign_symmetry_and_zero_trits():
    N, K, C = 6, 1024, 2
    t, d, x = _inputs(N, K, C, 12)
    pt = oracle.quantize_q8_1_pt(x)
    a, _ = oracle.mmvq_ptq1_0(oracle.ptq1_0_pack(t, d), pt)
    b, _ = oracle.mmvq_ptq1_0(oracle.ptq1_0_pack(-t, d), pt)
    z, _ = oracle.mmvq_ptq1_0(oracle.ptq1_0_pack(np.zeros_like(t), d), pt)
    assert np.array_equal(a, -b) and not z.any()


def test_mmvq_ptq1_1_equals_ptq1_0_with_escapes():
    N, K, C = 1000, 1152, 2
    t, d, x = _inputs(N, K, C, 13, outliers=0.9)
    pt = oracle.quantize_q8_1_pt(x)
    blocks = oracle.ptq1_0_pack(t, d)
    w = oracle.ptq1_1_encode(blocks)
    assert len(w.esc_idx) > 0
    a, ra = oracle.mmvq_ptq1_0(blocks, pt)
    b, rb = oracle.mmvq_ptq1_1(w, pt)
    assert np.array_equal(a, b) and np.array_equal(ra, rb)
    r, _ = oracle.mmvq_ptq1_1(w, pt, rows=(7, 9))
    assert np.array_equal(r[:, 7:9], a[:, 7:9]) and np.isnan(r[:, :7]).all()
