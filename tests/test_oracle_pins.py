"""Pins of the CPU oracle against what the source pages and mathematics fix.

Every oracle function is checked here against something other than itself:
the worked sequences printed on the Paddle permute page (tests/golden), the
packing order stated on the Vulkan GEMV page, closed forms, special cases
that reduce to a library matmul, and invariants.  A plausible mistake in the
oracle (a swapped nibble, a transposed operand, a dropped zero or scale, a
wrong rounding mode) fails at least one of these.
"""
import numpy as np
import pytest

import oracle
from helpers import bf16_bits, bf16_values, load_golden

G = load_golden("p1_permute_sequences.txt")


# ---------------------------------------------------------------------------
# Page-internal consistency of the permute derivation (these fix our reading
# of the page before the oracle is trusted with it).
# ---------------------------------------------------------------------------

def test_page_permute_kk_derivation_from_int8():
    """int8 permute_kk -> regroup -> %8*2 -> +1 on the second half = int4 permute_kk."""
    int8 = G["permute_kk_int8"]
    regrouped = G["permute_kk_int8_regrouped"]
    # the regrouping exchanges the second and third quarters
    assert regrouped == int8[0:4] + int8[8:12] + int8[4:8] + int8[12:16]
    mod = [(v % 8) * 2 for v in regrouped]
    assert mod == G["permute_kk_mod8x2"]
    int4 = [v + (1 if t >= 8 else 0) for t, v in enumerate(mod)]
    assert int4 == G["permute_kk_int4"]


def test_page_permute_kk_is_scatter_of_byte_order():
    """Moving source byte t to permute_kk[t] lays the bytes out in byte_order."""
    dst = G["permute_kk_int4"]
    assert sorted(dst) == list(range(16))
    laid = [None] * 16
    for t, d in enumerate(dst):
        laid[d] = t
    assert laid == G["byte_order"]


def test_page_byte_order_matches_pair_order():
    pairs = G["byte_pair_order"]
    assert [pairs[2 * i] // 2 for i in range(16)] == G["byte_order"]
    assert all(pairs[2 * i + 1] == pairs[2 * i] + 1 for i in range(16))


def test_page_fast_dequant_maps_pre_order_to_fragment_order():
    slots = G["fast_dequant_slots"]          # slot i holds element slots[i]
    pre = G["pre_dequant_order"]
    out = []
    for w in range(4):
        word = pre[8 * w:8 * w + 8]
        elem = [None] * 8
        for i in range(8):
            elem[slots[i]] = word[i]
        out += elem
    assert out == G["fragment_order"]


# ---------------------------------------------------------------------------
# Oracle permute, traced with nibble labels.
# ---------------------------------------------------------------------------

def _pack_rows(vals):
    """Two rows per byte along K, even row in the low nibble (the pack the
    quantiser page describes and the workload definition fixes)."""
    vals = np.asarray(vals, dtype=np.int64)
    return ((vals[0::2] & 0xF) | ((vals[1::2] & 0xF) << 4)).astype(np.uint8)


def _trace_permute(K, N):
    """Run the oracle permute on 4-bit planes of unique nibble ids.

    Returns src[pos] = id of the input nibble found at output nibble
    position pos (pos = 2*byte + (0 for low, 1 for high)); id = k*N + n.
    Valid because the permute only moves nibbles and never looks at them.
    """
    ids = np.arange(K * N, dtype=np.int64).reshape(K, N)
    planes = max(1, int(np.ceil(np.log2(K * N) / 4)))
    src = np.zeros(N * K, dtype=np.int64)
    for p in range(planes):
        out = oracle.permute(_pack_rows((ids >> (4 * p)) & 0xF), K, N)
        nib = np.empty(N * K, dtype=np.int64)
        nib[0::2] = out & 0xF
        nib[1::2] = out >> 4
        src |= nib << (4 * p)
    return src


@pytest.mark.parametrize("K,N", [(64, 4), (128, 8), (256, 12)])
def test_oracle_permute_matches_page_sequences(K, N):
    src = _trace_permute(K, N)
    assert np.array_equal(np.sort(src), np.arange(K * N)), "not a bijection"
    k_of, n_of = src // N, src % N
    runs_per_col = (K // 2) // 32          # 32-byte runs per column stream
    pre = np.array(G["pre_dequant_order"])
    frag = G["fragment_order"]
    slots = G["fast_dequant_slots"]
    for rho in range(N * K // 64):          # every 32-byte run of the output
        seg = slice(64 * rho, 64 * rho + 64)  # its 64 nibbles
        cols = set(n_of[seg].tolist())
        # "in four adjacent rows, every 32 elements are interleaved":
        # runs cycle through the four columns of a group, chunk by chunk
        group, rem = divmod(rho, 4 * runs_per_col)
        chunk, lane = divmod(rem, 4)
        assert cols == {4 * group + lane}
        ks = k_of[seg]
        for h in range(2):                  # two 16-byte groups per run
            g_k = ks[32 * h:32 * h + 32]
            base = 64 * chunk + 32 * h
            assert np.array_equal(g_k - base, pre), (rho, h)
            # the consumer's fast dequant then yields the fragment order
            out = []
            for w in range(4):
                word = (g_k - base)[8 * w:8 * w + 8].tolist()
                elem = [None] * 8
                for i in range(8):
                    elem[slots[i]] = word[i]
                out += elem
            assert out == frag


def test_oracle_permute_preserves_nibble_multiset():
    """The permute only moves nibbles: the multiset of nibble values of any
    input survives unchanged."""
    K, N = 64, 4
    rng = np.random.default_rng(1)
    packed = rng.integers(0, 256, (K // 2, N), dtype=np.uint8)
    out = oracle.permute(packed, K, N)
    # nibble multiset is preserved
    nib_in = np.concatenate([packed.ravel() & 0xF, packed.ravel() >> 4])
    nib_out = np.concatenate([out & 0xF, out >> 4])
    assert np.array_equal(np.bincount(nib_in, minlength=16), np.bincount(nib_out, minlength=16))


# ---------------------------------------------------------------------------
# Quantise + pack.
# ---------------------------------------------------------------------------

def _unpack_rows(packed):
    """Inverse of the pack along K (even row = low nibble), sign-extended."""
    lo = (packed & 0xF).astype(np.int64)
    hi = (packed >> 4).astype(np.int64)
    K2, N = packed.shape
    q = np.empty((2 * K2, N), np.int64)
    q[0::2], q[1::2] = lo, hi
    return np.where(q >= 8, q - 16, q)


def test_quantize_exact_grid():
    """W = (k-7)/16: absmax 7/16 gives scale exactly 1/16 and q = k - 7."""
    K = 16
    col = np.array([(k - 7) / 16.0 for k in range(15)] + [0.0])
    W = np.stack([col, -col, np.zeros(K), col * 2], axis=1)
    scale, packed = oracle.quantize_pack(bf16_bits(W))
    assert scale[0] == np.float32(1 / 16) and scale[1] == np.float32(1 / 16)
    assert scale[2] == 0.0 and scale[3] == np.float32(1 / 8)
    q = _unpack_rows(packed)
    expect = np.array([k - 7 for k in range(15)] + [0])
    assert np.array_equal(q[:, 0], expect)
    assert np.array_equal(q[:, 1], -expect)
    assert np.array_equal(q[:, 2], np.zeros(K))
    assert np.array_equal(q[:, 3], expect)


def test_quantize_rounds_half_away_from_zero():
    # scale 1/16; w/s = 0.5, 1.5, 2.5, -0.5, -2.5 exactly
    col = np.array([7, 0.5, 1.5, 2.5, -0.5, -2.5, 0, 0]) / 16.0
    scale, packed = oracle.quantize_pack(bf16_bits(col.reshape(-1, 1)))
    assert scale[0] == np.float32(1 / 16)
    assert _unpack_rows(packed)[:, 0].tolist() == [7, 1, 2, 3, -1, -3, 0, 0]


def test_quantize_pack_puts_even_row_in_low_nibble():
    col = np.array([7, 1, -7, 2]) / 16.0        # q = 7, 1, -7, 2
    _, packed = oracle.quantize_pack(bf16_bits(col.reshape(-1, 1)))
    assert packed[:, 0].tolist() == [0x17, 0x29]   # -7 & 0xF = 9


def test_quantize_invariants_random():
    rng = np.random.default_rng(0)
    K, N = 256, 48
    W = bf16_bits(rng.normal(0, 0.02, (K, N)))
    Wv = bf16_values(W)
    scale, packed = oracle.quantize_pack(W)
    amax = np.abs(Wv).max(axis=0)
    assert np.array_equal(scale, (amax.astype(np.float32) / np.float32(7)))
    q = _unpack_rows(packed)
    assert q.min() >= -7 and q.max() <= 7           # symmetric absmax never hits -8
    # each column's extreme maps to +-7
    assert np.all(np.abs(q).max(axis=0) == 7)
    err = np.abs(Wv - q * scale.astype(np.float64))
    assert np.all(err <= scale.astype(np.float64) * (0.5 + 1e-6))
    # sign symmetry of round-half-away
    _, packed_neg = oracle.quantize_pack(W ^ np.uint16(0x8000))
    assert np.array_equal(_unpack_rows(packed_neg), -q)


# ---------------------------------------------------------------------------
# GEMV.
# ---------------------------------------------------------------------------

def _pack_words(Q):
    """packed = (w7<<28)|...|(w1<<4)|w0 along K, eight weights per uint32."""
    N, K = Q.shape
    Q = Q.astype(np.uint64).reshape(N, K // 8, 8)
    words = np.zeros((N, K // 8), np.uint64)
    for j in range(8):
        words |= Q[:, :, j] << np.uint64(4 * j)
    return words.astype(np.uint32)


@pytest.mark.parametrize("act", [oracle.F32, oracle.BF16])
def test_gemv_matches_dense_matmul(act):
    rng = np.random.default_rng(2)
    N, K, C = 24, 64, 3
    Q = rng.integers(0, 16, (N, K))
    s = rng.uniform(0.5, 2.0, N)
    z = rng.uniform(6.0, 9.0, N)
    x = rng.normal(0, 1, (C, K))
    if act == oracle.BF16:
        s, z, x = bf16_bits(s), bf16_bits(z), bf16_bits(x)
        sv, zv, xv = bf16_values(s), bf16_values(z), bf16_values(x)
    else:
        s, z, x = s.astype(np.float32), z.astype(np.float32), x.astype(np.float32)
        sv, zv, xv = s.astype(np.float64), z.astype(np.float64), x.astype(np.float64)
    d, ref = oracle.gemv(_pack_words(Q), s, z, x, act)
    W = (Q - zv[:, None]) * sv[:, None]
    np.testing.assert_allclose(d, xv @ W.T, rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(ref, np.abs(xv) @ np.abs(W).T, rtol=1e-12, atol=1e-12)


def test_gemv_one_hot_picks_single_nibble():
    N, K = 4, 16
    Q = np.arange(N * K).reshape(N, K) % 16
    s = np.full(N, 1.0, np.float32)
    z = np.full(N, 8.0, np.float32)
    for k in range(K):
        x = np.zeros((1, K), np.float32)
        x[0, k] = 1.0
        d, _ = oracle.gemv(_pack_words(Q), s, z, x, oracle.F32)
        assert np.array_equal(d[0], Q[:, k] - 8.0)


def test_gemv_page_word_example():
    """Word 0x76543210 holds weights 0..7 at k = 0..7 (w0 in the low bits)."""
    qw = np.array([[0x76543210]], np.uint32)
    x = np.eye(8, dtype=np.float32)
    d, _ = oracle.gemv(qw, np.ones(1, np.float32), np.zeros(1, np.float32), x, oracle.F32)
    assert d[:, 0].tolist() == list(range(8))


def test_gemv_q_equal_zero_point_gives_zero_and_integers_exact():
    rng = np.random.default_rng(3)
    N, K = 8, 128
    Q = np.full((N, K), 8)
    x = rng.normal(0, 1, (2, K)).astype(np.float32)
    d, _ = oracle.gemv(_pack_words(Q), np.ones(N, np.float32), np.full(N, 8.0, np.float32), x, oracle.F32)
    assert np.all(d == 0.0)
    Q = rng.integers(0, 16, (N, K))
    xi = rng.integers(-5, 6, (2, K)).astype(np.float32)
    d, _ = oracle.gemv(_pack_words(Q), np.ones(N, np.float32), np.zeros(N, np.float32), xi, oracle.F32)
    assert np.array_equal(d, xi.astype(np.int64) @ Q.T)


def test_gemv_row_range_and_linearity():
    rng = np.random.default_rng(4)
    N, K = 16, 64
    qw = rng.integers(0, 2**32, (N, K // 8), dtype=np.uint64).astype(np.uint32)
    s = rng.uniform(0.1, 1, N).astype(np.float32)
    z = np.full(N, 8, np.float32)
    x1 = rng.normal(size=(1, K)).astype(np.float32)
    x2 = rng.normal(size=(1, K)).astype(np.float32)
    d1, _ = oracle.gemv(qw, s, z, x1, oracle.F32)
    d2, _ = oracle.gemv(qw, s, z, x2, oracle.F32)
    d12, _ = oracle.gemv(qw, s, z, np.concatenate([x1, x2]), oracle.F32)
    assert np.array_equal(d12, np.concatenate([d1, d2]))
    d3, _ = oracle.gemv(qw, s, z, (x1.astype(np.float64) * 2).astype(np.float32), oracle.F32)
    np.testing.assert_allclose(d3, 2 * d1, rtol=1e-12)
    part, _ = oracle.gemv(qw, s, z, x1, oracle.F32, rows=(3, 9))
    assert np.array_equal(part[0, 3:9], d1[0, 3:9]) and np.isnan(part[0, :3]).all()


# ---------------------------------------------------------------------------
# GEMM.
# ---------------------------------------------------------------------------

# ---------------------------------------------------------------------------
# GEMV over the quantiser's packed matrix (the operand of the permuted path).
# ---------------------------------------------------------------------------

def _pack_cols(Q):
    """Column pack of signed int4 Q [K, N]: byte (k/2, n) = (q[k] & 0xF) |
    (q[k+1] & 0xF) << 4 (two rows per byte, even row low)."""
    Q = np.asarray(Q)
    lo = (Q[0::2] & 0xF).astype(np.uint8)
    hi = (Q[1::2] & 0xF).astype(np.uint8)
    return (lo | (hi << 4)).astype(np.uint8)


def _signed_q(rng, K, N):
    return rng.integers(-8, 8, (K, N))


def test_gemv_packed_matches_dense_matmul():
    rng = np.random.default_rng(21)
    K, N, C = 64, 20, 3
    Q = _signed_q(rng, K, N)
    s = rng.uniform(0.01, 0.2, N).astype(np.float32)
    x = bf16_bits(rng.normal(0, 1, (C, K)))
    d, ref = oracle.gemv_packed(_pack_cols(Q), s, x)
    W = Q * s.astype(np.float64)[None, :]
    xv = bf16_values(x)
    np.testing.assert_allclose(d, xv @ W, rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(ref, np.abs(xv) @ np.abs(W), rtol=1e-12, atol=1e-12)


def test_gemm_packed_matches_dense_matmul_identity_and_gemv():
    """The GEMM over the quantiser's packed matrix: a numpy matmul of A and
    the signed weights, A = I returning q * scale exactly, a row of A equal
    to the packed GEMV of that row, and the bf16 GEMM of the same weights
    re-encoded as u = q + 8 with zero point 8 and a bf16 scale."""
    rng = np.random.default_rng(25)
    M, K, N = 20, 64, 24
    Q = _signed_q(rng, K, N)
    s = bf16_values(bf16_bits(rng.uniform(0.01, 0.2, N))).astype(np.float32)   # bf16-exact scales
    A = bf16_bits(rng.normal(0, 1, (M, K)))
    P = _pack_cols(Q)
    c, ref = oracle.gemm_packed_full(A, P, s)
    W = Q * s.astype(np.float64)[None, :]
    Ad = bf16_values(A)
    np.testing.assert_allclose(c, Ad @ W, rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(ref, np.abs(Ad) @ np.abs(W), rtol=1e-12, atol=1e-12)
    eye, _ = oracle.gemm_packed_full(bf16_bits(np.eye(K)), P, s)
    assert np.array_equal(eye, W)
    g, _ = oracle.gemv_packed(P, s, A[3:4])
    np.testing.assert_allclose(c[3], g[0], rtol=1e-13, atol=0)
    c8, _ = oracle.gemm_full(A, _pack_cols(Q + 8), bf16_bits(s), bf16_bits(np.full(N, 8.0)))
    np.testing.assert_allclose(c, c8, rtol=1e-12, atol=1e-12)


def test_gemv_packed_agrees_with_row_gemv_at_zero_point_8():
    """Two's complement q is the unsigned u = q + 8 with zero point 8: the
    row-layout GEMV over the re-encoded words must give the same products."""
    rng = np.random.default_rng(22)
    K, N, C = 128, 12, 4
    Q = _signed_q(rng, K, N)
    s = rng.uniform(0.01, 0.2, N).astype(np.float32)
    x = bf16_bits(rng.normal(0, 1, (C, K)))
    d, _ = oracle.gemv_packed(_pack_cols(Q), s, x)
    U = (Q + 8).T                     # [N, K], 0..15
    d_row, _ = oracle.gemv(_pack_words(U), s, np.full(N, 8.0, np.float32),
                           bf16_values(x).astype(np.float32), oracle.F32)
    np.testing.assert_allclose(d, d_row, rtol=1e-12, atol=1e-12)


def test_gemv_packed_one_hot_picks_signed_weight():
    rng = np.random.default_rng(23)
    K, N = 32, 8
    Q = _signed_q(rng, K, N)
    Q[5, 3], Q[6, 3] = -8, 7            # both ends of the range, both nibble positions
    s = np.linspace(0.5, 2.0, N).astype(np.float32)
    packed = _pack_cols(Q)
    for k in range(K):
        x = np.zeros((1, K), np.uint16)
        x[0, k] = 0x3F80                # bf16 1.0
        d, _ = oracle.gemv_packed(packed, s, x)
        assert np.array_equal(d[0], Q[k] * s.astype(np.float64))


def test_gemv_packed_of_quantised_matrix_is_within_half_step():
    """d over quantize_pack's output differs from x @ W by at most
    sum_k |x[k]| * scale[n] / 2 (each weight is off by at most half a step)."""
    rng = np.random.default_rng(24)
    K, N, C = 96, 10, 2
    W = bf16_bits(rng.normal(0, 0.02, (K, N)))
    scale, packed = oracle.quantize_pack(W)
    x = bf16_bits(rng.normal(0, 1, (C, K)))
    d, _ = oracle.gemv_packed(packed, scale, x)
    xv = bf16_values(x)
    exact = xv @ bf16_values(W)
    bound = np.abs(xv).sum(axis=1)[:, None] * scale.astype(np.float64)[None, :] / 2
    assert np.all(np.abs(d - exact) <= bound * (1 + 1e-9) + 1e-12)


def test_gemm_matches_dense_matmul():
    rng = np.random.default_rng(5)
    M, N, K = 12, 20, 32
    Q = rng.integers(0, 16, (K, N))
    A = bf16_bits(rng.normal(0, 1, (M, K)))
    s = bf16_bits(rng.uniform(0.005, 0.02, N))
    z = bf16_bits(rng.uniform(6, 9, N))
    c, ref = oracle.gemm_full(A, _pack_rows(Q), s, z)
    W = (Q - bf16_values(z)[None, :]) * bf16_values(s)[None, :]
    np.testing.assert_allclose(c, bf16_values(A) @ W, rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(ref, np.abs(bf16_values(A)) @ np.abs(W), rtol=1e-12, atol=1e-12)


def test_gemm_identity_A_returns_dequantised_weights():
    K, N = 16, 8
    rng = np.random.default_rng(6)
    Q = rng.integers(0, 16, (K, N))
    A = bf16_bits(np.eye(K))
    c, _ = oracle.gemm_full(A, _pack_rows(Q), bf16_bits(np.full(N, 0.25)), bf16_bits(np.full(N, 8.0)))
    assert np.array_equal(c, (Q - 8) * 0.25)


def test_gemm_sampled_equals_full():
    rng = np.random.default_rng(7)
    M, N, K = 9, 7, 20
    A = bf16_bits(rng.normal(size=(M, K)))
    B = rng.integers(0, 256, (K // 2, N), dtype=np.uint8)
    s, z = bf16_bits(np.full(N, 0.01)), bf16_bits(np.full(N, 8.0))
    full, _ = oracle.gemm_full(A, B, s, z)
    mi = rng.integers(0, M, 30)
    ni = rng.integers(0, N, 30)
    part, _ = oracle.gemm_at(A, B, s, z, mi, ni)
    assert np.array_equal(part, full[mi, ni])


# ---------------------------------------------------------------------------
# int8 weight-only variant: quantiser, permute, GEMV
# ---------------------------------------------------------------------------

def test_quantize_int8_exact_grid_and_ties():
    """Column max 127/128 gives scale exactly 2^-7 (IEEE fp32 division of a
    value 127 * 2^-7 by 127); multiples k * 2^-7 quantise to k, and the
    exact ties (k + 1/2) * 2^-7 round away from zero."""
    ks = np.arange(-127, 128)
    grid = ks * 2.0 ** -7
    ties = (np.arange(-127, 127) + 0.5) * 2.0 ** -7       # every half step inside the range
    K = max(grid.size, ties.size)
    W = np.zeros((K, 2))
    W[: grid.size, 0] = grid
    W[: ties.size, 1] = ties
    W[0, 1] = 127 * 2.0 ** -7                               # column 1 max |w| = 127/128 as well
    s, q = oracle.quantize_int8(bf16_bits(W))
    assert s[0] == np.float32(2.0 ** -7) and s[1] == np.float32(2.0 ** -7)
    assert np.array_equal(q[: grid.size, 0], ks)
    t = ties[1:]
    expect = np.where(t > 0, np.floor(t * 128) + 1, np.ceil(t * 128) - 1)   # away from zero
    assert np.array_equal(q[1: ties.size, 1], expect.astype(np.int64))
    assert q[0, 1] == 127


def test_quantize_int8_invariants_random():
    rng = np.random.default_rng(7)
    W = (rng.standard_normal((300, 24)) * 0.02).astype(np.float32)
    W[:, 5] = 0.0
    bits = bf16_bits(W)
    w = bf16_values(bits)
    s, q = oracle.quantize_int8(bits)
    amax = np.abs(w).max(axis=0)
    assert np.array_equal(s, (amax.astype(np.float32) / np.float32(127.0)).astype(np.float32))
    assert s[5] == 0 and not q[:, 5].any()
    qi = q.astype(np.int64)
    assert np.abs(qi).max() <= 127
    # the column maximum quantises to +-127
    top = np.abs(w).argmax(axis=0)
    for n in range(24):
        if n != 5:
            assert abs(qi[top[n], n]) == 127
    # within half a step, plus the rounding of the fp32 quotient (|w/s| <= 127,
    # so at most 2^-17 of a step) that decides ties
    err = np.abs(w - qi * s.astype(np.float64))
    assert np.all(err <= s.astype(np.float64) * (0.5 + 2.0 ** -16))
    # sign symmetric
    s2, q2 = oracle.quantize_int8(bf16_bits(-W))
    assert np.array_equal(s2, s) and np.array_equal(q2, -q)


@pytest.mark.parametrize("K,N", [(64, 2), (128, 2), (64, 4)])
def test_permute_int8_places_elements_by_page_rules(K, N):
    """Every element lands where the page puts it: inside each 16-element
    group source t goes to permute_kk_int8[t]; two adjacent columns share
    each 128-byte line, 64 elements each."""
    dst16 = G["permute_kk_int8"]
    ids = np.arange(K * N).reshape(K, N)
    # label planes of 7 bits (int8 values 0..127) until every id is covered
    planes = int(np.ceil(np.log2(K * N) / 7))
    found = np.zeros(N * K, np.int64)
    for p in range(planes):
        out = oracle.permute_int8(((ids >> (7 * p)) & 0x7F).astype(np.int8), K, N)
        found |= out.astype(np.int64) << (7 * p)
    assert np.array_equal(np.sort(found), np.arange(K * N)), "not a bijection"
    for k in range(K):
        for n in range(N):
            pk = 16 * (k // 16) + dst16[k % 16]
            pos = pk % 64 + (pk // 64) * 128 + 64 * (n % 2) + K * 2 * (n // 2)
            assert found[pos] == k * N + n


def test_permute_int8_groups_pair_even_and_odd_halves():
    """Read back in output order, each 16-element group alternates the first
    and second halves of the source group: 0 8 1 9 2 10 ... (the inverse
    of the page's destination list)."""
    K, N = 64, 2
    q = np.tile(np.arange(K, dtype=np.int8)[:, None], (1, N))
    out = oracle.permute_int8(q, K, N)
    first = out[:16].tolist()
    assert first == [0, 8, 1, 9, 2, 10, 3, 11, 4, 12, 5, 13, 6, 14, 7, 15]


def test_gemv_int8_matches_dense_matmul_and_one_hot():
    rng = np.random.default_rng(3)
    K, N, C = 96, 40, 3
    q = rng.integers(-128, 128, (K, N), dtype=np.int64).astype(np.int8)
    s = rng.uniform(1e-3, 1e-2, N).astype(np.float32)
    x = bf16_bits(rng.standard_normal((C, K)))
    d, ref = oracle.gemv_int8(q, s, x)
    Wd = q.astype(np.float64) * s.astype(np.float64)[None, :]
    xd = bf16_values(x)
    assert np.allclose(d, xd @ Wd, rtol=1e-12, atol=1e-12)
    assert np.allclose(ref, np.abs(xd) @ np.abs(Wd), rtol=1e-12, atol=1e-12)
    onehot = np.zeros((1, K))
    onehot[0, 17] = 1.0
    d1, _ = oracle.gemv_int8(q, s, bf16_bits(onehot))
    assert np.array_equal(d1[0], q[17].astype(np.float64) * s.astype(np.float64))


def test_gemm_int8_matches_dense_matmul_identity_and_gemv():
    """The int8 GEMM: a numpy matmul of A and the dequantised weights; A = I
    returns q * scale exactly; a single row of A is the int8 GEMV of that
    row; sampled coordinates equal the full product."""
    rng = np.random.default_rng(4)
    M, K, N = 24, 64, 40
    q = rng.integers(-128, 128, (K, N), dtype=np.int64).astype(np.int8)
    s = rng.uniform(1e-3, 1e-2, N).astype(np.float32)
    A = bf16_bits(rng.standard_normal((M, K)))
    c, ref = oracle.gemm_int8_full(A, q, s)
    Wd = q.astype(np.float64) * s.astype(np.float64)[None, :]
    Ad = bf16_values(A)
    assert np.allclose(c, Ad @ Wd, rtol=1e-12, atol=1e-12)
    assert np.allclose(ref, np.abs(Ad) @ np.abs(Wd), rtol=1e-12, atol=1e-12)
    eye, _ = oracle.gemm_int8_full(bf16_bits(np.eye(K)), q, s)
    assert np.array_equal(eye, Wd)
    g, _ = oracle.gemv_int8(q, s, A[5:6])
    assert np.allclose(c[5], g[0], rtol=1e-13, atol=0)
    mi, ni = rng.integers(0, M, 50), rng.integers(0, N, 50)
    part, _ = oracle.gemm_int8_at(A, q, s, mi, ni)
    assert np.array_equal(part, c[mi, ni])


# ---------------------------------------------------------------------------
# W4A8: block_q8_1 activations in the PT plane layout
# ---------------------------------------------------------------------------

def _pt_offset(e, i, K):
    """The page's byte of element e of 128-block i: 16(floor(e/16) K/128 + i) + e mod 16."""
    return 16 * ((e // 16) * (K // 128) + i) + e % 16


def _pt_ds(pt, K, i, j):
    """(d, s) of q8_1 block j of 128-block i, from plane 8, as float64 (numpy's half)."""
    o = 16 * (8 * (K // 128) + i) + 4 * j
    return (float(np.frombuffer(bytes(pt[o:o + 2]), np.float16)[0]),
            float(np.frombuffer(bytes(pt[o + 2:o + 4]), np.float16)[0]))


def _int_activations(C, K, seed):
    """Integer activations with a 127 in every 32-block (so d = 1 exactly),
    the rest in -15..15 (so s = sum qs is exact in half)."""
    rng = np.random.default_rng(seed)
    x = rng.integers(-15, 16, (C, K)).astype(np.float64)
    x[:, ::32] = 127
    return x


def test_q8_1_pt_layout_places_elements_by_page_formula():
    K, C = 5120, 2
    x = _int_activations(C, K, 5)
    pt = oracle.quantize_q8_1_pt(bf16_bits(x))
    assert pt.shape == (C, 144 * K // 128)
    for c in range(C):
        qs = pt[c].view(np.int8)
        for i in range(K // 128):
            for e in range(128):
                assert qs[_pt_offset(e, i, K)] == x[c, 128 * i + e]
            for j in range(4):
                d, s = _pt_ds(pt[c], K, i, j)
                blk = x[c, 128 * i + 32 * j:128 * i + 32 * j + 32]
                assert d == 1.0 and s == blk.sum()


def test_q8_1_quantiser_rounds_half_away_and_stores_halves():
    K = 128
    x = np.zeros((1, K))
    x[0, :32] = np.arange(32) - 15.5          # block 0: ties (k + 1/2) around a max of 127 ...
    x[0, 0] = 127.0                            # ... so d = 1
    x[0, 32:64] = np.linspace(-0.3, 0.7, 32)  # block 1: a general block
    # block 2 all zero: d = s = 0
    x[0, 96:128] = 1e-3                        # block 3: tiny values, d a subnormal-free half
    xb = bf16_bits(x)
    xv = bf16_values(xb)[0]
    pt = oracle.quantize_q8_1_pt(xb)[0]
    qs = np.array([pt.view(np.int8)[_pt_offset(e, 0, K)] for e in range(128)], dtype=np.int64)
    t = xv[1:32]
    assert np.array_equal(qs[1:32], np.where(t > 0, np.floor(t) + 1, np.ceil(t) - 1))  # away from zero
    assert qs[0] == 127
    for j, blk in enumerate((xv[:32], xv[32:64], xv[64:96], xv[96:128])):
        d32 = np.float32(np.abs(blk).max()) / np.float32(127.0)
        q = qs[32 * j:32 * j + 32]
        if d32 != 0:
            # within half a step (plus the fp32 quotient's rounding)
            assert np.all(np.abs(blk - q * np.float64(d32)) <= np.float64(d32) * (0.5 + 2.0 ** -16))
        else:
            assert not q.any()
        d, s = _pt_ds(pt, K, 0, j)
        assert d == float(np.float16(d32))
        assert s == float(np.float16(np.float32(d32) * np.float32(q.sum())))


def test_half_conversion_rounds_ties_to_even_at_every_midpoint():
    """d and s are stored as IEEE binary16 (ggml_half), rounded to nearest
    even.  Checked against numpy's float16 cast on the midpoint between every
    pair of neighbouring halves (subnormal, normal, and 65520 between the
    largest half and the overflow), one fp32 step either side of each, every
    half itself, both signs, and random fp32 patterns."""
    grid = np.arange(0x7C00, dtype=np.uint16).view(np.float16).astype(np.float64)
    mids = (grid[:-1] + grid[1:]) / 2
    mids = np.append(mids, 65520.0)
    m32 = mids.astype(np.float32)
    assert np.array_equal(m32.astype(np.float64), mids)        # every midpoint is an fp32 value
    vals = np.concatenate([m32, np.nextafter(m32, np.float32(np.inf)), np.nextafter(m32, np.float32(0)),
                           grid.astype(np.float32), np.float32([65519.0, 65536.0, 1e30, 1e-30, np.inf])])
    rng = np.random.default_rng(20)
    rand = rng.integers(0, 2 ** 32, 200000, dtype=np.uint64).astype(np.uint32).view(np.float32)
    vals = np.concatenate([vals, -vals, rand[~np.isnan(rand)]])
    got = oracle.float_to_half(vals)
    with np.errstate(over="ignore"):
        want = vals.astype(np.float16).view(np.uint16)
    assert np.array_equal(got, want)
    # ties go to the even neighbour: 1 + 2^-11 lies between 1 and 1 + 2^-10
    assert oracle.float_to_half(np.float32([1 + 2.0 ** -11]))[0] == 0x3C00
    assert oracle.float_to_half(np.float32([1 + 3 * 2.0 ** -11]))[0] == 0x3C02
    assert oracle.float_to_half(np.float32([2.0 ** -25, 3 * 2.0 ** -25]))[0] == 0x0000
    assert oracle.float_to_half(np.float32([3 * 2.0 ** -25]))[0] == 0x0002


def test_half_decoding_is_exact_for_every_pattern():
    """The W4A8 GEMV reads d and s back as exact doubles: all 65536 binary16
    patterns against numpy's float16 widening, with the closed forms of the
    smallest subnormal, one, the largest half and infinity."""
    h = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    got = oracle.half_to_double(h)
    want = h.view(np.float16).astype(np.float64)
    nan = np.isnan(want)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan], want[~nan])
    assert np.array_equal(np.signbit(got[~nan]), np.signbit(want[~nan]))
    assert got[0x0001] == 2.0 ** -24 and got[0x3C00] == 1.0 and got[0x7BFF] == 65504.0
    assert got[0x7C00] == np.inf and got[0xFC00] == -np.inf


def test_w4a8_gemv_reduces_to_exact_gemv_on_integer_activations():
    """With d = 1 and s = sum qs exact, the W4A8 product equals the plain
    int4 GEMV of the same weights and activations."""
    N, K, C = 24, 256, 3
    rng = np.random.default_rng(8)
    qw = rng.integers(0, 2 ** 32, (N, K // 8), dtype=np.uint64).astype(np.uint32)
    scale = bf16_bits(rng.uniform(0.01, 0.05, N))
    zero = bf16_bits(np.full(N, 8.0))
    x = _int_activations(C, K, 9)
    pt = oracle.quantize_q8_1_pt(bf16_bits(x))
    d8, _ = oracle.gemv_w4a8(qw, scale, zero, pt, K)
    d, _ = oracle.gemv(qw, scale, zero, bf16_bits(x), oracle.BF16)
    assert np.allclose(d8, d, rtol=1e-12, atol=1e-12)


def test_w4a8_gemv_matches_dense_matmul_of_dequantised_operands():
    """Zero point 0: d = W_deq @ x_hat with x_hat = d_b * qs, by a library matmul."""
    N, K, C = 16, 384, 2
    rng = np.random.default_rng(10)
    qw = rng.integers(0, 2 ** 32, (N, K // 8), dtype=np.uint64).astype(np.uint32)
    scale_v = rng.uniform(0.01, 0.05, N)
    scale = bf16_bits(scale_v)
    zero = bf16_bits(np.zeros(N))
    x = rng.standard_normal((C, K))
    pt = oracle.quantize_q8_1_pt(bf16_bits(x))
    d8, _ = oracle.gemv_w4a8(qw, scale, zero, pt, K)
    # dequantised weights from the page's packing: nibble j of word i is k = 8i + j
    q = np.zeros((N, K))
    for j in range(8):
        q[:, j::8] = (qw >> (4 * j)) & 0xF
    Wd = q * bf16_values(scale)[:, None]
    xh = np.zeros((C, K))
    for c in range(C):
        qs = pt[c].view(np.int8)
        for i in range(K // 128):
            for e in range(128):
                d, _ = _pt_ds(pt[c], K, i, e // 32)
                xh[c, 128 * i + e] = d * qs[_pt_offset(e, i, K)]
    assert np.allclose(d8, xh @ Wd.T, rtol=1e-12, atol=1e-12)


def test_q8_1_pt_layout_matches_page_example():
    """The page's K = 5120 example: 40 blocks of 128 elements, 4 (d, s) pairs
    each, planes 0..7 of 16-byte blocks holding elements 16p..16p+15, and
    plane 8 holding every (d, s)."""
    P = load_golden("p4_pt_layout.txt")
    K = P["k"][0]
    nb = P["blocks"][0]
    assert K // P["elements_per_block"][0] == nb
    assert P["elements_per_block"][0] // P["q8_1_elements"][0] == P["ds_pairs_per_block"][0]
    B = P["block_bytes_per_plane"][0]
    rng = np.random.default_rng(4)
    x = rng.integers(-15, 16, (1, K)).astype(np.float64)
    x[:, ::32] = 127
    pt = oracle.quantize_q8_1_pt(bf16_bits(x))[0]
    assert pt.size == (P["ds_plane"][0] + 1) * nb * B
    qs = pt.view(np.int8)
    for p, e0 in enumerate(P["plane_first_elements"]):
        plane = qs[p * nb * B:(p + 1) * nb * B].reshape(nb, B)
        assert np.array_equal(plane, x[0].reshape(nb, 128)[:, e0:e0 + 16])
    ds = pt[P["ds_plane"][0] * nb * B:].view(np.float16).reshape(nb, P["ds_pairs_per_block"][0], 2)
    sums = x[0].reshape(nb, 4, 32).sum(axis=2)
    assert np.all(ds[:, :, 0] == 1.0) and np.array_equal(ds[:, :, 1].astype(np.float64), sums)
