"""GPU parity: every CUDA entry point against the CPU oracle.

Pack and permute must match bit-exactly; products must satisfy
|gpu - exact| <= tol * sum_k |w * x| per output, with tol = 2e-3 for bf16
inputs and 1e-5 for the fp32-input GEMV.  Inputs come from the seeded
generators in synth/, shaped like the pages' workloads, at full size and at
small sizes with ragged tails and degenerate cases.
"""
import numpy as np
import pytest
import torch

import oracle
import synth
from helpers import parity_violations
from synth import np_bits

pytestmark = pytest.mark.gpu

BF16_TOL = 2e-3
F32_TOL = 1e-5


@pytest.fixture(scope="module")
def w4():
    import gemm_int4_dequant_gb300 as m
    return m


def _dev():
    return torch.device("cuda:0")


def _guarded(n_elems, dtype, fill):
    """A contiguous view of n_elems with 64-byte guard bands on both sides."""
    esz = torch.tensor([], dtype=dtype).element_size()
    pad = 64 // esz
    buf = torch.full((n_elems + 2 * pad,), fill, dtype=dtype, device=_dev())
    return buf, buf[pad:pad + n_elems], pad


def _guards_intact(buf, pad, n_elems, fill):
    return bool(torch.all(buf[:pad] == fill)) and bool(torch.all(buf[pad + n_elems:] == fill))


# ---------------------------------------------------------------------------
# quantize_pack_int4 + permute_int4 (bit-exact)
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("K,N", [
    (2, 8), (128, 64), (130, 37), (64, 1), (1024, 1000), (8192, 8192),
    (1000, 64),      # rows per CTA not a whole number of TMA boxes
    (4098, 8),       # five CTAs per cluster, the last holding two rows
    (20000, 40),     # eight CTAs of 2560 rows; a strip past the last column
    (26624, 16),     # longest K of the single-read kernel
    (26626, 16),     # first K of the two-pass kernel
])
def test_quantize_pack_bit_exact(w4, K, N):
    W = synth.quant_inputs(K, N, seed=K + N)
    if N > 3:
        W[:, 3] = 0  # a column of zeros: scale 0, q 0
    buf, packed, pad = _guarded((K // 2) * N, torch.uint8, 0xA5)
    packed, scale = w4.quantize_pack_int4(W.to(_dev()), packed=packed)
    s_ref, p_ref = oracle.quantize_pack(np_bits(W))
    assert np.array_equal(scale.cpu().numpy().view(np.uint32), s_ref.view(np.uint32))
    assert np.array_equal(packed.cpu().numpy().reshape(K // 2, N), p_ref)
    assert _guards_intact(buf, pad, (K // 2) * N, 0xA5)


def test_quantize_pack_k_zero(w4):
    scale = torch.full((16,), 3.0, device=_dev())
    w4.quantize_pack_int4(torch.empty((0, 16), dtype=torch.bfloat16, device=_dev()), scale=scale)
    assert torch.all(scale == 0)


@pytest.mark.parametrize("K,N", [
    (64, 4), (128, 132), (1024, 4096), (8192, 8192),
    (64, 16),        # one chunk, two column groups: TMA tile mostly outside the matrix
    (192, 48),       # partial tile in both directions
    (4160, 1040),    # 65 chunks and 260 groups: ragged last tiles
])
def test_permute_bit_exact(w4, K, N):
    g = torch.Generator().manual_seed(K * 7 + N)
    packed = torch.randint(0, 256, (K // 2, N), dtype=torch.uint8, generator=g)
    buf, out, pad = _guarded(N * K // 2, torch.uint8, 0x5A)
    w4.permute_int4(packed.to(_dev()), out=out)
    ref = oracle.permute(packed.numpy(), K, N)
    assert np.array_equal(out.cpu().numpy(), ref)
    assert _guards_intact(buf, pad, N * K // 2, 0x5A)


@pytest.mark.parametrize("K,N", [
    (64, 8), (128, 64), (256, 40),   # one TMA box per CTA; a strip past the last column
    (8192, 8192),                    # the quantise+pack+permute workload
    (4160, 32),                      # five CTAs per cluster, the last holding 64 rows
    (20480, 24),                     # eight CTAs of 2560 rows, partial strip
    (26624, 16),                     # longest K accepted
    (1024, 4104),                    # many strips, N % 32 == 8
])
def test_quantize_pack_permute_bit_exact(w4, K, N):
    """The one-pass call equals permute(quantize_pack(W)) of the oracle."""
    W = synth.quant_inputs(K, N, seed=K + 3 * N)
    W[:, 3] = 0                                    # a column of zeros: scale 0, q 0
    if N > 5:
        # exact ties of W / s: column 5 holds multiples of max / 14 (k + 1/2 for odd multiples)
        m = float(W[:, 5].float().abs().max())
        ties = (torch.arange(K) % 15 - 7).float() * (m / 7.0) * 0.5
        W[:, 5] = ties.to(torch.bfloat16)
        W[0, 5] = m
    buf, out, pad = _guarded(N * K // 2, torch.uint8, 0x3C)
    sbuf, scale, spad = _guarded(N, torch.float32, -1.0)
    w4.quantize_pack_permute_int4(W.to(_dev()), out=out, scale=scale)
    s_ref, p_ref = oracle.quantize_pack(np_bits(W))
    assert np.array_equal(scale.cpu().numpy().view(np.uint32), s_ref.view(np.uint32))
    ref = oracle.permute(p_ref, K, N)
    got = out.cpu().numpy()
    if not np.array_equal(got, ref):
        bad = np.nonzero(got != ref)[0]
        raise AssertionError("%d bytes differ, first at %s" % (bad.size, bad[:8]))
    assert _guards_intact(buf, pad, N * K // 2, 0x3C)
    assert _guards_intact(sbuf, spad, N, -1.0)


def test_quantize_pack_permute_k_zero(w4):
    scale = torch.full((16,), 3.0, device=_dev())
    out = torch.full((8,), 7, dtype=torch.int8, device=_dev())
    w4.quantize_pack_permute_int4(torch.empty((0, 16), dtype=torch.bfloat16, device=_dev()), out=out[:0],
                                  scale=scale)
    assert torch.all(scale == 0)
    assert torch.all(out == 7)


def test_quantize_pack_permute_chain_full_size(w4):
    cfg = synth.QUANT
    W = synth.quant_inputs(cfg["K"], cfg["N"], seed=0)
    packed, scale = w4.quantize_pack_int4(W.to(_dev()))
    out = w4.permute_int4(packed)
    s_ref, p_ref = oracle.quantize_pack(np_bits(W))
    assert np.array_equal(scale.cpu().numpy(), s_ref)
    assert np.array_equal(np_bits(out.cpu()), oracle.permute(p_ref, cfg["K"], cfg["N"]))


# ---------------------------------------------------------------------------
# gemv_w4
# ---------------------------------------------------------------------------

def _check_gemv(w4, N, K, C, act, seed=0, **kw):
    g = synth.gemv_inputs(N, K, C, act=act, seed=seed, **kw)
    dt = torch.float32 if act == "f32" else torch.bfloat16
    buf, out, pad = _guarded(C * N, dt, -7.0)
    w4.gemv_w4(g.qweight.to(_dev()), g.scale.to(_dev()), g.zero.to(_dev()), g.x.to(_dev()), out=out)
    code = oracle.F32 if act == "f32" else oracle.BF16
    ref, ref_abs = oracle.gemv(np_bits(g.qweight), np_bits(g.scale), np_bits(g.zero), np_bits(g.x), code)
    got = out.float().cpu().numpy().astype(np.float64).reshape(C, N)
    tol = F32_TOL if act == "f32" else BF16_TOL
    bad = parity_violations(got, ref, ref_abs, tol, bf16_out=(act == "bf16"))
    err = np.abs(got - ref)
    assert not bad.any(), "max err/ref_abs = %g at %s" % ((err / ref_abs).max(), np.argwhere(bad)[:5])
    assert _guards_intact(buf, pad, C * N, -7.0)


def test_gemv_tiny_f32(w4):
    _check_gemv(w4, **synth.TINY)


def test_gemv_decode_full_size(w4):
    _check_gemv(w4, **synth.DECODE)


@pytest.mark.parametrize("cfg", synth.SMALL_BATCH, ids=lambda c: "N%dK%dC%d" % (c["N"], c["K"], c["C"]))
def test_gemv_small_batch_full_size(w4, cfg):
    _check_gemv(w4, **cfg)


@pytest.mark.parametrize("N,K,C,act", [
    (1, 8, 1, "bf16"),          # smallest legal problem
    (77, 520, 3, "bf16"),       # K % 32 != 0: single-word loads
    (130, 1000, 8, "f32"),      # K % 32 == 8
    (300, 4096, 2, "bf16"),
    (65, 2048, 5, "f32"),
    (63, 64, 6, "bf16"),        # fewer rows than one CTA tile
    (1000, 40000, 2, "bf16"),   # long K: split across a cluster
    (333, 24008, 7, "bf16"),    # long ragged K, cluster split, word loads
    (257, 12288, 8, "f32"),     # fp32 x split across a cluster
    (1, 256, 1, "bf16"),        # one row, one band
    (3, 288, 8, "bf16"),        # partial band (x zero-padded), rows < one lane quarter
    (40000, 512, 3, "bf16"),    # several row tiles per CTA
    (1001, 17312, 8, "bf16"),   # cluster split with a partial last band per slice
    (5, 40960, 8, "bf16"),      # longest K accepted
    (400000, 256, 1, "bf16"),   # more row tiles than one wave holds
    (1001, 4096, 3, "bf16"),    # tensor boxes running past the last row (zero-filled)
    (2000, 12800, 6, "bf16"),   # tensor boxes with a cluster split and a 12-row tile (three 4-row boxes)
    (4099, 384, 4, "bf16"),     # box of 3 chunks over a 3-chunk row, partial last tile
])
def test_gemv_ragged_and_edge(w4, N, K, C, act):
    _check_gemv(w4, N, K, C, act, seed=N + K + C)


@pytest.mark.parametrize("N,K", [
    (50, 5120),      # fewer 16-row tiles than SMs, a short last tile
    (1001, 4096),    # rows not a multiple of 16 or of the SM count
    (153, 128),      # one 128-k unit per stage
    (2000, 6144),    # 48 units per stage
    (777, 1152),     # nine units per stage
    (17296, 5120),   # the decode shape plus one tile
])
def test_gemv_one_column_shapes(w4, N, K):
    """One column of bf16 x (the fp16 tensor-core loop): fewer 16-row tiles
    than SMs, ragged row counts, a single 128-k unit, long and odd unit
    counts, and rows at the zero point (exactly 0)."""
    _check_gemv(w4, N, K, 1, "bf16", seed=N + K)
    g = synth.gemv_inputs(N, K, 1, act="bf16", seed=N + 2 * K, zero_value=8, zero_rows=7)
    got = w4.gemv_w4(g.qweight.to(_dev()), g.scale.to(_dev()), g.zero.to(_dev()), g.x.to(_dev()))
    assert torch.all(got.float()[0, ::7] == 0)


def test_gemv_non_integer_zero_and_wide_scales(w4):
    _check_gemv(w4, 500, 2048, 4, "bf16", seed=3, zero_value=7.3, scale_range=(0.5, 4.0))
    _check_gemv(w4, 500, 2048, 2, "f32", seed=4, zero_value=0.013, scale_range=(1e-3, 1.0))


@pytest.mark.parametrize("N,K", [(300, 4096), (200, 24576)])   # one CTA per row range; K split over a cluster
def test_gemv_x_magnitudes(w4, N, K):
    """x columns far outside fp16's range, tiny, spanning 2^40 within a
    column, and all zero: the tensor-core path scales each column of x by a
    power of two before its fp16 conversion."""
    C = 5
    g = synth.gemv_inputs(N, K, C, act="bf16", seed=11)
    x = g.x.float()
    x[0] *= 2.0 ** 40                      # beyond fp16's largest finite value
    x[1] *= 2.0 ** -60                     # below fp16's smallest subnormal
    span = torch.ones(K)
    span[::3] = 2.0 ** 20
    span[1::3] = 2.0 ** -20
    x[2] *= span                           # 2^40 between elements of one column
    x[3] = 0.0
    x[4, : K // 2] = 0.0                   # half zero
    g.x = x.to(torch.bfloat16)
    buf, out, pad = _guarded(C * N, torch.bfloat16, -7.0)
    w4.gemv_w4(g.qweight.to(_dev()), g.scale.to(_dev()), g.zero.to(_dev()), g.x.to(_dev()), out=out)
    ref, ref_abs = oracle.gemv(np_bits(g.qweight), np_bits(g.scale), np_bits(g.zero), np_bits(g.x), oracle.BF16)
    got = out.float().cpu().numpy().astype(np.float64).reshape(C, N)
    bad = parity_violations(got, ref, ref_abs, BF16_TOL, bf16_out=True)
    err = np.abs(got - ref)
    assert not bad.any(), "max err/ref_abs = %g at %s" % ((err / np.maximum(ref_abs, 1e-300)).max(),
                                                          np.argwhere(bad)[:5])
    assert np.all(got[3] == 0)
    assert _guards_intact(buf, pad, C * N, -7.0)


def test_gemv_k_zero_gives_zero(w4):
    x = torch.empty((2, 0), dtype=torch.bfloat16, device=_dev())
    q = torch.empty((16, 0), dtype=torch.int32, device=_dev())
    s = torch.ones(16, dtype=torch.bfloat16, device=_dev())
    out = torch.full((2, 16), 5.0, dtype=torch.bfloat16, device=_dev())
    w4.gemv_w4(q, s, s, x, out=out)
    assert torch.all(out == 0)


def test_gemv_through_raw_c_abi(w4):
    from gemm_int4_dequant_gb300 import _lib as L
    g = synth.gemv_inputs(96, 256, 2, act="bf16", seed=9)
    q, s, z, x = (t.to(_dev()) for t in (g.qweight, g.scale, g.zero, g.x))
    d = torch.empty((2, 96), dtype=torch.bfloat16, device=_dev())
    st = L.load().gemv_w4(q.data_ptr(), s.data_ptr(), z.data_ptr(), x.data_ptr(), d.data_ptr(), 96, 256, 2,
                          L.W4_BF16, torch.cuda.current_stream().cuda_stream)
    assert st == 0
    ref, ref_abs = oracle.gemv(np_bits(g.qweight), np_bits(g.scale), np_bits(g.zero), np_bits(g.x), oracle.BF16)
    assert not parity_violations(d.float().cpu().numpy(), ref, ref_abs, BF16_TOL, bf16_out=True).any()


# ---------------------------------------------------------------------------
# gemv_w4_permuted (permute_int4's output consumed directly)
# ---------------------------------------------------------------------------

def _check_gemv_permuted(w4, N, K, C, seed):
    g = synth.packed_gemv_inputs(N, K, C, seed=seed)
    perm = w4.permute_int4(g.packed.to(_dev()))
    buf, out, pad = _guarded(C * N, torch.bfloat16, -7.0)
    w4.gemv_w4_permuted(perm, g.scale.to(_dev()), g.x.to(_dev()), out=out)
    ref, ref_abs = oracle.gemv_packed(g.packed.numpy(), g.scale.numpy(), np_bits(g.x))
    got = out.float().cpu().numpy().astype(np.float64).reshape(C, N)
    bad = parity_violations(got, ref, ref_abs, BF16_TOL, bf16_out=True)
    err = np.abs(got - ref)
    assert not bad.any(), "max err/ref_abs = %g at %s" % ((err / ref_abs).max(), np.argwhere(bad)[:5])
    assert _guards_intact(buf, pad, C * N, -7.0)


@pytest.mark.parametrize("N,K,C", [
    (4, 64, 1),          # one column group, one line
    (12, 128, 3),        # three groups: a partial 16-column tile
    (100, 192, 8),       # 6 full tiles and a 4-column one; K % 128 == 64 (half unit)
    (1000, 512, 2),
    (4096, 4160, 5),     # a half unit at the end of every row
    (260, 40960, 8),     # x split over an eight-CTA cluster
    (17280, 5120, 1),    # decode shape
    (5120, 17280, 4),    # small-batch shapes of the pages' workloads
    (5120, 17280, 8),
    (6144, 5120, 4),
    (6144, 5120, 8),
])
def test_gemv_permuted(w4, N, K, C):
    _check_gemv_permuted(w4, N, K, C, seed=N + K + C)


def test_quantize_permute_gemv_chain(w4):
    """W -> quantize_pack_int4 -> permute_int4 -> gemv_w4_permuted against the
    oracle GEMV over the oracle's own quantised matrix."""
    K, N, C = 2048, 1024, 4
    W = synth.quant_inputs(K, N, seed=7)
    x = synth.packed_gemv_inputs(N, K, C, seed=8).x
    packed, scale = w4.quantize_pack_int4(W.to(_dev()))
    out = w4.gemv_w4_permuted(w4.permute_int4(packed), scale, x.to(_dev()))
    s_ref, p_ref = oracle.quantize_pack(np_bits(W))
    ref, ref_abs = oracle.gemv_packed(p_ref, s_ref, np_bits(x))
    got = out.float().cpu().numpy().astype(np.float64)
    assert not parity_violations(got, ref, ref_abs, BF16_TOL, bf16_out=True).any()
    assert w4.device_error() == 0


# ---------------------------------------------------------------------------
# gemm_w4
# ---------------------------------------------------------------------------

def _check_gemm_full(w4, M, N, K, seed=0, **kw):
    gi = synth.gemm_inputs(M, N, K, seed=seed, **kw)
    buf, out, pad = _guarded(M * N, torch.bfloat16, -3.0)
    w4.gemm_w4(gi.A.to(_dev()), gi.B.to(_dev()), gi.scale.to(_dev()), gi.zero.to(_dev()), out=out)
    ref, ref_abs = oracle.gemm_full(np_bits(gi.A), gi.B.numpy(), np_bits(gi.scale), np_bits(gi.zero))
    got = out.float().cpu().numpy().astype(np.float64).reshape(M, N)
    err = np.abs(got - ref)
    bad = parity_violations(got, ref, ref_abs, BF16_TOL, bf16_out=True)
    assert not bad.any(), "max err/ref_abs = %g at %s" % ((err / ref_abs).max(), np.argwhere(bad)[:5])
    assert _guards_intact(buf, pad, M * N, -3.0)
    assert w4.device_error() == 0


@pytest.mark.parametrize("M,N,K", [
    (128, 256, 64),     # one tile, one k-tile
    (256, 512, 256),
    (200, 272, 128),    # ragged M and N (N % 256 != 0)
    (1, 16, 64),        # degenerate
    (300, 1008, 1024),
    (129, 528, 512),
    (257, 256, 128),    # second 256-row tile holds one row; its odd CTA has no rows
    (384, 784, 192),    # ragged M tile pair and a last column tile of 16 columns
    (2048, 4096, 64),   # 256 tiles, one k-tile each: ring and accumulators wrap across tiles
    (1280, 2320, 192),  # several tiles per CTA pair with ragged last row and column tiles
])
def test_gemm_small(w4, M, N, K):
    _check_gemm_full(w4, M, N, K, seed=M + N + K)


def test_gemm_non_integer_zero_random_scale(w4):
    _check_gemm_full(w4, 256, 512, 512, seed=11, zero_value=7.5, random_scale=True)
    _check_gemm_full(w4, 256, 256, 256, seed=12, zero_value=0.013, random_scale=True)


def test_gemm_full_size_sampled(w4):
    cfg = synth.GEMM
    M, N, K = cfg["M"], cfg["N"], cfg["K"]
    gi = synth.gemm_inputs(M, N, K, seed=0)
    C = w4.gemm_w4(gi.A.to(_dev()), gi.B.to(_dev()), gi.scale.to(_dev()), gi.zero.to(_dev()))
    assert w4.device_error() == 0
    Cn = C.float().cpu().numpy().astype(np.float64)
    rng = np.random.default_rng(0)
    mi = list(rng.integers(0, M, 65536))
    ni = list(rng.integers(0, N, 65536))
    # full rows and columns at tile edges
    for m in (0, 127, 128, M - 1):
        mi += [m] * N
        ni += list(range(N))
    for n in (0, 255, 256, N - 1):
        mi += list(range(M))
        ni += [n] * M
    mi, ni = np.array(mi), np.array(ni)
    ref, ref_abs = oracle.gemm_at(np_bits(gi.A), gi.B.numpy(), np_bits(gi.scale), np_bits(gi.zero), mi, ni)
    err = np.abs(Cn[mi, ni] - ref)
    bad = parity_violations(Cn[mi, ni], ref, ref_abs, BF16_TOL, bf16_out=True)
    assert not bad.any(), "max err/ref_abs %g" % (err / ref_abs).max()


def test_gemm_k_zero(w4):
    A = torch.empty((4, 0), dtype=torch.bfloat16, device=_dev())
    B = torch.empty((0, 16), dtype=torch.uint8, device=_dev())
    s = torch.ones(16, dtype=torch.bfloat16, device=_dev())
    out = torch.full((4, 16), 2.0, dtype=torch.bfloat16, device=_dev())
    w4.gemm_w4(A, B, s, s, out=out)
    assert torch.all(out == 0)


# ---------------------------------------------------------------------------
# int8 weight-only variant: quantize_int8, permute_int8 (bit-exact), gemv_w8
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("K,N", [
    (64, 2), (130, 37),                       # N % 8 != 0: the two-pass kernel
    (1, 8), (7, 120),                         # single-read clusters: ranks without rows; a partial strip
    (1024, 1000), (8192, 8192), (26624, 72),  # ... up to the longest K a cluster holds
    (26626, 16),                              # one step past it: the two-pass kernel again
])
def test_quantize_int8_bit_exact(w4, K, N):
    W = synth.quant_inputs(K, N, seed=K + 5 * N)
    if N > 3:
        W[:, 3] = 0                                  # a column of zeros: scale 0, q 0
    if N > 5 and K > 1:
        # exact ties of W / s: half steps of a column whose max is 127/128 (scale 2^-7)
        t = (torch.arange(K) % 253 - 126).float() + 0.5
        W[:, 5] = (t * 2.0 ** -7).to(torch.bfloat16)
        W[0, 5] = 127 * 2.0 ** -7
    buf, q, pad = _guarded(K * N, torch.int8, 91)
    q, scale = w4.quantize_int8(W.to(_dev()), q=q)
    s_ref, q_ref = oracle.quantize_int8(np_bits(W))
    assert np.array_equal(scale.cpu().numpy().view(np.uint32), s_ref.view(np.uint32))
    assert np.array_equal(q.cpu().numpy().reshape(K, N), q_ref)
    assert _guards_intact(buf, pad, K * N, 91)


@pytest.mark.parametrize("K,N", [
    (64, 2), (128, 6), (1024, 1000), (4160, 1042),   # N % 16 != 0: one thread per line
    (64, 16), (4160, 1040), (1024, 4096),            # tiles of 64 x 128 (a partial last tile)
])
def test_permute_int8_bit_exact(w4, K, N):
    g = torch.Generator().manual_seed(K * 3 + N)
    q = torch.randint(-128, 128, (K, N), dtype=torch.int16, generator=g).to(torch.int8)
    buf, out, pad = _guarded(N * K, torch.uint8, 0x5A)
    w4.permute_int8(q.view(torch.uint8).to(_dev()), out=out)
    assert np.array_equal(out.cpu().numpy(), oracle.permute_int8(q.numpy(), K, N))
    assert _guards_intact(buf, pad, N * K, 0x5A)


@pytest.mark.parametrize("N,K,C", [
    (1, 1, 1), (37, 100, 3), (300, 4096, 8), (1000, 5120, 1),     # N % 16 != 0: the plain kernel
    (17280, 5120, 1), (5120, 17280, 4), (5120, 17280, 8),          # N % 16 == 0: 128-column strips, K split
    (6144, 5120, 2), (16, 7, 3),                                   # a cluster rank with no rows of K
    (272, 100, 5), (48, 8192, 6),                                  # a partial strip; eight columns a thread
])
def test_gemv_w8(w4, N, K, C):
    gi = synth.int8_gemv_inputs(N, K, C, seed=N + K + C)
    buf, out, pad = _guarded(C * N, torch.bfloat16, -7.0)
    w4.gemv_w8(gi.q.to(_dev()), gi.scale.to(_dev()), gi.x.to(_dev()), out=out)
    ref, ref_abs = oracle.gemv_int8(gi.q.numpy(), gi.scale.numpy(), np_bits(gi.x))
    got = out.float().cpu().numpy().astype(np.float64).reshape(C, N)
    bad = parity_violations(got, ref, ref_abs, BF16_TOL, bf16_out=True)
    assert not bad.any(), "max err/ref_abs = %g" % (np.abs(got - ref) / np.maximum(ref_abs, 1e-300)).max()
    assert _guards_intact(buf, pad, C * N, -7.0)


def test_int8_quantise_permute_gemv_chain(w4):
    """quantize_int8 -> permute_int8 and quantize_int8 -> gemv_w8 on one
    weight, each against the oracle applied to the oracle's quantisation."""
    K, N, C = 1024, 512, 2
    W = synth.quant_inputs(K, N, seed=21)
    x = synth.int8_gemv_inputs(N, K, C, seed=22).x
    q, scale = w4.quantize_int8(W.to(_dev()))
    s_ref, q_ref = oracle.quantize_int8(np_bits(W))
    perm = w4.permute_int8(q)
    assert np.array_equal(perm.cpu().numpy().view(np.uint8), oracle.permute_int8(q_ref, K, N))
    d = w4.gemv_w8(q, scale, x.to(_dev()))
    ref, ref_abs = oracle.gemv_int8(q_ref, s_ref, np_bits(x))
    assert not parity_violations(d.float().cpu().numpy(), ref, ref_abs, BF16_TOL, bf16_out=True).any()


# ---------------------------------------------------------------------------
# gemm_w8: bf16 x int8 on the tensor cores
# ---------------------------------------------------------------------------

def _w8_gemm_case(M, N, K, seed):
    gi = synth.int8_gemv_inputs(N, K, 1, seed=seed)
    A = synth.gemm_inputs(M, 16, K, seed=seed + 1).A
    return A, gi.q, gi.scale


@pytest.mark.parametrize("M,N,K", [(256, 256, 64), (300, 528, 192), (1, 16, 64), (777, 1040, 640), (512, 1024, 1024)])
def test_gemm_w8_small(w4, M, N, K):
    A, q, s = _w8_gemm_case(M, N, K, seed=M + N + K)
    buf, out, pad = _guarded(M * N, torch.bfloat16, -3.0)
    w4.gemm_w8(A.to(_dev()), q.to(_dev()), s.to(_dev()), out=out.view(M, N))
    assert w4.device_error() == 0
    ref, ref_abs = oracle.gemm_int8_full(np_bits(A), q.numpy(), s.numpy())
    got = out.float().cpu().numpy().astype(np.float64).reshape(M, N)
    bad = parity_violations(got, ref, ref_abs, BF16_TOL, bf16_out=True)
    assert not bad.any(), "max err/ref_abs %g" % (np.abs(got - ref) / ref_abs).max()
    assert _guards_intact(buf, pad, M * N, -3.0)


def test_gemm_w8_full_size_sampled(w4):
    M = N = K = 8192
    A, q, s = _w8_gemm_case(M, N, K, seed=3)
    C = w4.gemm_w8(A.to(_dev()), q.to(_dev()), s.to(_dev()))
    assert w4.device_error() == 0
    Cn = C.float().cpu().numpy().astype(np.float64)
    rng = np.random.default_rng(1)
    mi = list(rng.integers(0, M, 32768))
    ni = list(rng.integers(0, N, 32768))
    for m in (0, 127, 128, M - 1):
        mi += [m] * 1024
        ni += list(rng.integers(0, N, 1024))
    for n in (0, 255, 256, N - 1):
        mi += list(rng.integers(0, M, 1024))
        ni += [n] * 1024
    mi, ni = np.array(mi), np.array(ni)
    ref, ref_abs = oracle.gemm_int8_at(np_bits(A), q.numpy(), s.numpy(), mi, ni)
    bad = parity_violations(Cn[mi, ni], ref, ref_abs, BF16_TOL, bf16_out=True)
    assert not bad.any()


def test_quantize_int8_then_gemm_w8(w4):
    """quantize_int8 on the device, then gemm_w8, against the oracle's
    quantisation and product."""
    K, N, M = 1024, 512, 384
    W = synth.quant_inputs(K, N, seed=31)
    A = synth.gemm_inputs(M, 16, K, seed=32).A
    q, scale = w4.quantize_int8(W.to(_dev()))
    C = w4.gemm_w8(A.to(_dev()), q, scale)
    s_ref, q_ref = oracle.quantize_int8(np_bits(W))
    ref, ref_abs = oracle.gemm_int8_full(np_bits(A), q_ref, s_ref)
    assert not parity_violations(C.float().cpu().numpy(), ref, ref_abs, BF16_TOL, bf16_out=True).any()


# ---------------------------------------------------------------------------
# gemm_w4_permuted: the GEMM reading permute_int4's layout
# ---------------------------------------------------------------------------

def _perm_gemm_case(M, N, K, seed):
    g = synth.packed_gemv_inputs(N, K, 1, seed=seed)
    A = synth.gemm_inputs(M, 16, K, seed=seed + 1).A
    permuted = oracle.permute(g.packed.numpy(), K, N)
    return A, g.packed.numpy(), permuted, g.scale


@pytest.mark.parametrize("M,N,K", [(256, 256, 64), (300, 528, 192), (1, 16, 64), (777, 1040, 640), (512, 1024, 1024)])
def test_gemm_w4_permuted_small(w4, M, N, K):
    A, packed, permuted, s = _perm_gemm_case(M, N, K, seed=M + N + K)
    buf, out, pad = _guarded(M * N, torch.bfloat16, -3.0)
    w4.gemm_w4_permuted(A.to(_dev()), torch.from_numpy(permuted).to(_dev()), s.to(_dev()), out=out.view(M, N))
    assert w4.device_error() == 0
    ref, ref_abs = oracle.gemm_packed_full(np_bits(A), packed, s.numpy())
    got = out.float().cpu().numpy().astype(np.float64).reshape(M, N)
    bad = parity_violations(got, ref, ref_abs, BF16_TOL, bf16_out=True)
    assert not bad.any(), "max err/ref_abs %g" % (np.abs(got - ref) / ref_abs).max()
    assert _guards_intact(buf, pad, M * N, -3.0)


def test_gemm_w4_permuted_full_size_sampled(w4):
    M = N = K = 8192
    A, packed, permuted, s = _perm_gemm_case(M, N, K, seed=5)
    C = w4.gemm_w4_permuted(A.to(_dev()), torch.from_numpy(permuted).to(_dev()), s.to(_dev()))
    assert w4.device_error() == 0
    Cn = C.float().cpu().numpy().astype(np.float64)
    rng = np.random.default_rng(2)
    mi = list(rng.integers(0, M, 32768))
    ni = list(rng.integers(0, N, 32768))
    for n in (0, 3, 4, 127, 128, 255, 256, N - 1):      # group and tile edges
        mi += list(rng.integers(0, M, 512))
        ni += [n] * 512
    mi, ni = np.array(mi), np.array(ni)
    ref, ref_abs = oracle.gemm_packed_at(np_bits(A), packed, s.numpy(), mi, ni)
    assert not parity_violations(Cn[mi, ni], ref, ref_abs, BF16_TOL, bf16_out=True).any()


def test_quantise_permute_then_gemm(w4):
    """quantize_pack_permute_int4 on the device, then gemm_w4_permuted,
    against the oracle's quantisation and product."""
    K, N, M = 1024, 512, 384
    W = synth.quant_inputs(K, N, seed=41)
    A = synth.gemm_inputs(M, 16, K, seed=42).A
    permuted, scale = w4.quantize_pack_permute_int4(W.to(_dev()))
    C = w4.gemm_w4_permuted(A.to(_dev()), permuted, scale)
    s_ref, p_ref = oracle.quantize_pack(np_bits(W))
    ref, ref_abs = oracle.gemm_packed_full(np_bits(A), p_ref, s_ref)
    assert not parity_violations(C.float().cpu().numpy(), ref, ref_abs, BF16_TOL, bf16_out=True).any()



# ---------------------------------------------------------------------------
# the device error path
# ---------------------------------------------------------------------------

def test_bounded_wait_gives_up_reports_and_leaves_the_context_usable(w4):
    """A wait on a barrier nothing completes ends after its limit with error
    code 1 (read and cleared by w4_device_error); the next calls work."""
    from gemm_int4_dequant_gb300 import _lib as L
    waited = torch.full((1,), 7, dtype=torch.int32, device=_dev())
    assert w4.device_error() == 0
    st = L.load().w4_selftest_wait_timeout(waited.data_ptr(), torch.cuda.current_stream().cuda_stream)
    assert st == L.W4_OK
    assert w4.device_error() == 1
    assert int(waited.item()) == 0
    assert w4.device_error() == 0
    _check_gemv(w4, 300, 4096, 2, "bf16", seed=9)


def _selftest_configure(limit_clocks, short_first_stage):
    from gemm_int4_dequant_gb300 import _lib as L
    assert L.load().w4_selftest_configure(limit_clocks, short_first_stage) == L.W4_OK


# about 2 ms of SM clock: every wait that cannot complete gives up quickly
_SHORT_LIMIT = 1 << 22


@pytest.mark.parametrize("N,K,C", [(1000, 5120, 1), (700, 4096, 4)])
def test_gemv_stage_that_never_completes_runs_out_and_recovers(w4, N, K, C):
    """The producer announces 16 bytes more than it copies for its first
    stage (a test switch), so that stage's wait runs out its shortened
    limit: the kernel records code 1, stops issuing, drains and returns with
    the guard bands around its output intact; with the switch off again the
    next call is within the bound and records nothing."""
    g = synth.gemv_inputs(N, K, C, act="bf16", seed=21)
    assert w4.device_error() == 0
    buf, out, pad = _guarded(C * N, torch.bfloat16, -7.0)
    try:
        _selftest_configure(_SHORT_LIMIT, 1)
        w4.gemv_w4(g.qweight.to(_dev()), g.scale.to(_dev()), g.zero.to(_dev()), g.x.to(_dev()), out=out)
        assert w4.device_error() == 1
    finally:
        _selftest_configure(0, 0)
    assert _guards_intact(buf, pad, C * N, -7.0)
    assert w4.device_error() == 0
    _check_gemv(w4, N, K, C, "bf16", seed=22)
    assert w4.device_error() == 0


def test_gemv_permuted_stage_that_never_completes_runs_out_and_recovers(w4):
    N, K, C = 512, 5120, 4
    g = synth.packed_gemv_inputs(N, K, C, seed=23)
    perm = w4.permute_int4(g.packed.to(_dev()))
    assert w4.device_error() == 0
    buf, out, pad = _guarded(C * N, torch.bfloat16, -7.0)
    try:
        _selftest_configure(_SHORT_LIMIT, 1)
        w4.gemv_w4_permuted(perm, g.scale.to(_dev()), g.x.to(_dev()), out=out)
        assert w4.device_error() == 1
    finally:
        _selftest_configure(0, 0)
    assert _guards_intact(buf, pad, C * N, -7.0)
    assert w4.device_error() == 0
    _check_gemv_permuted(w4, N, K, C, seed=24)
    assert w4.device_error() == 0


def test_gemm_stage_that_never_completes_runs_out_frees_tmem_and_recovers(w4):
    """The same switch on the tensor-memory GEMM: every role of both CTAs
    of a pair gives up, the pair frees its tensor memory (a later launch
    allocates it again) and the next call is exact."""
    M, N, K = 256, 512, 256
    gi = synth.gemm_inputs(M, N, K, seed=25)
    assert w4.device_error() == 0
    buf, out, pad = _guarded(M * N, torch.bfloat16, -3.0)
    try:
        _selftest_configure(_SHORT_LIMIT, 1)
        w4.gemm_w4(gi.A.to(_dev()), gi.B.to(_dev()), gi.scale.to(_dev()), gi.zero.to(_dev()), out=out)
        assert w4.device_error() == 1
    finally:
        _selftest_configure(0, 0)
    assert _guards_intact(buf, pad, M * N, -3.0)
    assert w4.device_error() == 0
    _check_gemm_full(w4, M, N, K, seed=26)
    _check_gemm_full(w4, 2048, 4096, 64, seed=27)   # a multi-tile launch after the aborted one
