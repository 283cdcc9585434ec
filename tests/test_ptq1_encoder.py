"""The library's host-side PTQ1_0 -> PTQ1_1 conversion (no GPU): bit-exact
with the oracle's encoder -- superblocks, codebook and escape table -- on
tensors with and without escapes, padded last superblocks and the pages'
K values, and its rejection of inputs the format cannot hold."""
import ctypes

import numpy as np
import pytest

import oracle
import synth
from synth import np_bits


@pytest.fixture(scope="module")
def w4():
    import __graft_entry__
    __graft_entry__._load_builder().build_library()
    import gemm_int4_dequant_gb300 as m
    return m


def _blocks(N, K, seed, outliers=0.0):
    ti = synth.ternary_inputs(N, K, 1, seed=seed, outlier_fraction=outliers)
    return oracle.ptq1_0_pack(ti.trits.numpy(), np_bits(ti.d))


@pytest.mark.parametrize("N,K,outliers", [
    (300, 1152, 0.9),     # nine blocks a row: a padded last superblock
    (2048, 1024, 0.5),    # a full codebook, free-trit indices and escapes
    (64, 17280, 0.1), (40, 5120, 0.0), (12, 6144, 1.0),
    (0, 1024, 0.0),       # no rows
])
def test_encoder_matches_oracle(w4, N, K, outliers):
    blocks = _blocks(N, K, N + K, outliers)
    ref = oracle.ptq1_1_encode(blocks)
    sb, code, ei, ep = w4.ptq1_1_encode(blocks)
    assert np.array_equal(sb, ref.sblocks)
    assert np.array_equal(code, ref.codebook)
    assert np.array_equal(ei, ref.esc_idx) and np.array_equal(ep, ref.esc_patt)
    if N:
        t, d = oracle.ptq1_0_unpack(blocks)
        t2, d2 = oracle.ptq1_1_unpack(oracle.Ptq1_1(sb, code, ei, ep, K))
        assert np.array_equal(t, t2) and np.array_equal(d, d2)


def test_encoder_escapes_when_the_codebook_is_full(w4):
    blocks = _blocks(2048, 1024, 7, outliers=0.5)
    sb, code, ei, ep = w4.ptq1_1_encode(blocks)
    assert code.shape == (767, 8) and len(ei) > 0
    assert np.all(np.diff(ei) > 0)
    idx = sb[:, 0, 215].astype(int) + 256 * ((sb[:, 0, 204].astype(int) // 81) % 3)
    assert np.array_equal(np.nonzero(idx == 767)[0], ei)


@pytest.mark.parametrize("corrupt", ["negative_d", "qs_byte", "qh_field"])
def test_encoder_rejects_values_the_format_cannot_hold(w4, corrupt):
    blocks = _blocks(4, 1024, 9).copy()
    if corrupt == "negative_d":
        blocks[2, 3, 27] |= 0x80
    elif corrupt == "qs_byte":
        blocks[1, 5, 7] = 243
    else:
        blocks[0, 0, 25] |= 0xC0          # field 7 = 3
    with pytest.raises(w4.W4Error) as e:
        w4.ptq1_1_encode(blocks)
    assert e.value.status == -7


def test_encoder_shape_and_capacity_errors(w4):
    from gemm_int4_dequant_gb300 import _lib as L
    lib = L.load()
    blocks = _blocks(64, 1024, 10, outliers=1.0)       # every superblock its own pattern
    ptr = lambda a: a.ctypes.data_as(ctypes.c_void_p)
    code = np.zeros((767, 8), np.uint8)
    n = ctypes.c_int64(-1)
    assert lib.ptq1_1_codebook(ptr(blocks), 64, 1000, ptr(code), ctypes.byref(n)) == L.W4_ERR_SHAPE
    assert lib.ptq1_1_codebook(None, 64, 1024, ptr(code), ctypes.byref(n)) == L.W4_ERR_NULL
    sb = np.zeros((64, 1, 216), np.uint8)
    ei = np.zeros(4, np.int64)
    ep = np.zeros((4, 8), np.uint8)
    # an empty codebook sends all 64 superblocks to an escape table of 4
    assert lib.ptq1_1_encode(ptr(blocks), 64, 1024, None, 0, ptr(sb), ptr(ei), ptr(ep), 4,
                             ctypes.byref(n)) == L.W4_ERR_SHAPE
    assert lib.ptq1_1_encode(ptr(blocks), 64, 1024, ptr(code), 768, ptr(sb), ptr(ei), ptr(ep), 4,
                             ctypes.byref(n)) == L.W4_ERR_SHAPE
    ei64 = np.zeros(64, np.int64)
    ep64 = np.zeros((64, 8), np.uint8)
    assert lib.ptq1_1_encode(ptr(blocks), 64, 1024, None, 0, ptr(sb), ptr(ei64), ptr(ep64), 64,
                             ctypes.byref(n)) == L.W4_OK
    assert n.value == 64 and np.array_equal(ei64, np.arange(64))
