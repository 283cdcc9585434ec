"""Exhaustive parity of the quantiser's rounding on the GPU.

The quantiser (page "[PHI] add int4 weight only quant kernel, add int4 weight
only permute kernel", section "int4量化kernel"; symmetric per-column scale
s = max|W| / 7, q = clamp(round(W / s), -8, 7), round half away from zero,
IEEE fp32 division) must agree bit for bit with the oracle on every bf16
weight it can meet.  For each column maximum below, the columns of W hold
every finite bf16 value v with |v| <= max (both signs, zeros and subnormals
included), each column also holding the maximum itself so that its scale
is the same; every weight therefore reaches the kernels' rounding once
with that scale, ties and near-ties included.  The columns run through
the single-read cluster kernel (N % 8 == 0, K <= 26624), the two-pass
kernel (N % 8 != 0) and the one-pass quantise + permute, against the
oracle's quantise + pack and permute.
"""
import numpy as np
import pytest
import torch

import oracle
from synth import np_bits

pytestmark = pytest.mark.gpu

K = 26624          # longest K of the single-read kernel


def _bf16_from_bits(bits):
    return torch.from_numpy(np.ascontiguousarray(bits, dtype=np.uint16).view(np.int16)).view(torch.bfloat16)


def _all_finite_bf16():
    """Every finite bf16 value, as (bit patterns, float64 values)."""
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    finite = ((bits >> 7) & 0xFF) != 0xFF
    bits = bits[finite]
    vals = _bf16_from_bits(bits).double().numpy()
    return bits, vals


# column maxima: typical (N(0, 0.02) weights), powers of two, scales that
# make exact halves common (7: s = 1; 3.5: s = 0.5), an odd mantissa, the
# smallest normal and a subnormal maximum (fp32 scale subnormal), large
# and near the top of bf16's range
MAXIMA = [0.02, 0.0625, 1.0, 7.0, 3.5, 1.2265625, 2.0 ** -126, 2.0 ** -130, 2.0 ** 100, 3.3895313892515355e38]


def _columns():
    bits, vals = _all_finite_bf16()
    cols = []
    for m in MAXIMA:
        mb = np_bits(torch.tensor([m], dtype=torch.bfloat16))[0]
        mv = _bf16_from_bits(np.array([mb])).double().item()
        sel = bits[np.abs(vals) <= mv]
        per = K - 1
        for j in range(0, sel.size, per):
            col = np.zeros(K, dtype=np.uint16)      # +0 pads the last column of a maximum
            chunk = sel[j:j + per]
            col[:chunk.size] = chunk
            col[K - 1] = mb                         # the column's maximum, exactly max
            cols.append(col)
    cols.append(np.zeros(K, dtype=np.uint16))       # an all-zero column: scale 0, q 0
    return cols


@pytest.fixture(scope="module")
def weights():
    cols = _columns()
    n = (len(cols) + 7) // 8 * 8
    W = np.zeros((K, n), dtype=np.uint16)
    for j, c in enumerate(cols):
        W[:, j] = c
    return W


@pytest.fixture(scope="module")
def w4():
    import gemm_int4_dequant_gb300 as m
    return m


def _check_quant(w4, Wbits):
    W = _bf16_from_bits(Wbits)
    packed, scale = w4.quantize_pack_int4(W.to("cuda"))
    s_ref, p_ref = oracle.quantize_pack(Wbits)
    got_s = scale.cpu().numpy()
    assert np.array_equal(got_s.view(np.uint32), s_ref.view(np.uint32)), np.flatnonzero(
        got_s.view(np.uint32) != s_ref.view(np.uint32))[:8]
    got = np_bits(packed.cpu()).reshape(p_ref.shape)
    bad = np.argwhere(got != p_ref)
    assert bad.size == 0, "%d bytes differ, first (row pair, column) %s" % (len(bad), bad[:6].tolist())
    return s_ref, p_ref


def test_every_bf16_weight_single_read_kernel(w4, weights):
    assert weights.shape[1] % 8 == 0
    _check_quant(w4, weights)


def test_every_bf16_weight_two_pass_kernel(w4, weights):
    W = np.concatenate([weights, np.zeros((K, 1), dtype=np.uint16)], axis=1)   # N % 8 != 0
    _check_quant(w4, W)


def test_every_bf16_weight_quantise_and_permute_in_one_pass(w4, weights):
    n = weights.shape[1]
    out, scale = w4.quantize_pack_permute_int4(_bf16_from_bits(weights).to("cuda"))
    s_ref, p_ref = oracle.quantize_pack(weights)
    assert np.array_equal(scale.cpu().numpy().view(np.uint32), s_ref.view(np.uint32))
    ref = oracle.permute(p_ref, K, n)
    got = np_bits(out.cpu())
    bad = np.flatnonzero(got != ref)
    assert bad.size == 0, "%d bytes differ, first at %s" % (bad.size, bad[:8])


# int8 variant (the int4 definition with the int8 range: s = max|W| / 127,
# q = clamp(round(W / s), -128, 127)); columns of 12800 rows stay within the
# single-read kernel's K limit (26624)
K8 = 12800


def _int8_weights():
    bits, vals = _all_finite_bf16()
    cols = []
    for m in MAXIMA:
        mb = np_bits(torch.tensor([m], dtype=torch.bfloat16))[0]
        mv = _bf16_from_bits(np.array([mb])).double().item()
        sel = bits[np.abs(vals) <= mv]
        for j in range(0, sel.size, K8 - 1):
            col = np.zeros(K8, dtype=np.uint16)
            chunk = sel[j:j + K8 - 1]
            col[:chunk.size] = chunk
            col[K8 - 1] = mb
            cols.append(col)
    n = (len(cols) + 7) // 8 * 8
    W = np.zeros((K8, n), dtype=np.uint16)
    for j, c in enumerate(cols):
        W[:, j] = c
    return W


@pytest.mark.parametrize("extra_col", [False, True], ids=["single_read", "plain"])
def test_every_bf16_weight_int8(w4, extra_col):
    W = _int8_weights()
    if extra_col:   # N % 8 != 0: the plain kernel
        W = np.concatenate([W, np.zeros((K8, 1), dtype=np.uint16)], axis=1)
    q, scale = w4.quantize_int8(_bf16_from_bits(W).to("cuda"))
    s_ref, q_ref = oracle.quantize_int8(W)
    assert np.array_equal(scale.cpu().numpy().view(np.uint32), s_ref.view(np.uint32))
    got = q.cpu().numpy()
    bad = np.argwhere(got != q_ref)
    assert bad.size == 0, "%d weights differ, first (row, column) %s" % (len(bad), bad[:6].tolist())
