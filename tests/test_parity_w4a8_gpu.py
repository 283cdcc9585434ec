"""GPU parity of the W4A8 path: quantize_q8_1_pt bit-exact against the
oracle's block_q8_1 / PT quantiser, and gemv_w4a8 within
2e-3 * sum_k |(q - zero) scale d_b qs| (plus the bf16 rounding) of the
oracle's fp64 product, on the pages' Qwen shapes and small ragged ones."""
import numpy as np
import pytest
import torch

import oracle
import synth
from helpers import bf16_bits, parity_violations
from synth import np_bits

pytestmark = pytest.mark.gpu

BF16_TOL = 2e-3


@pytest.fixture(scope="module")
def w4():
    import gemm_int4_dequant_gb300 as m
    return m


def _dev():
    return torch.device("cuda:0")


def _guarded(n_elems, dtype, fill):
    esz = torch.tensor([], dtype=dtype).element_size()
    pad = 64 // esz
    buf = torch.full((n_elems + 2 * pad,), fill, dtype=dtype, device=_dev())
    return buf, buf[pad:pad + n_elems], pad


def _guards_intact(buf, pad, n_elems, fill):
    return bool(torch.all(buf[:pad] == fill)) and bool(torch.all(buf[pad + n_elems:] == fill))


def _special_x(C, K, seed):
    """N(0,1) activations with an all-zero q8_1 block, a block of exact
    half-step ties (x / d = k + 1/2 with d = 1) and a block of tiny values."""
    x = synth.gemv_inputs(1, K, C, act="bf16", seed=seed).x.float().numpy()
    x[0, 0:32] = 0.0
    if K >= 128:
        x[0, 32:64] = np.arange(32) - 15.5
        x[0, 32] = 127.0
        x[0, 64:96] = 1e-6 * (np.arange(32) - 16)
    return torch.from_numpy(bf16_bits(x).view(np.int16)).view(torch.bfloat16)


@pytest.mark.parametrize("C,K", [(1, 128), (1, 5120), (3, 1152), (2, 6144), (8, 17280), (4, 17280)])
def test_quantize_q8_1_pt_bit_exact(w4, C, K):
    x = _special_x(C, K, seed=C * K)
    n = C * 144 * (K // 128)
    buf, out, pad = _guarded(n, torch.uint8, 0xA5)
    w4.quantize_q8_1_pt(x.to(_dev()), out=out)
    ref = oracle.quantize_q8_1_pt(np_bits(x))
    assert np.array_equal(out.cpu().numpy().reshape(C, -1), ref)
    assert _guards_intact(buf, pad, n, 0xA5)


def test_quantize_q8_1_pt_k_zero_is_a_no_op(w4):
    out = torch.full((16,), 7, dtype=torch.uint8, device=_dev())
    w4.quantize_q8_1_pt(torch.empty((2, 0), dtype=torch.bfloat16, device=_dev()), out=out[:0])
    assert torch.all(out == 7)


@pytest.mark.parametrize("N,K,C", [
    (1, 128, 1), (17, 256, 2), (1000, 1152, 3),
    (17280, 5120, 1),     # decode shape
    (6144, 5120, 8), (5120, 17280, 4), (5120, 17280, 8),
    (37, 23168, 8),       # the largest K whose x fits shared memory at C = 8
    (40000, 1024, 4),     # one warp per row group (partial sums by shuffles)
    (200000, 256, 2),     # more groups in a CTA than half its threads: one thread per group
    (700000, 128, 1),     # more groups in a CTA than threads: threads take several groups
])
def test_gemv_w4a8(w4, N, K, C):
    g = synth.gemv_inputs(N, K, C, act="bf16", seed=N + K + C)
    pt = oracle.quantize_q8_1_pt(np_bits(g.x))
    buf, out, pad = _guarded(C * N, torch.bfloat16, -7.0)
    w4.gemv_w4a8(g.qweight.to(_dev()), g.scale.to(_dev()), g.zero.to(_dev()), torch.from_numpy(pt).to(_dev()),
                 out=out)
    ref, ref_abs = oracle.gemv_w4a8(np_bits(g.qweight), np_bits(g.scale), np_bits(g.zero), pt, K)
    got = out.float().cpu().numpy().astype(np.float64).reshape(C, N)
    bad = parity_violations(got, ref, ref_abs, BF16_TOL, bf16_out=True)
    assert not bad.any(), "max err/ref_abs = %g" % (np.abs(got - ref) / np.maximum(ref_abs, 1e-300)).max()
    assert _guards_intact(buf, pad, C * N, -7.0)


def test_w4a8_chain_quantise_then_gemv(w4):
    """quantize_q8_1_pt -> gemv_w4a8 on the device, against the oracle's
    quantiser and product."""
    N, K, C = 2048, 5120, 2
    g = synth.gemv_inputs(N, K, C, act="bf16", seed=41)
    pt = w4.quantize_q8_1_pt(g.x.to(_dev()))
    d = w4.gemv_w4a8(g.qweight.to(_dev()), g.scale.to(_dev()), g.zero.to(_dev()), pt)
    pt_ref = oracle.quantize_q8_1_pt(np_bits(g.x))
    assert np.array_equal(pt.cpu().numpy(), pt_ref)
    ref, ref_abs = oracle.gemv_w4a8(np_bits(g.qweight), np_bits(g.scale), np_bits(g.zero), pt_ref, K)
    assert not parity_violations(d.float().cpu().numpy(), ref, ref_abs, BF16_TOL, bf16_out=True).any()


def test_gemv_w4a8_k_zero_gives_zero(w4):
    d = torch.full((2, 16), 3.0, dtype=torch.bfloat16, device=_dev())
    w4.gemv_w4a8(torch.empty((16, 0), dtype=torch.int32, device=_dev()),
                 torch.ones(16, dtype=torch.bfloat16, device=_dev()), torch.ones(16, dtype=torch.bfloat16, device=_dev()),
                 torch.empty((2, 0), dtype=torch.uint8, device=_dev()), out=d)
    assert torch.all(d == 0)
