"""GPU parity of the ternary MMVQ: mmvq_ptq1_0 against the oracle's fp64
product on PTQ1_0 blocks the oracle packed, with x as block_q8_1 / PT.

The integer dots are exact on both sides; the kernel's products and sums
are fp32, so each output is within (K/128 + 5) * 2^-24 of sum_k |w x|
(8.3e-6 at K = 17280); the test uses 2e-5."""
import numpy as np
import pytest
import torch

import oracle
import synth
from synth import np_bits

pytestmark = pytest.mark.gpu

TOL = 2e-5


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


def _case(N, K, C, seed):
    ti = synth.ternary_inputs(N, K, C, seed=seed)
    blocks = oracle.ptq1_0_pack(ti.trits.numpy(), np_bits(ti.d))
    return blocks, np_bits(ti.x)


@pytest.mark.parametrize("N,K,C", [
    (1, 128, 1), (7, 256, 2),         # one block; a ragged row group
    (600, 1152, 3), (33, 640, 5),     # nine and five blocks a row; two rows a group at C > 4
    (17280, 5120, 1),                 # decode shape of the page's model
    (6144, 5120, 8), (5120, 17280, 4), (5120, 17280, 8),
    (37, 23168, 8),                   # the largest K whose x fits shared memory at C = 8
    (10336, 4096, 2),                 # one warp per row group (partial sums by shuffles)
    (320000, 128, 1),                 # more groups in a CTA than threads: threads take several groups
])
def test_mmvq_ptq1_0(w4, N, K, C):
    blocks, xb = _case(N, K, C, seed=N + K + C)
    pt = oracle.quantize_q8_1_pt(xb)
    buf, out, pad = _guarded(C * N, torch.float32, -7.0)
    w4.mmvq_ptq1_0(torch.from_numpy(blocks).to(_dev()), torch.from_numpy(pt).to(_dev()), out=out)
    ref, ref_abs = oracle.mmvq_ptq1_0(blocks, pt)
    got = out.cpu().numpy().astype(np.float64).reshape(C, N)
    err = np.abs(got - ref)
    assert np.all(err <= TOL * ref_abs), "max err/ref_abs = %g" % (err / np.maximum(ref_abs, 1e-300)).max()
    assert _guards_intact(buf, pad, C * N, -7.0)


def test_mmvq_ptq1_0_chain_with_device_quantiser(w4):
    N, K, C = 2048, 5120, 2
    blocks, xb = _case(N, K, C, seed=51)
    x = torch.from_numpy(xb.view(np.int16)).view(torch.bfloat16)
    pt = w4.quantize_q8_1_pt(x.to(_dev()))
    d = w4.mmvq_ptq1_0(torch.from_numpy(blocks).to(_dev()), pt)
    pt_ref = oracle.quantize_q8_1_pt(xb)
    assert np.array_equal(pt.cpu().numpy(), pt_ref)
    ref, ref_abs = oracle.mmvq_ptq1_0(blocks, pt_ref)
    assert np.all(np.abs(d.cpu().numpy() - ref) <= TOL * ref_abs)


def test_mmvq_ptq1_0_zero_trits_and_k_zero(w4):
    N, K, C = 64, 1024, 1
    _, xb = _case(N, K, C, seed=52)
    ti = synth.ternary_inputs(N, K, C, seed=52)
    blocks = oracle.ptq1_0_pack(np.zeros((N, K), np.int8), np_bits(ti.d))
    pt = oracle.quantize_q8_1_pt(xb)
    d = w4.mmvq_ptq1_0(torch.from_numpy(blocks).to(_dev()), torch.from_numpy(pt).to(_dev()))
    assert not d.any()
    d0 = torch.full((2, 16), 3.0, device=_dev())
    w4.mmvq_ptq1_0(torch.empty((16, 0), dtype=torch.uint8, device=_dev()),
                   torch.empty((2, 0), dtype=torch.uint8, device=_dev()), out=d0)
    assert torch.all(d0 == 0)


def _ptq1_1_case(N, K, C, seed, outliers):
    ti = synth.ternary_inputs(N, K, C, seed=seed, outlier_fraction=outliers)
    blocks = oracle.ptq1_0_pack(ti.trits.numpy(), np_bits(ti.d))
    return blocks, oracle.ptq1_1_encode(blocks), np_bits(ti.x)


def _dev_tables(w):
    code = torch.from_numpy(np.ascontiguousarray(w.codebook)).to(_dev())
    ei = torch.from_numpy(np.ascontiguousarray(w.esc_idx)).to(_dev())
    ep = torch.from_numpy(np.ascontiguousarray(w.esc_patt)).to(_dev())
    return torch.from_numpy(w.sblocks).to(_dev()), code, ei, ep


@pytest.mark.parametrize("N,K,C,outliers", [
    (1000, 1152, 2, 0.9),      # full codebook, free-trit indices and escapes; a padded last superblock
    (17280, 5120, 1, 0.002),   # decode shape
    (5120, 17280, 8, 0.0),     # 135 blocks a row: seventeen superblocks, the last holding seven blocks
    (37, 22528, 8, 0.5),       # the largest K whose x and codebook fit shared memory at C = 8
])
def test_mmvq_ptq1_1(w4, N, K, C, outliers):
    blocks, w, xb = _ptq1_1_case(N, K, C, N + K + C, outliers)
    pt = oracle.quantize_q8_1_pt(xb)
    sb, code, ei, ep = _dev_tables(w)
    buf, out, pad = _guarded(C * N, torch.float32, -7.0)
    w4.mmvq_ptq1_1(sb, code, ei, ep, torch.from_numpy(pt).to(_dev()), K, out=out)
    assert w4.device_error() == 0
    ref, ref_abs = oracle.mmvq_ptq1_1(w, pt)
    got = out.cpu().numpy().astype(np.float64).reshape(C, N)
    err = np.abs(got - ref)
    assert np.all(err <= TOL * ref_abs), "max err/ref_abs = %g" % (err / np.maximum(ref_abs, 1e-300)).max()
    assert _guards_intact(buf, pad, C * N, -7.0)
    # the same weights as PTQ1_0 blocks give the same products (the oracle says so exactly)
    d0 = w4.mmvq_ptq1_0(torch.from_numpy(blocks).to(_dev()), torch.from_numpy(pt).to(_dev()))
    assert np.all(np.abs(d0.cpu().numpy() - ref) <= TOL * ref_abs)


def test_mmvq_ptq1_1_unresolvable_pattern_reports_device_error(w4):
    """A codebook cut short and an escape table with an entry missing: the
    kernel's own lookups find nothing, record device error 2 and go on."""
    N, K, C = 1000, 1152, 1
    _, w, xb = _ptq1_1_case(N, K, C, 61, 0.9)
    assert len(w.esc_idx) > 1 and len(w.codebook) == 767
    pt = torch.from_numpy(oracle.quantize_q8_1_pt(xb)).to(_dev())
    sb, code, ei, ep = _dev_tables(w)
    assert w4.device_error() == 0
    w4.mmvq_ptq1_1(sb, code[:100].contiguous(), ei, ep, pt, K)
    assert w4.device_error() == 2
    assert w4.device_error() == 0          # read and cleared
    w4.mmvq_ptq1_1(sb, code, ei[1:].clone(), ep[1:].clone(), pt, K)   # fresh, 16-byte aligned copies
    assert w4.device_error() == 2
