"""The seeded input generators are deterministic and have the stated shapes."""
import numpy as np
import torch

import synth


def test_gemv_inputs_deterministic_and_shaped():
    a = synth.gemv_inputs(64, 256, 2, act="bf16", seed=0)
    b = synth.gemv_inputs(64, 256, 2, act="bf16", seed=0)
    c = synth.gemv_inputs(64, 256, 2, act="bf16", seed=1)
    assert torch.equal(a.qweight, b.qweight) and torch.equal(a.x, b.x)
    assert not torch.equal(a.qweight, c.qweight)
    assert a.qweight.shape == (64, 32) and a.qweight.dtype == torch.int32
    assert a.x.shape == (2, 256) and a.x.dtype == torch.bfloat16
    s = a.scale.float()
    assert s.min() >= 0.001 - 1e-5 and s.max() <= 0.01 + 1e-4
    assert torch.all(a.zero.float() == 8.0)


def test_gemv_inputs_nibbles_uniform():
    t = synth.gemv_inputs(512, 1024, 1, act="f32", seed=0)
    words = synth.np_bits(t.qweight)
    nib = np.concatenate([(words >> (4 * j)) & 0xF for j in range(8)]).ravel()
    counts = np.bincount(nib, minlength=16)
    assert counts.min() > 0.9 * counts.mean() and counts.max() < 1.1 * counts.mean()
    assert t.scale.dtype == torch.float32 and float(t.scale.max()) <= 2.0 / 16


def test_gemm_and_quant_inputs():
    g = synth.gemm_inputs(16, 32, 64, seed=0)
    assert g.A.shape == (16, 64) and g.B.shape == (32, 32) and g.B.dtype == torch.uint8
    assert torch.all(g.zero.float() == 8.0) and torch.all(g.scale.float() == torch.tensor(0.01).bfloat16().float())
    w = synth.quant_inputs(64, 32, seed=0)
    assert w.dtype == torch.bfloat16 and w.shape == (64, 32)
    assert torch.equal(w, synth.quant_inputs(64, 32, seed=0))


def test_bf16_half_ulp_helper():
    import sys
    from helpers import bf16_half_ulp, parity_violations
    assert list(bf16_half_ulp([1.0, 1.5, 255.0, 256.0, 0.0, -3.0])) == [2**-8, 2**-8, 0.5, 1.0, 0.0, 2**-7]
    # a correctly rounded bf16 value of 1 + 2**-8 + tiny passes, a value two ulps off fails
    ref = np.array([1.0 + 2**-8 + 1e-6])
    assert not parity_violations(np.array([1.0]), ref, np.array([1.0]), 2e-3, True).any()
    assert parity_violations(np.array([1.0 - 2**-6]), ref, np.array([1.0]), 2e-3, True).any()


def test_ternary_inputs_deterministic_and_shaped():
    a = synth.ternary_inputs(64, 1152, 2, seed=0)
    b = synth.ternary_inputs(64, 1152, 2, seed=0)
    assert torch.equal(a.trits, b.trits) and torch.equal(a.d, b.d) and torch.equal(a.x, b.x)
    assert a.trits.shape == (64, 1152) and a.trits.dtype == torch.int8
    assert a.d.shape == (64, 9) and a.x.shape == (2, 1152) and a.x.dtype == torch.bfloat16
    counts = np.bincount(a.trits.numpy().ravel() + 1, minlength=3)
    assert counts.min() > 0.95 * counts.mean()
    d = synth.np_bits(a.d)
    e = (d >> 10) & 31
    assert (d < 0x8000).all() and e.min() >= 5 and e.max() <= 14      # positive halves, exponents in range
    steps = np.abs(np.diff(e.astype(int), axis=1))
    assert steps.max() <= 1 and 0.85 < (steps == 0).mean() < 0.99
    wild = synth.ternary_inputs(64, 1152, 1, seed=0, outlier_fraction=1.0)
    assert (np.abs(np.diff(((synth.np_bits(wild.d) >> 10) & 31).astype(int), axis=1)) > 1).any()


def test_ptq1_0_blocks_are_valid_blocks():
    """Every qs byte is a five-trit byte, every qh field a digit; the bytes
    decode (through the oracle) to trits uniform over {-1, 0, 1}."""
    import oracle
    b = synth.ptq1_0_blocks(40, 1152, seed=0)
    assert b.shape == (40, 9, 28) and b.dtype == np.uint8
    assert np.array_equal(b, synth.ptq1_0_blocks(40, 1152, seed=0))
    assert b[..., :24].max() <= 242
    qh = b[..., 24:26]
    for j in range(4):
        assert ((qh >> (2 * j)) & 3).max() <= 2
    t, d = oracle.ptq1_0_unpack(b)
    counts = np.bincount(t.ravel() + 1, minlength=3)
    assert counts.min() > 0.95 * counts.mean()
    assert np.array_equal(oracle.ptq1_0_pack(t, d), b)
