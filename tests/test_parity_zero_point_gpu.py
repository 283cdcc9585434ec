"""GPU parity where the zero point decides the result.

Weights that sit at their zero point contribute exactly nothing: a row whose
nibbles all equal z has d = 0 and sum_k |w x| = 0, so the per-output bound
2e-3 * sum_k |w x| (1e-5 for fp32) leaves no room at all.  Real asymmetric
int4 weights cluster around z, one-hot x picks single weights, and small
integer x with s = 1 gives exact integers: each of these checks that the
kernels remove the zero point before any rounding (page "怎样在安卓端利用
Vulkan 编写 4-bit 专用算子", section 2: (q - zero) * scale inside the dot
loop).  Every GEMV path is covered: one column of x (fp16 MMAs), several
columns (bf16 MMAs), fp32 inputs and rows that are not whole 16-byte lines
(CUDA-core FMA), a K split over a cluster, and the permuted operand.
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

PATHS = [
    (1000, 5120, 1, "bf16"),    # one column of x: fp16 tensor-core path
    (700, 4096, 4, "bf16"),     # several columns: bf16 tensor-core path
    (300, 2048, 8, "bf16"),
    (256, 512, 1, "f32"),       # fp32 inputs: CUDA-core FMA path
    (130, 1000, 3, "f32"),
    (77, 520, 3, "bf16"),       # K % 32 != 0: CUDA-core path for bf16
    (300, 40000, 2, "bf16"),    # K split over a cluster, bf16
    (200, 40960, 1, "bf16"),    # K split over a cluster, fp16
]
PATH_IDS = ["N%dK%dC%d%s" % p for p in PATHS]


@pytest.fixture(scope="module")
def w4():
    import gemm_int4_dequant_gb300 as m
    return m


def _dev():
    return torch.device("cuda:0")


def _gemv(w4, g):
    d = w4.gemv_w4(g.qweight.to(_dev()), g.scale.to(_dev()), g.zero.to(_dev()), g.x.to(_dev()))
    code = oracle.F32 if g.act == "f32" else oracle.BF16
    ref, ref_abs = oracle.gemv(np_bits(g.qweight), np_bits(g.scale), np_bits(g.zero), np_bits(g.x), code)
    got = d.float().cpu().numpy().astype(np.float64).reshape(g.C, g.N)
    return got, ref, ref_abs


def _assert_parity(got, ref, ref_abs, act):
    tol = F32_TOL if act == "f32" else BF16_TOL
    bad = parity_violations(got, ref, ref_abs, tol, bf16_out=(act == "bf16"))
    if bad.any():
        i = np.argwhere(bad)[:5]
        raise AssertionError("%d outputs outside the bound; first %s: got %s ref %s ref_abs %s" % (
            bad.sum(), i.tolist(), got[tuple(i.T)], ref[tuple(i.T)], ref_abs[tuple(i.T)]))


def _set_nibble(qweight, rows, k, value):
    """Set weight k of the given rows to `value` (word k/8, bits 4(k%8)..+3:
    the packing order of the Vulkan page, section 1)."""
    w = qweight.view(torch.int32).numpy().view(np.uint32)
    sh = 4 * (k % 8)
    w[rows, k // 8] = (w[rows, k // 8] & ~np.uint32(0xF << sh)) | np.uint32(value << sh)


@pytest.mark.parametrize("N,K,C,act", PATHS, ids=PATH_IDS)
@pytest.mark.parametrize("z,zero_rows", [(8, 3), (0, 5), (15, 1)])
def test_rows_at_the_zero_point_give_exact_zero(w4, N, K, C, act, z, zero_rows):
    g = synth.gemv_inputs(N, K, C, act=act, seed=N + K + z, zero_value=z, zero_rows=zero_rows)
    got, ref, ref_abs = _gemv(w4, g)
    rows = np.arange(0, N, zero_rows)
    assert np.all(ref[:, rows] == 0) and np.all(ref_abs[:, rows] == 0)
    nz = np.flatnonzero(got[:, rows])
    assert nz.size == 0, "%d outputs of zero-point rows are not 0, e.g. %s" % (nz.size, got[:, rows].ravel()[nz[:4]])
    _assert_parity(got, ref, ref_abs, act)


@pytest.mark.parametrize("N,K,C,act", PATHS, ids=PATH_IDS)
@pytest.mark.parametrize("z", [8, 3])
def test_weights_clustered_at_the_zero_point(w4, N, K, C, act, z):
    g = synth.gemv_inputs(N, K, C, act=act, seed=2 * N + K, zero_value=z, q_dist="near", q_sigma=0.6)
    _assert_parity(*_gemv(w4, g), act)


@pytest.mark.parametrize("N,K,C,act", PATHS, ids=PATH_IDS)
def test_one_hot_x_picks_single_weights(w4, N, K, C, act):
    g = synth.gemv_inputs(N, K, C, act=act, seed=3 * N + K)
    dt = g.x.dtype
    x = torch.zeros(C, K, dtype=torch.float32)
    ks = [0, K - 1, K // 2 + 3, 8 * (K // 16) + 7, 37 % K, K - 9, 129 % K, 1]
    for c in range(C):
        x[c, ks[c]] = [1.0, -2.5, 0.3, 7.0, -1.0, 0.015625, 3.0, -0.75][c]
    g.x = x.to(dt)
    got, ref, ref_abs = _gemv(w4, g)
    _assert_parity(got, ref, ref_abs, act)
    assert np.all(got[ref_abs == 0] == 0)   # weights equal to z (1 in 16 with uniform nibbles)


@pytest.mark.parametrize("N,K,C,act", PATHS, ids=PATH_IDS)
@pytest.mark.parametrize("z", [0, 8])
def test_small_integer_x_gives_exact_integers(w4, N, K, C, act, z):
    """s = 1, integer z and integer x: every product and partial sum is an
    integer below 2^24, so fp32 accumulation is exact and the output is the
    exact integer rounded once to the output type."""
    g = synth.gemv_inputs(N, K, C, act=act, seed=4 * N + K + z, zero_value=z, scale_range=(1.0, 1.0))
    gen = torch.Generator().manual_seed(N + C)
    g.x = torch.randint(-3, 4, (C, K), generator=gen).to(g.x.dtype)
    got, ref, _ = _gemv(w4, g)
    assert np.all(ref == np.round(ref)) and np.abs(ref).max() < 2 ** 24
    want = torch.from_numpy(ref).to(torch.float32 if act == "f32" else torch.bfloat16).double().numpy()
    bad = np.flatnonzero(got != want)
    assert bad.size == 0, "%d outputs differ, e.g. got %s want %s" % (bad.size, got.ravel()[bad[:4]],
                                                                      want.ravel()[bad[:4]])


@pytest.mark.parametrize("N,K,C", [(1000, 5120, 1), (300, 40960, 1), (700, 4096, 2), (300, 2048, 8)])
def test_dominant_x_element_on_zero_point_weights(w4, N, K, C):
    """One x element 2^40 times the rest, its weight equal to z in every
    other row: there sum |w x| holds only the small elements, which must
    survive (an fp16 conversion of x scaled to the large element would drop
    them)."""
    g = synth.gemv_inputs(N, K, C, act="bf16", seed=5 * N + K)
    k0 = K // 3
    x = g.x.float()
    x[:, k0] = 2.0 ** 40 * torch.sign(x[:, k0] + 0.5)
    g.x = x.to(torch.bfloat16)
    _set_nibble(g.qweight, np.arange(0, N, 2), k0, 8)
    got, ref, ref_abs = _gemv(w4, g)
    _assert_parity(got, ref, ref_abs, "bf16")


@pytest.mark.parametrize("N,K,C", [(1000, 5120, 1), (300, 40960, 1), (700, 4096, 2), (300, 2048, 8)])
@pytest.mark.parametrize("exp", [-130, -100, 100])
def test_extreme_x_exponents(w4, N, K, C, exp):
    """x scaled to bf16 subnormals (2^-130: 3 to 7 significant bits), near
    the bottom of the normal range and near the top."""
    g = synth.gemv_inputs(N, K, C, act="bf16", seed=6 * N + K + exp)
    g.x = (g.x.float() * 2.0 ** exp).to(torch.bfloat16)
    got, ref, ref_abs = _gemv(w4, g)
    _assert_parity(got, ref, ref_abs, "bf16")
    assert np.all(np.isfinite(got))


# ---------------------------------------------------------------------------
# gemv_w4_permuted: the symmetric operand (zero weight = nibble 0)
# ---------------------------------------------------------------------------

PERM_SHAPES = [(1000, 512, 1), (512, 5120, 4), (260, 40960, 8), (100, 192, 3)]


def _gemv_permuted(w4, g):
    perm = w4.permute_int4(g.packed.to(_dev()))
    d = w4.gemv_w4_permuted(perm, g.scale.to(_dev()), g.x.to(_dev()))
    ref, ref_abs = oracle.gemv_packed(g.packed.numpy(), g.scale.numpy(), np_bits(g.x))
    return d.float().cpu().numpy().astype(np.float64).reshape(g.C, g.N), ref, ref_abs


@pytest.mark.parametrize("N,K,C", PERM_SHAPES)
def test_permuted_zero_columns_give_exact_zero(w4, N, K, C):
    g = synth.packed_gemv_inputs(N, K, C, seed=N + K, zero_cols=3)
    got, ref, ref_abs = _gemv_permuted(w4, g)
    cols = np.arange(0, N, 3)
    assert np.all(ref[:, cols] == 0)
    assert np.all(got[:, cols] == 0)
    _assert_parity(got, ref, ref_abs, "bf16")


@pytest.mark.parametrize("N,K,C", PERM_SHAPES)
def test_permuted_weights_clustered_at_zero(w4, N, K, C):
    g = synth.packed_gemv_inputs(N, K, C, seed=2 * N + K, q_dist="near", q_sigma=0.6)
    _assert_parity(*_gemv_permuted(w4, g), "bf16")


@pytest.mark.parametrize("N,K,C", PERM_SHAPES)
def test_permuted_one_hot_x(w4, N, K, C):
    g = synth.packed_gemv_inputs(N, K, C, seed=3 * N + K)
    x = torch.zeros(C, K)
    for c in range(C):
        x[c, (c * 97 + 5) % K] = [1.0, -2.5, 0.3, 7.0, -1.0, 0.015625, 3.0, -0.75][c]
    g.x = x.to(torch.bfloat16)
    got, ref, ref_abs = _gemv_permuted(w4, g)
    _assert_parity(got, ref, ref_abs, "bf16")
    assert np.all(got[ref_abs == 0] == 0)


# ---------------------------------------------------------------------------
# gemm_w4: columns of B at the zero point
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("M,N,K", [(256, 512, 256), (300, 1008, 1024)])
def test_gemm_zero_point_columns_give_exact_zero(w4, M, N, K):
    gi = synth.gemm_inputs(M, N, K, seed=M + N)
    B = gi.B.clone()
    B[:, ::3] = 0x88          # both nibbles 8 = the zero point
    C = w4.gemm_w4(gi.A.to(_dev()), B.to(_dev()), gi.scale.to(_dev()), gi.zero.to(_dev()))
    got = C.float().cpu().numpy().astype(np.float64)
    assert np.all(got[:, ::3] == 0)
    ref, ref_abs = oracle.gemm_full(np_bits(gi.A), B.numpy(), np_bits(gi.scale), np_bits(gi.zero))
    _assert_parity(got, ref, ref_abs, "bf16")
