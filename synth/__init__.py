"""Seeded synthetic inputs for the int4 weight-only workloads.

Shared by the tests, the package smoke check and the benchmark.  This module
holds none of the method's arithmetic: it only draws random bits and values
with torch's CPU generator and casts dtypes.  Packed int4 operands are drawn
directly as uniform random bytes, which is the same distribution as eight (or
two) independent uniform 0..15 nibbles, so no packing code is needed here.

Draw order for every workload is fixed (weights, scale, zero, activations)
so the same seed gives the same bytes on every machine.
"""
from dataclasses import dataclass

import numpy as np
import torch

# Workload shapes (synthetic stand-ins shaped like the pages' workloads: the
# Qwen K values 5120, 6144 and 17280 of the MMVQ section, and the 8192^3
# bf16 x int4 example of the Helion issue).
TINY = dict(N=256, K=512, C=1, act="f32")
DECODE = dict(N=17280, K=5120, C=1, act="bf16")
SMALL_BATCH = [dict(N=5120, K=17280, C=4, act="bf16"), dict(N=5120, K=17280, C=8, act="bf16"),
               dict(N=6144, K=5120, C=4, act="bf16"), dict(N=6144, K=5120, C=8, act="bf16")]
QUANT = dict(K=8192, N=8192)
GEMM = dict(M=8192, N=8192, K=8192)


def _gen(seed):
    return torch.Generator(device="cpu").manual_seed(int(seed))


@dataclass
class GemvInputs:
    qweight: torch.Tensor  # int32 [N, K/8]: bit patterns of the packed uint32 words
    scale: torch.Tensor    # [N] float32 or bfloat16
    zero: torch.Tensor     # [N] same dtype as scale
    x: torch.Tensor        # [C, K] same dtype as scale
    N: int
    K: int
    C: int
    act: str


def gemv_inputs(N, K, C, act="bf16", seed=0, scale_range=None, zero_value=8.0, q_dist="uniform", q_sigma=0.7,
                zero_rows=0):
    """Packed uint4 weights uniform 0..15, per-row scale, constant zero, x ~ N(0,1).

    act="bf16": scale U[0.001, 0.01], zero 8, x N(0,1), all bf16.
    act="f32":  scale U[0.5, 2]/16, zero 8.0, x N(0,1), all fp32.

    q_dist picks the nibble distribution (each nibble drawn independently, so
    the two nibbles of a byte are interchangeable and no packing order is
    involved):
      "uniform"  0..15 (the workloads' draw: uniform random bytes);
      "near"     round(zero_value + N(0, q_sigma)) clamped to 0..15, the
                 shape of real asymmetric int4 weights clustered at their
                 zero point (zero_value must be an integer);
      "zero"     every nibble equal to zero_value (an integer 0..15).
    zero_rows = m > 0 additionally sets every nibble of rows 0, m, 2m, ... to
    zero_value.  The uniform draw leaves the bytes of the default call
    unchanged.
    """
    if K % 8:
        raise ValueError("K must be a multiple of 8")
    g = _gen(seed)
    zi = int(round(float(zero_value)))
    if q_dist != "uniform" or zero_rows:
        if float(zero_value) != zi or not 0 <= zi <= 15:
            raise ValueError("q_dist / zero_rows need an integer zero_value in 0..15")
    if q_dist == "uniform":
        qbytes = torch.randint(0, 256, (N, K // 2), dtype=torch.uint8, generator=g)
    elif q_dist == "near":
        nib = torch.round(torch.randn(N, K, generator=g, dtype=torch.float64) * q_sigma + zi).clamp(0, 15)
        nib = nib.to(torch.uint8).view(N, K // 2, 2)
        qbytes = nib[:, :, 0] + 16 * nib[:, :, 1]
    elif q_dist == "zero":
        qbytes = torch.full((N, K // 2), 17 * zi, dtype=torch.uint8)
    else:
        raise ValueError(q_dist)
    if zero_rows:
        qbytes[::zero_rows] = 17 * zi
    qweight = qbytes.contiguous().view(torch.int32)
    if act == "f32":
        lo, hi = scale_range or (0.5 / 16, 2.0 / 16)
        dt = torch.float32
    elif act == "bf16":
        lo, hi = scale_range or (0.001, 0.01)
        dt = torch.bfloat16
    else:
        raise ValueError(act)
    scale = (torch.rand(N, generator=g, dtype=torch.float32) * (hi - lo) + lo).to(dt)
    zero = torch.full((N,), float(zero_value), dtype=dt)
    x = torch.randn(C, K, generator=g, dtype=torch.float32).to(dt)
    return GemvInputs(qweight, scale, zero, x, N, K, C, act)


@dataclass
class PackedGemvInputs:
    packed: torch.Tensor  # uint8 [K/2, N]: two two's complement nibbles per byte along K
    scale: torch.Tensor   # float32 [N]
    x: torch.Tensor       # bf16 [C, K]
    N: int
    K: int
    C: int


def packed_gemv_inputs(N, K, C, seed=0, scale_range=(0.005, 0.02), q_dist="uniform", q_sigma=0.7, zero_cols=0):
    """The quantiser's operand layout: uniform random bytes (= independent
    uniform nibbles), fp32 per-column scale in the range the quantiser gives
    for N(0, 0.02) weights, x ~ N(0,1) bf16.

    q_dist: "uniform" (uniform bytes), "near" (two's complement nibbles
    round(N(0, q_sigma)) clamped to -8..7, each drawn independently) or
    "zero" (every weight 0); zero_cols = m > 0 also zeroes columns 0, m, 2m,
    ... (the operand is symmetric: a zero weight is the nibble 0)."""
    if K % 2:
        raise ValueError("K must be even")
    g = _gen(seed)
    if q_dist == "uniform":
        packed = torch.randint(0, 256, (K // 2, N), dtype=torch.uint8, generator=g)
    elif q_dist == "near":
        nib = torch.round(torch.randn(K, N, generator=g, dtype=torch.float64) * q_sigma).clamp(-8, 7)
        nib = nib.to(torch.int16).view(K // 2, 2, N) & 15
        packed = (nib[:, 0, :] + 16 * nib[:, 1, :]).to(torch.uint8)
    elif q_dist == "zero":
        packed = torch.zeros((K // 2, N), dtype=torch.uint8)
    else:
        raise ValueError(q_dist)
    if zero_cols:
        packed[:, ::zero_cols] = 0
    packed = packed.contiguous()
    lo, hi = scale_range
    scale = torch.rand(N, generator=g, dtype=torch.float32) * (hi - lo) + lo
    x = torch.randn(C, K, generator=g, dtype=torch.float32).to(torch.bfloat16)
    return PackedGemvInputs(packed, scale, x, N, K, C)


@dataclass
class Int8GemvInputs:
    q: torch.Tensor       # int8 [K, N]
    scale: torch.Tensor   # float32 [N]
    x: torch.Tensor       # bf16 [C, K]
    N: int
    K: int
    C: int


def int8_gemv_inputs(N, K, C, seed=0, scale_range=(2.0e-4, 8.0e-4)):
    """The int8 quantiser's operand: uniform int8 weights, fp32 per-column
    scale in the range the int8 quantiser gives for N(0, 0.02) weights,
    x ~ N(0,1) bf16."""
    g = _gen(seed)
    q = torch.randint(-128, 128, (K, N), dtype=torch.int16, generator=g).to(torch.int8)
    lo, hi = scale_range
    scale = torch.rand(N, generator=g, dtype=torch.float32) * (hi - lo) + lo
    x = torch.randn(C, K, generator=g, dtype=torch.float32).to(torch.bfloat16)
    return Int8GemvInputs(q, scale, x, N, K, C)


@dataclass
class TernaryInputs:
    trits: torch.Tensor   # int8 [N, K] in {-1, 0, 1}
    d: torch.Tensor       # int16 [N, K/128]: bit patterns of positive IEEE halves, one per 128 weights
    x: torch.Tensor       # bf16 [C, K]
    N: int
    K: int
    C: int


def ternary_inputs(N, K, C, seed=0, outlier_fraction=0.0):
    """Ternary weights shaped like a trained model's PTQ1_0 tensors: trits
    uniform over {-1, 0, 1}; one positive half scale per 128 weights whose
    exponent drifts along the row (first block uniform in 8..11, each next
    block steps -1 / 0 / +1 with probability 0.035 / 0.93 / 0.035, kept
    within 5..14: about 0.44 bits per step, near the 0.41 bits the ternary
    compression page measured on its model), mantissas uniform.  A fraction
    `outlier_fraction` of rows draws every exponent uniformly in 5..14
    instead.  x ~ N(0,1) bf16 [C, K]."""
    if K % 128:
        raise ValueError("K must be a multiple of 128")
    g = _gen(seed)
    bpr = K // 128
    trits = (torch.randint(0, 3, (N, K), dtype=torch.int16, generator=g) - 1).to(torch.int8)
    start = torch.randint(8, 12, (N,), dtype=torch.int32, generator=g)
    u = torch.rand(N, max(bpr - 1, 0), generator=g)
    steps = (u > 0.965).to(torch.int32) - (u < 0.035).to(torch.int32)
    outlier = torch.rand(N, generator=g) < outlier_fraction
    wild = torch.randint(5, 15, (N, bpr), dtype=torch.int32, generator=g)
    mant = torch.randint(0, 1024, (N, bpr), dtype=torch.int32, generator=g)
    exps = torch.empty(N, bpr, dtype=torch.int32)
    if bpr:
        exps[:, 0] = start
    for b in range(1, bpr):
        exps[:, b] = (exps[:, b - 1] + steps[:, b - 1]).clamp(5, 14)
    exps = torch.where(outlier[:, None], wild, exps)
    d = ((exps << 10) | mant).to(torch.int16)
    x = torch.randn(C, K, generator=g, dtype=torch.float32).to(torch.bfloat16)
    return TernaryInputs(trits, d, x, N, K, C)


def ptq1_0_blocks(N, K, seed=0):
    """PTQ1_0 tensors drawn directly as bytes (uint8 [N, K/128, 28]): each qs
    byte uniform over 0..242 (= five independent uniform trits), each 2-bit
    field of qh uniform over 0..2 (one uniform trit), d as ternary_inputs
    draws it.  The same distribution as packing ternary_inputs' trits, with
    no packing code here."""
    if K % 128:
        raise ValueError("K must be a multiple of 128")
    bpr = K // 128
    g = _gen(seed)
    qs = torch.randint(0, 243, (N, bpr, 24), dtype=torch.int16, generator=g).to(torch.uint8)
    fields = torch.randint(0, 3, (N, bpr, 2, 4), dtype=torch.int16, generator=g)
    qh = (fields[..., 0] | (fields[..., 1] << 2) | (fields[..., 2] << 4) | (fields[..., 3] << 6)).to(torch.uint8)
    d = np_bits(ternary_inputs(N, 128 * bpr, 1, seed=seed + 1).d).reshape(N, bpr, 1).view(np.uint8)
    out = np.concatenate([qs.numpy(), qh.numpy(), d], axis=2)
    return np.ascontiguousarray(out)


def quant_inputs(K, N, seed=0, std=0.02):
    """W bf16 [K, N] ~ N(0, std)."""
    g = _gen(seed)
    return (torch.randn(K, N, generator=g, dtype=torch.float32) * std).to(torch.bfloat16)


@dataclass
class GemmInputs:
    A: torch.Tensor      # bf16 [M, K]
    B: torch.Tensor      # uint8 [K/2, N]: two unsigned nibbles per byte along K
    scale: torch.Tensor  # bf16 [N]
    zero: torch.Tensor   # bf16 [N]
    M: int
    N: int
    K: int


def gemm_inputs(M, N, K, seed=0, scale_value=0.01, zero_value=8.0, random_scale=False):
    """A ~ N(0,1) bf16; B uniform bytes; zero 8; scale 0.01 (or U[0.005,0.02])."""
    if K % 2:
        raise ValueError("K must be even")
    g = _gen(seed)
    A = torch.randn(M, K, generator=g, dtype=torch.float32).to(torch.bfloat16)
    B = torch.randint(0, 256, (K // 2, N), dtype=torch.uint8, generator=g)
    if random_scale:
        scale = (torch.rand(N, generator=g) * 0.015 + 0.005).to(torch.bfloat16)
    else:
        scale = torch.full((N,), float(scale_value), dtype=torch.bfloat16)
    zero = torch.full((N,), float(zero_value), dtype=torch.bfloat16)
    return GemmInputs(A, B, scale, zero, M, N, K)


def np_bits(t):
    """numpy view of a CPU tensor's raw bits: bf16 -> uint16, int32 -> uint32,
    uint8 -> uint8, float32 -> float32."""
    t = t.detach().contiguous().cpu()
    if t.dtype == torch.bfloat16:
        return t.view(torch.int16).numpy().view(np.uint16)
    if t.dtype == torch.int32:
        return t.numpy().view(np.uint32)
    if t.dtype == torch.int16:
        return t.numpy().view(np.uint16)
    if t.dtype == torch.int8:
        return t.numpy().view(np.uint8)
    return t.numpy()
