"""CPU oracle for the int4 weight-only hot path (TEST INFRASTRUCTURE ONLY).

Only tests/, the package smoke check and bench.py's CPU-baseline leg may
import this package.  The product library never imports, links or calls it,
and it shares no code with the CUDA path.  The arithmetic lives in
w4_oracle.c (plain C, fp64 products); this module only marshals numpy
arrays through ctypes.

Every function is pinned against facts the source pages fix, in
tests/test_oracle_pins.py and tests/test_oracle_ternary_pins.py.
"""
import ctypes
import os

import numpy as np

from .build import build_oracle

_lib = None

F32, BF16 = 0, 1


def _load():
    global _lib
    if _lib is None:
        # W4_ORACLE_LIB names another build of the same source (the pin
        # suite's mutation check loads deliberately broken copies this way).
        lib = ctypes.CDLL(os.environ.get("W4_ORACLE_LIB") or build_oracle())
        P = ctypes.c_void_p
        L = ctypes.c_long
        lib.w4o_gemv.argtypes = [P, P, P, P, ctypes.c_int, L, L, L, L, L, P, P]
        lib.w4o_gemv.restype = None
        lib.w4o_gemm_at.argtypes = [P, P, P, P, L, L, L, P, P, L, P, P]
        lib.w4o_gemm_at.restype = None
        lib.w4o_quantize_pack.argtypes = [P, L, L, P, P]
        lib.w4o_quantize_pack.restype = None
        lib.w4o_permute.argtypes = [P, L, L, P]
        lib.w4o_permute.restype = ctypes.c_int
        lib.w4o_gemv_packed.argtypes = [P, P, P, L, L, L, L, L, P, P]
        lib.w4o_gemv_packed.restype = None
        lib.w4o_quantize_int8.argtypes = [P, L, L, P, P]
        lib.w4o_quantize_int8.restype = None
        lib.w4o_permute_int8.argtypes = [P, L, L, P]
        lib.w4o_permute_int8.restype = ctypes.c_int
        lib.w4o_gemv_int8.argtypes = [P, P, P, L, L, L, L, L, P, P]
        lib.w4o_gemv_int8.restype = None
        lib.w4o_gemm_int8_at.argtypes = [P, P, P, L, L, L, P, P, L, P, P]
        lib.w4o_gemm_int8_at.restype = None
        lib.w4o_gemm_packed_at.argtypes = [P, P, P, L, L, L, P, P, L, P, P]
        lib.w4o_gemm_packed_at.restype = None
        lib.w4o_quantize_q8_1_pt.argtypes = [P, L, L, P]
        lib.w4o_quantize_q8_1_pt.restype = None
        lib.w4o_gemv_w4a8.argtypes = [P, P, P, P, L, L, L, L, L, P, P]
        lib.w4o_gemv_w4a8.restype = None
        lib.w4o_float_to_half.argtypes = [P, L, P]
        lib.w4o_float_to_half.restype = None
        lib.w4o_half_to_double.argtypes = [P, L, P]
        lib.w4o_half_to_double.restype = None
        lib.w4o_ptq1_0_pack.argtypes = [P, P, L, L, P]
        lib.w4o_ptq1_0_pack.restype = ctypes.c_int
        lib.w4o_ptq1_0_unpack.argtypes = [P, L, L, P, P]
        lib.w4o_ptq1_0_unpack.restype = None
        lib.w4o_ptq1_1_codebook.argtypes = [P, L, L, P]
        lib.w4o_ptq1_1_codebook.restype = L
        lib.w4o_ptq1_1_encode.argtypes = [P, L, L, P, L, P, P, P, L]
        lib.w4o_ptq1_1_encode.restype = L
        lib.w4o_ptq1_1_unpack.argtypes = [P, L, L, P, L, P, P, L, P, P]
        lib.w4o_ptq1_1_unpack.restype = ctypes.c_int
        lib.w4o_mmvq_ptq1_0.argtypes = [P, P, L, L, L, L, L, P, P]
        lib.w4o_mmvq_ptq1_0.restype = None
        lib.w4o_mmvq_ptq1_1.argtypes = [P, P, L, P, P, L, P, L, L, L, L, L, P, P]
        lib.w4o_mmvq_ptq1_1.restype = ctypes.c_int
        _lib = lib
    return _lib


def _ptr(a):
    return a.ctypes.data_as(ctypes.c_void_p)


def _act(a, dtype):
    """Return a C-contiguous array of the raw element type for `dtype`."""
    if dtype == BF16:
        a = np.ascontiguousarray(a)
        if a.dtype != np.uint16:
            raise TypeError("bf16 operands are passed as raw uint16 bit patterns")
        return a
    return np.ascontiguousarray(a, dtype=np.float32)


def gemv(packed_weights, scales, zeros, x, act_dtype, rows=None):
    """d[c, r] = sum_k x[c, k] * (q[r, k] - zero[r]) * scale[r], in fp64.

    packed_weights: uint32 [N, K/8] (nibble j of word i is k = 8i + j).
    scales, zeros: [N]; x: [C, K]; fp32 arrays, or uint16 bf16 bit patterns
    when act_dtype == BF16.  rows: optional (begin, end) row range; rows
    outside it are left as NaN.  Returns (d, ref_abs), both float64 [C, N].
    """
    lib = _load()
    qw = np.ascontiguousarray(packed_weights, dtype=np.uint32)
    N, kb = qw.shape
    K = kb * 8
    x = _act(x, act_dtype)
    if x.ndim == 1:
        x = x.reshape(1, -1)
    C = x.shape[0]
    if x.shape[1] != K:
        raise ValueError("x has %d columns, weights imply K=%d" % (x.shape[1], K))
    s = _act(scales, act_dtype)
    z = _act(zeros, act_dtype)
    if s.shape != (N,) or z.shape != (N,):
        raise ValueError("scales/zeros must be [N]")
    r0, r1 = (0, N) if rows is None else rows
    d = np.full((C, N), np.nan)
    ref = np.full((C, N), np.nan)
    lib.w4o_gemv(_ptr(qw), _ptr(s), _ptr(z), _ptr(x), act_dtype, N, K, C, r0, r1,
                 _ptr(d), _ptr(ref))
    return d, ref


def gemm_at(A_bits, B_packed, scale_bits, zero_bits, m_idx, n_idx):
    """C[m, n] = sum_k A[m, k] * (u[k, n] - zero[n]) * scale[n] at the given
    coordinates, in fp64.

    A_bits: uint16 bf16 patterns [M, K]; B_packed: uint8 [K/2, N] (low nibble
    = even k, unsigned); scale_bits, zero_bits: uint16 bf16 patterns [N].
    Returns (c, ref_abs) float64 arrays shaped like m_idx.
    """
    lib = _load()
    A = np.ascontiguousarray(A_bits, dtype=np.uint16)
    B = np.ascontiguousarray(B_packed, dtype=np.uint8)
    M, K = A.shape
    if B.shape[0] * 2 != K:
        raise ValueError("B must be [K/2, N]")
    N = B.shape[1]
    s = np.ascontiguousarray(scale_bits, dtype=np.uint16)
    z = np.ascontiguousarray(zero_bits, dtype=np.uint16)
    mi = np.ascontiguousarray(m_idx, dtype=np.int64).ravel()
    ni = np.ascontiguousarray(n_idx, dtype=np.int64).ravel()
    if mi.shape != ni.shape:
        raise ValueError("m_idx and n_idx differ in size")
    if mi.size and (mi.min() < 0 or mi.max() >= M or ni.min() < 0 or ni.max() >= N):
        raise IndexError("coordinate out of range")
    c = np.empty(mi.shape, np.float64)
    ref = np.empty(mi.shape, np.float64)
    lib.w4o_gemm_at(_ptr(A), _ptr(B), _ptr(s), _ptr(z), M, N, K, _ptr(mi), _ptr(ni),
                    mi.size, _ptr(c), _ptr(ref))
    shape = np.shape(m_idx)
    return c.reshape(shape), ref.reshape(shape)


def gemm_full(A_bits, B_packed, scale_bits, zero_bits):
    """Every element of C (small shapes only)."""
    M = np.shape(A_bits)[0]
    N = np.shape(B_packed)[1]
    mm, nn = np.meshgrid(np.arange(M), np.arange(N), indexing="ij")
    return gemm_at(A_bits, B_packed, scale_bits, zero_bits, mm, nn)


def gemm_int8_at(A_bits, q, scale, m_idx, n_idx):
    """C[m, n] = sum_k A[m, k] * q[k, n] * scale[n] at the given coordinates,
    in fp64.  A_bits: uint16 bf16 patterns [M, K]; q: int8 [K, N]; scale:
    fp32 [N].  Returns (c, ref_abs) float64 arrays shaped like m_idx."""
    lib = _load()
    A = np.ascontiguousarray(A_bits, dtype=np.uint16)
    Q = np.ascontiguousarray(q, dtype=np.int8)
    M, K = A.shape
    if Q.shape[0] != K:
        raise ValueError("q must be [K, N]")
    N = Q.shape[1]
    s = np.ascontiguousarray(scale, dtype=np.float32)
    mi = np.ascontiguousarray(m_idx, dtype=np.int64).ravel()
    ni = np.ascontiguousarray(n_idx, dtype=np.int64).ravel()
    if mi.shape != ni.shape:
        raise ValueError("m_idx and n_idx differ in size")
    if mi.size and (mi.min() < 0 or mi.max() >= M or ni.min() < 0 or ni.max() >= N):
        raise IndexError("coordinate out of range")
    c = np.empty(mi.shape, np.float64)
    ref = np.empty(mi.shape, np.float64)
    lib.w4o_gemm_int8_at(_ptr(A), _ptr(Q), _ptr(s), M, N, K, _ptr(mi), _ptr(ni), mi.size, _ptr(c), _ptr(ref))
    shape = np.shape(m_idx)
    return c.reshape(shape), ref.reshape(shape)


def gemm_int8_full(A_bits, q, scale):
    """Every element of the int8 GEMM (small shapes only)."""
    M, N = np.shape(A_bits)[0], np.shape(q)[1]
    mm, nn = np.meshgrid(np.arange(M), np.arange(N), indexing="ij")
    return gemm_int8_at(A_bits, q, scale, mm, nn)


def gemm_packed_at(A_bits, packed, scale, m_idx, n_idx):
    """C[m, n] = sum_k A[m, k] * q[k, n] * scale[n] at the given coordinates,
    in fp64, over the quantiser's packed matrix (uint8 [K/2, N], two's
    complement nibbles, even k low) and fp32 scale [N]."""
    lib = _load()
    A = np.ascontiguousarray(A_bits, dtype=np.uint16)
    P_ = np.ascontiguousarray(packed, dtype=np.uint8)
    M, K = A.shape
    if P_.shape[0] * 2 != K:
        raise ValueError("packed must be [K/2, N]")
    N = P_.shape[1]
    s = np.ascontiguousarray(scale, dtype=np.float32)
    mi = np.ascontiguousarray(m_idx, dtype=np.int64).ravel()
    ni = np.ascontiguousarray(n_idx, dtype=np.int64).ravel()
    if mi.shape != ni.shape:
        raise ValueError("m_idx and n_idx differ in size")
    if mi.size and (mi.min() < 0 or mi.max() >= M or ni.min() < 0 or ni.max() >= N):
        raise IndexError("coordinate out of range")
    c = np.empty(mi.shape, np.float64)
    ref = np.empty(mi.shape, np.float64)
    lib.w4o_gemm_packed_at(_ptr(A), _ptr(P_), _ptr(s), M, N, K, _ptr(mi), _ptr(ni), mi.size, _ptr(c), _ptr(ref))
    shape = np.shape(m_idx)
    return c.reshape(shape), ref.reshape(shape)


def gemm_packed_full(A_bits, packed, scale):
    """Every element of the GEMM over the packed matrix (small shapes only)."""
    M, N = np.shape(A_bits)[0], np.shape(packed)[1]
    mm, nn = np.meshgrid(np.arange(M), np.arange(N), indexing="ij")
    return gemm_packed_at(A_bits, packed, scale, mm, nn)


def quantize_pack(W_bits):
    """Symmetric per-column int4 quantisation + column pack.

    W_bits: uint16 bf16 patterns [K, N], K even.  Returns (scale float32 [N],
    packed uint8 [K/2, N]).
    """
    lib = _load()
    W = np.ascontiguousarray(W_bits, dtype=np.uint16)
    K, N = W.shape
    if K % 2:
        raise ValueError("K must be even")
    scale = np.empty(N, np.float32)
    packed = np.empty((K // 2, N), np.uint8)
    lib.w4o_quantize_pack(_ptr(W), K, N, _ptr(scale), _ptr(packed))
    return scale, packed


def gemv_packed(packed, scale, x_bits, cols=None):
    """d[c, n] = sum_k x[c, k] * q[k, n] * scale[n], in fp64, over the
    quantiser's packed matrix.

    packed: uint8 [K/2, N] (low nibble = even k, two's complement);
    scale: float32 [N]; x_bits: uint16 bf16 patterns [C, K].  cols: optional
    (begin, end) column range; columns outside it are NaN.  Returns
    (d, ref_abs), both float64 [C, N].
    """
    lib = _load()
    p = np.ascontiguousarray(packed, dtype=np.uint8)
    s = np.ascontiguousarray(scale, dtype=np.float32)
    xb = np.ascontiguousarray(x_bits, dtype=np.uint16)
    Kp, N = p.shape
    K = 2 * Kp
    C = xb.shape[0] if xb.ndim == 2 else 1
    if xb.size != C * K or s.size != N:
        raise ValueError("shape mismatch")
    b, e = (0, N) if cols is None else cols
    d = np.full((C, N), np.nan)
    ref = np.full((C, N), np.nan)
    lib.w4o_gemv_packed(_ptr(p), _ptr(s), _ptr(xb), N, K, C, b, e, _ptr(d), _ptr(ref))
    return d, ref


def permute(packed, K, N):
    """Page-1 int4 permute of packed [K/2, N] into N*K/2 interleaved bytes."""
    lib = _load()
    p = np.ascontiguousarray(packed, dtype=np.uint8)
    if p.shape != (K // 2, N):
        raise ValueError("packed must be [K/2, N]")
    if K % 64 or N % 4:
        raise ValueError("permute needs K % 64 == 0 and N % 4 == 0")
    out = np.zeros(N * K // 2, np.uint8)
    if lib.w4o_permute(_ptr(p), K, N, _ptr(out)) != 0:
        raise MemoryError("oracle permute could not allocate its stream")
    return out


# ---------------------------------------------------------------------------
# int8 weight-only variant
# ---------------------------------------------------------------------------

def quantize_int8(W_bits):
    """Symmetric per-column int8 quantisation of W [K, N] (uint16 bf16
    patterns).  Returns (scale float32 [N], q int8 [K, N])."""
    lib = _load()
    W = np.ascontiguousarray(W_bits, dtype=np.uint16)
    K, N = W.shape
    scale = np.empty(N, np.float32)
    q = np.empty((K, N), np.int8)
    lib.w4o_quantize_int8(_ptr(W), K, N, _ptr(scale), _ptr(q))
    return scale, q


def permute_int8(q, K, N):
    """Page-1 int8 permute of q [K, N] into N*K interleaved bytes."""
    lib = _load()
    a = np.ascontiguousarray(q, dtype=np.int8)
    if a.shape != (K, N):
        raise ValueError("q must be [K, N]")
    if K % 64 or N % 2:
        raise ValueError("the int8 permute needs K % 64 == 0 and N % 2 == 0")
    out = np.zeros(N * K, np.uint8)
    if lib.w4o_permute_int8(_ptr(a), K, N, _ptr(out)) != 0:
        raise MemoryError("oracle permute could not allocate its stream")
    return out


def gemv_int8(q, scale, x_bits, cols=None):
    """d[c, n] = sum_k x[c, k] * q[k, n] * scale[n], in fp64.

    q: int8 [K, N]; scale: float32 [N]; x_bits: uint16 bf16 patterns [C, K].
    cols: optional (begin, end) column range; columns outside it are NaN.
    Returns (d, ref_abs), both float64 [C, N].
    """
    lib = _load()
    a = np.ascontiguousarray(q, dtype=np.int8)
    s = np.ascontiguousarray(scale, dtype=np.float32)
    xb = np.ascontiguousarray(x_bits, dtype=np.uint16)
    K, N = a.shape
    C = xb.shape[0] if xb.ndim == 2 else 1
    if xb.size != C * K or s.size != N:
        raise ValueError("shape mismatch")
    b, e = (0, N) if cols is None else cols
    d = np.full((C, N), np.nan)
    ref = np.full((C, N), np.nan)
    lib.w4o_gemv_int8(_ptr(a), _ptr(s), _ptr(xb), N, K, C, b, e, _ptr(d), _ptr(ref))
    return d, ref


# ---------------------------------------------------------------------------
# W4A8: activations as block_q8_1 in the PT plane layout
# ---------------------------------------------------------------------------

def quantize_q8_1_pt(x_bits):
    """x [C, K] (uint16 bf16 patterns, K % 128 == 0) -> uint8 [C, 144*K/128]:
    per vector, planes 0..7 of int8 qs and plane 8 of (d, s) half pairs."""
    lib = _load()
    xb = np.ascontiguousarray(x_bits, dtype=np.uint16)
    if xb.ndim == 1:
        xb = xb.reshape(1, -1)
    C, K = xb.shape
    if K % 128:
        raise ValueError("K must be a multiple of 128")
    pt = np.zeros((C, 144 * (K // 128)), np.uint8)
    lib.w4o_quantize_q8_1_pt(_ptr(xb), C, K, _ptr(pt))
    return pt


def gemv_w4a8(packed_weights, scale_bits, zero_bits, pt, K, rows=None):
    """W4A8 GEMV of the int4 row-layout weights (uint32 [N, K/8], bf16 scale
    and zero [N] as uint16 patterns) against PT activations (uint8
    [C, 144*K/128]).  Returns (d, ref_abs) float64 [C, N]."""
    lib = _load()
    qw = np.ascontiguousarray(packed_weights, dtype=np.uint32)
    N = qw.shape[0]
    if qw.shape[1] * 8 != K:
        raise ValueError("weights imply another K")
    s = np.ascontiguousarray(scale_bits, dtype=np.uint16)
    z = np.ascontiguousarray(zero_bits, dtype=np.uint16)
    p = np.ascontiguousarray(pt, dtype=np.uint8)
    if p.ndim == 1:
        p = p.reshape(1, -1)
    C = p.shape[0]
    if p.shape[1] != 144 * (K // 128):
        raise ValueError("pt must hold 144*K/128 bytes per vector")
    r0, r1 = (0, N) if rows is None else rows
    d = np.full((C, N), np.nan)
    ref = np.full((C, N), np.nan)
    lib.w4o_gemv_w4a8(_ptr(qw), _ptr(s), _ptr(z), _ptr(p), N, K, C, r0, r1, _ptr(d), _ptr(ref))
    return d, ref


def float_to_half(a):
    """fp32 array -> uint16 IEEE binary16 bit patterns, the conversion the
    block_q8_1 quantiser stores d and s with (round to nearest even)."""
    lib = _load()
    f = np.ascontiguousarray(a, dtype=np.float32).ravel()
    out = np.zeros(f.size, np.uint16)
    lib.w4o_float_to_half(_ptr(f), f.size, _ptr(out))
    return out.reshape(np.shape(a))


def half_to_double(h):
    """uint16 IEEE binary16 bit patterns -> float64 values (exact), the
    decoding the W4A8 GEMV reads d and s with."""
    lib = _load()
    b = np.ascontiguousarray(h, dtype=np.uint16).ravel()
    out = np.zeros(b.size, np.float64)
    lib.w4o_half_to_double(_ptr(b), b.size, _ptr(out))
    return out.reshape(np.shape(h))


# ---------------------------------------------------------------------------
# Ternary weights: PTQ1_0 blocks, PTQ1_1 superblocks, MMVQ
# ---------------------------------------------------------------------------

PTQ1_0_BYTES = 28
PTQ1_1_BYTES = 216
PTQ1_1_ESCAPE = 767


def ptq1_0_pack(trits, d_bits):
    """trits int8 [N, K] in {-1, 0, 1} (K % 128 == 0), d [N, K/128] half bit
    patterns -> uint8 [N, K/128, 28] PTQ1_0 blocks."""
    lib = _load()
    t = np.ascontiguousarray(trits, dtype=np.int8)
    N, K = t.shape
    if K % 128:
        raise ValueError("K must be a multiple of 128")
    d = np.ascontiguousarray(d_bits, dtype=np.uint16)
    if d.shape != (N, K // 128):
        raise ValueError("d must be [N, K/128]")
    out = np.zeros((N, K // 128, PTQ1_0_BYTES), np.uint8)
    if lib.w4o_ptq1_0_pack(_ptr(t), _ptr(d), N, K, _ptr(out)):
        raise ValueError("trits must lie in {-1, 0, 1}")
    return out


def ptq1_0_unpack(blocks):
    """uint8 [N, K/128, 28] -> (trits int8 [N, K], d uint16 [N, K/128])."""
    lib = _load()
    b = np.ascontiguousarray(blocks, dtype=np.uint8)
    N, bpr = b.shape[:2]
    K = 128 * bpr
    t = np.zeros((N, K), np.int8)
    d = np.zeros((N, bpr), np.uint16)
    lib.w4o_ptq1_0_unpack(_ptr(b), N, K, _ptr(t), _ptr(d))
    return t, d


class Ptq1_1:
    """A tensor in PTQ1_1 form: superblocks uint8 [N, ceil(K/1024), 216],
    the codebook uint8 [n_code, 8] and the escape table (esc_idx int64
    [n_esc] ascending superblock indices, esc_patt uint8 [n_esc, 8])."""

    def __init__(self, sblocks, codebook, esc_idx, esc_patt, K):
        self.sblocks, self.codebook, self.esc_idx, self.esc_patt, self.K = sblocks, codebook, esc_idx, esc_patt, K


def ptq1_1_encode(blocks):
    """PTQ1_0 blocks uint8 [N, K/128, 28] -> Ptq1_1 (codebook built from
    the tensor's own exponent patterns)."""
    lib = _load()
    b = np.ascontiguousarray(blocks, dtype=np.uint8)
    N, bpr = b.shape[:2]
    K = 128 * bpr
    sbpr = (bpr + 7) // 8
    code = np.zeros((PTQ1_1_ESCAPE, 8), np.uint8)
    n_code = lib.w4o_ptq1_1_codebook(_ptr(b), N, K, _ptr(code))
    if n_code < 0:
        raise MemoryError("codebook")
    out = np.zeros((N, sbpr, PTQ1_1_BYTES), np.uint8)
    cap = max(1, N * sbpr)
    esc_idx = np.zeros(cap, np.int64)
    esc_patt = np.zeros((cap, 8), np.uint8)
    n_esc = lib.w4o_ptq1_1_encode(_ptr(b), N, K, _ptr(code), n_code, _ptr(out), _ptr(esc_idx), _ptr(esc_patt), cap)
    if n_esc == -1:
        raise ValueError("PTQ1_1 stores no sign: every d must be non-negative")
    if n_esc < 0:
        raise RuntimeError("escape table overflow")
    return Ptq1_1(out, code[:n_code].copy(), esc_idx[:n_esc].copy(), esc_patt[:n_esc].copy(), K)


def _ptq1_1_args(w):
    code = np.ascontiguousarray(w.codebook, dtype=np.uint8)
    ei = np.ascontiguousarray(w.esc_idx, dtype=np.int64)
    ep = np.ascontiguousarray(w.esc_patt, dtype=np.uint8)
    # keep at least one element so that every pointer is valid
    return (code if code.size else np.zeros((1, 8), np.uint8), code.shape[0],
            ei if ei.size else np.zeros(1, np.int64), ep if ep.size else np.zeros((1, 8), np.uint8), ei.shape[0])


def ptq1_1_unpack(w):
    """Ptq1_1 -> (trits int8 [N, K], d uint16 [N, K/128])."""
    lib = _load()
    sb = np.ascontiguousarray(w.sblocks, dtype=np.uint8)
    N, K = sb.shape[0], w.K
    code, n_code, ei, ep, n_esc = _ptq1_1_args(w)
    t = np.zeros((N, K), np.int8)
    d = np.zeros((N, K // 128), np.uint16)
    if lib.w4o_ptq1_1_unpack(_ptr(sb), N, K, _ptr(code), n_code, _ptr(ei), _ptr(ep), n_esc, _ptr(t), _ptr(d)):
        raise ValueError("a superblock's pattern index names no codebook entry or escape")
    return t, d


def mmvq_ptq1_0(blocks, pt, rows=None):
    """MMVQ of PTQ1_0 weights (uint8 [N, K/128, 28]) against x as block_q8_1
    in the PT layout (uint8 [C, 144 K/128]).  Returns (d, ref_abs) float64
    [C, N]; rows outside `rows` stay NaN."""
    lib = _load()
    b = np.ascontiguousarray(blocks, dtype=np.uint8)
    N, bpr = b.shape[:2]
    K = 128 * bpr
    p = np.ascontiguousarray(pt, dtype=np.uint8)
    if p.ndim == 1:
        p = p.reshape(1, -1)
    C = p.shape[0]
    if p.shape[1] != 144 * bpr:
        raise ValueError("pt must hold 144*K/128 bytes per vector")
    r0, r1 = (0, N) if rows is None else rows
    d = np.full((C, N), np.nan)
    ref = np.full((C, N), np.nan)
    lib.w4o_mmvq_ptq1_0(_ptr(b), _ptr(p), N, K, C, r0, r1, _ptr(d), _ptr(ref))
    return d, ref


def mmvq_ptq1_1(w, pt, rows=None):
    """MMVQ of a Ptq1_1 tensor against PT activations; as mmvq_ptq1_0."""
    lib = _load()
    sb = np.ascontiguousarray(w.sblocks, dtype=np.uint8)
    N, K = sb.shape[0], w.K
    code, n_code, ei, ep, n_esc = _ptq1_1_args(w)
    p = np.ascontiguousarray(pt, dtype=np.uint8)
    if p.ndim == 1:
        p = p.reshape(1, -1)
    C = p.shape[0]
    if p.shape[1] != 144 * (K // 128):
        raise ValueError("pt must hold 144*K/128 bytes per vector")
    r0, r1 = (0, N) if rows is None else rows
    d = np.full((C, N), np.nan)
    ref = np.full((C, N), np.nan)
    if lib.w4o_mmvq_ptq1_1(_ptr(sb), _ptr(code), n_code, _ptr(ei), _ptr(ep), n_esc, _ptr(p), N, K, C, r0, r1,
                           _ptr(d), _ptr(ref)):
        raise ValueError("a superblock's pattern index names no codebook entry or escape")
    return d, ref
