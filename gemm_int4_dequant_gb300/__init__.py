"""int4 weight-only GEMV / GEMM with fused dequantisation for GB300 (sm_103a).

Thin PyTorch-facing binding over the C ABI in include/w4.h.  Tensors are
only used as device memory: each function checks dtypes, shapes and
devices, allocates missing outputs with torch, and passes raw pointers and
the current CUDA stream to libw4.so.  The computation itself runs entirely
in the library's CUDA kernels; there is no CPU or eager fallback.

    quantize_pack_int4(W)               -> (packed [K/2, N] int8, scale [N] fp32)
    permute_int4(packed)                -> out [N*K/2] int8 (interleaved)
    quantize_pack_permute_int4(W)       -> (out [N*K/2] int8, scale [N] fp32), both in one pass
    gemv_w4(qweight, scale, zero, x)    -> d [C, N]
    gemv_w4_permuted(permuted, scale, x) -> d [C, N] bf16 (over permute_int4's output)
    gemm_w4(A, B, scale, zero)          -> C [M, N] bf16
    quantize_int8(W)                    -> (q [K, N] int8, scale [N] fp32)
    permute_int8(q)                     -> out [N*K] int8 (interleaved)
    gemv_w8(q, scale, x)                -> d [C, N] bf16
    gemm_w8(A, q, scale)                -> C [M, N] bf16 (bf16 x int8 on the tensor cores)
    gemm_w4_permuted(A, permuted, scale) -> C [M, N] bf16 (over permute_int4's output)
    quantize_q8_1_pt(x)                 -> pt [C, 144*K/128] uint8 (block_q8_1 in PT planes)
    gemv_w4a8(qweight, scale, zero, pt) -> d [C, N] bf16 (int4 weights x int8 activations)
    mmvq_ptq1_0(blocks, pt)             -> d [C, N] fp32 (ternary PTQ1_0 weights x int8 activations)
    mmvq_ptq1_1(sblocks, codebook, esc_idx, esc_patt, pt, K) -> d [C, N] fp32 (PTQ1_1 superblocks)
    ptq1_1_encode(blocks)               -> (sblocks, codebook, esc_idx, esc_patt): PTQ1_0 -> PTQ1_1 (host)
"""
import torch

from . import _lib
from ._lib import W4Error, W4_BF16, W4_F32

__all__ = ["quantize_pack_int4", "permute_int4", "quantize_pack_permute_int4", "gemv_w4", "gemv_w4_permuted", "gemm_w4",
           "quantize_int8", "permute_int8", "gemv_w8", "gemm_w8", "gemm_w4_permuted", "quantize_q8_1_pt", "gemv_w4a8", "mmvq_ptq1_0", "mmvq_ptq1_1",
           "ptq1_1_encode", "device_error", "W4Error"]

_lib.load()  # fail loudly at import if the CUDA library is missing


def _stream(stream):
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes_ptr(stream.cuda_stream)


def ctypes_ptr(v):
    return int(v) if v else None


def _need(t, name, dtypes, ndim=None):
    if not isinstance(t, torch.Tensor):
        raise TypeError("%s must be a torch.Tensor" % name)
    if t.device.type != "cuda":
        raise ValueError("%s must be a CUDA tensor" % name)
    if t.dtype not in dtypes:
        raise TypeError("%s has dtype %s, expected one of %s" % (name, t.dtype, dtypes))
    if ndim is not None and t.dim() != ndim:
        raise ValueError("%s must have %d dims" % (name, ndim))
    if not t.is_contiguous():
        raise ValueError("%s must be contiguous" % name)


def quantize_pack_int4(W, packed=None, scale=None, stream=None):
    """Symmetric per-column int4 quantisation of W [K, N] bf16 plus the
    column pack (two rows per byte, even row in the low nibble)."""
    _need(W, "W", (torch.bfloat16,), 2)
    K, N = W.shape
    if packed is None:
        packed = torch.empty((K // 2, N), dtype=torch.int8, device=W.device)
    if scale is None:
        scale = torch.empty((N,), dtype=torch.float32, device=W.device)
    _need(packed, "packed", (torch.int8, torch.uint8))
    _need(scale, "scale", (torch.float32,))
    if packed.numel() != (K // 2) * N or scale.numel() != N:
        raise ValueError("output shapes do not match W")
    st = _lib.load().quantize_pack_int4(W.data_ptr(), packed.data_ptr(), scale.data_ptr(), K, N, _stream(stream))
    _lib.check("quantize_pack_int4", st)
    return packed, scale


def quantize_pack_permute_int4(W, out=None, scale=None, stream=None):
    """quantize_pack_int4 then permute_int4 in one pass over W [K, N] bf16
    (K % 64 == 0, N % 8 == 0, K <= 26624): the permuted N*K/2 bytes and the
    fp32 scale, bit-exact with the two separate calls."""
    _need(W, "W", (torch.bfloat16,), 2)
    K, N = W.shape
    if out is None:
        out = torch.empty((N * (K // 2),), dtype=torch.int8, device=W.device)
    if scale is None:
        scale = torch.empty((N,), dtype=torch.float32, device=W.device)
    _need(out, "out", (torch.int8, torch.uint8))
    _need(scale, "scale", (torch.float32,))
    if out.numel() != N * (K // 2) or scale.numel() != N:
        raise ValueError("output shapes do not match W")
    st = _lib.load().quantize_pack_permute_int4(W.data_ptr(), out.data_ptr(), scale.data_ptr(), K, N,
                                                _stream(stream))
    _lib.check("quantize_pack_permute_int4", st)
    return out, scale


def permute_int4(packed, out=None, stream=None):
    """Page-1 int4 interleave permute of packed [K/2, N] into N*K/2 bytes."""
    _need(packed, "packed", (torch.int8, torch.uint8), 2)
    Kp, N = packed.shape
    K = 2 * Kp
    if out is None:
        out = torch.empty((N * Kp,), dtype=packed.dtype, device=packed.device)
    _need(out, "out", (torch.int8, torch.uint8))
    if out.numel() != N * Kp:
        raise ValueError("out must hold N*K/2 bytes")
    st = _lib.load().permute_int4(packed.data_ptr(), out.data_ptr(), K, N, _stream(stream))
    _lib.check("permute_int4", st)
    return out


def gemv_w4(qweight, scale, zero, x, out=None, stream=None):
    """d[c, r] = sum_k (q[r, k] - zero[r]) * scale[r] * x[c, k].

    qweight: int32/uint32 [N, K/8] packed words; scale, zero: [N]; x: [C, K]
    (C <= 8) -- scale, zero, x and the output share one dtype, fp32 or bf16.
    """
    _need(qweight, "qweight", (torch.int32, torch.uint32) if hasattr(torch, "uint32") else (torch.int32,), 2)
    _need(x, "x", (torch.float32, torch.bfloat16))
    dt = x.dtype
    _need(scale, "scale", (dt,), 1)
    _need(zero, "zero", (dt,), 1)
    xx = x if x.dim() == 2 else x.reshape(1, -1)
    N, K = qweight.shape[0], qweight.shape[1] * 8
    C = xx.shape[0]
    if xx.shape[1] != K or scale.numel() != N or zero.numel() != N:
        raise ValueError("shape mismatch: qweight %s, x %s, scale %s" % (tuple(qweight.shape), tuple(x.shape), tuple(scale.shape)))
    if out is None:
        out = torch.empty((C, N), dtype=dt, device=x.device)
    _need(out, "out", (dt,))
    if out.numel() != C * N:
        raise ValueError("out must hold C*N elements")
    st = _lib.load().gemv_w4(qweight.data_ptr(), scale.data_ptr(), zero.data_ptr(), xx.data_ptr(), out.data_ptr(),
                             N, K, C, W4_F32 if dt == torch.float32 else W4_BF16, _stream(stream))
    _lib.check("gemv_w4", st)
    return out


def gemv_w4_permuted(permuted, scale, x, out=None, stream=None):
    """d[c, n] = sum_k q[k, n] * scale[n] * x[c, k] over permute_int4's output.

    permuted: int8/uint8 with N*K/2 bytes; scale: fp32 [N] (quantize_pack_int4's);
    x: bf16 [C, K] (C <= 8).  Returns bf16 [C, N].
    """
    _need(permuted, "permuted", (torch.int8, torch.uint8))
    _need(scale, "scale", (torch.float32,), 1)
    _need(x, "x", (torch.bfloat16,))
    xx = x if x.dim() == 2 else x.reshape(1, -1)
    C, K = xx.shape
    N = scale.numel()
    if permuted.numel() * 2 != N * K:
        raise ValueError("permuted must hold N*K/2 bytes (N = scale.numel(), K = x.shape[-1])")
    if out is None:
        out = torch.empty((C, N), dtype=torch.bfloat16, device=x.device)
    _need(out, "out", (torch.bfloat16,))
    if out.numel() != C * N:
        raise ValueError("out must hold C*N elements")
    st = _lib.load().gemv_w4_permuted(permuted.data_ptr(), scale.data_ptr(), xx.data_ptr(), out.data_ptr(),
                                      N, K, C, _stream(stream))
    _lib.check("gemv_w4_permuted", st)
    return out


def gemm_w4(A, B, scale, zero, out=None, stream=None):
    """C[m, n] = scale[n] * sum_k A[m, k] * (u[k, n] - zero[n]); A bf16 [M, K],
    B int8/uint8 [K/2, N] (low nibble = even k, unsigned), scale/zero bf16 [N]."""
    _need(A, "A", (torch.bfloat16,), 2)
    _need(B, "B", (torch.int8, torch.uint8), 2)
    _need(scale, "scale", (torch.bfloat16,), 1)
    _need(zero, "zero", (torch.bfloat16,), 1)
    M, K = A.shape
    if B.shape[0] * 2 != K:
        raise ValueError("B must be [K/2, N]")
    N = B.shape[1]
    if scale.numel() != N or zero.numel() != N:
        raise ValueError("scale/zero must be [N]")
    if out is None:
        out = torch.empty((M, N), dtype=torch.bfloat16, device=A.device)
    _need(out, "out", (torch.bfloat16,))
    if out.numel() != M * N:
        raise ValueError("out must hold M*N elements")
    st = _lib.load().gemm_w4(A.data_ptr(), B.data_ptr(), scale.data_ptr(), zero.data_ptr(), out.data_ptr(),
                             M, N, K, _stream(stream))
    _lib.check("gemm_w4", st)
    return out


def quantize_int8(W, q=None, scale=None, stream=None):
    """Symmetric per-column int8 quantisation of W [K, N] bf16."""
    _need(W, "W", (torch.bfloat16,), 2)
    K, N = W.shape
    if q is None:
        q = torch.empty((K, N), dtype=torch.int8, device=W.device)
    if scale is None:
        scale = torch.empty((N,), dtype=torch.float32, device=W.device)
    _need(q, "q", (torch.int8,))
    _need(scale, "scale", (torch.float32,))
    if q.numel() != K * N or scale.numel() != N:
        raise ValueError("output shapes do not match W")
    st = _lib.load().quantize_int8(W.data_ptr(), q.data_ptr(), scale.data_ptr(), K, N, _stream(stream))
    _lib.check("quantize_int8", st)
    return q, scale


def permute_int8(q, out=None, stream=None):
    """Page-1 int8 interleave permute of q [K, N] into N*K bytes."""
    _need(q, "q", (torch.int8, torch.uint8), 2)
    K, N = q.shape
    if out is None:
        out = torch.empty((N * K,), dtype=q.dtype, device=q.device)
    _need(out, "out", (torch.int8, torch.uint8))
    if out.numel() != N * K:
        raise ValueError("out must hold N*K bytes")
    st = _lib.load().permute_int8(q.data_ptr(), out.data_ptr(), K, N, _stream(stream))
    _lib.check("permute_int8", st)
    return out


def gemv_w8(q, scale, x, out=None, stream=None):
    """d[c, n] = sum_k q[k, n] * scale[n] * x[c, k]; q int8 [K, N], scale fp32 [N],
    x bf16 [C, K] (C <= 8).  Returns bf16 [C, N]."""
    _need(q, "q", (torch.int8,), 2)
    _need(scale, "scale", (torch.float32,), 1)
    _need(x, "x", (torch.bfloat16,))
    xx = x if x.dim() == 2 else x.reshape(1, -1)
    K, N = q.shape
    C = xx.shape[0]
    if xx.shape[1] != K or scale.numel() != N:
        raise ValueError("shape mismatch")
    if out is None:
        out = torch.empty((C, N), dtype=torch.bfloat16, device=x.device)
    _need(out, "out", (torch.bfloat16,))
    if out.numel() != C * N:
        raise ValueError("out must hold C*N elements")
    st = _lib.load().gemv_w8(q.data_ptr(), scale.data_ptr(), xx.data_ptr(), out.data_ptr(), N, K, C,
                             _stream(stream))
    _lib.check("gemv_w8", st)
    return out


def gemm_w8(A, q, scale, out=None, stream=None):
    """C[m, n] = scale[n] * sum_k A[m, k] q[k, n]: A bf16 [M, K] (K % 64 == 0),
    q int8 [K, N] (N % 16 == 0), scale fp32 [N].  Returns bf16 [M, N]."""
    _need(A, "A", (torch.bfloat16,), 2)
    _need(q, "q", (torch.int8,), 2)
    _need(scale, "scale", (torch.float32,), 1)
    M, K = A.shape
    if q.shape[0] != K or scale.numel() != q.shape[1]:
        raise ValueError("shape mismatch")
    N = q.shape[1]
    if out is None:
        out = torch.empty((M, N), dtype=torch.bfloat16, device=A.device)
    _need(out, "out", (torch.bfloat16,))
    if out.numel() != M * N:
        raise ValueError("out must hold M*N elements")
    st = _lib.load().gemm_w8(A.data_ptr(), q.data_ptr(), scale.data_ptr(), out.data_ptr(), M, N, K, _stream(stream))
    _lib.check("gemm_w8", st)
    return out


def gemm_w4_permuted(A, permuted, scale, out=None, stream=None):
    """C[m, n] = scale[n] * sum_k A[m, k] q[k, n] with the int4 weights read
    straight from permute_int4's output (N*K/2 bytes): A bf16 [M, K]
    (K % 64 == 0), scale fp32 [N] (N % 16 == 0).  Returns bf16 [M, N]."""
    _need(A, "A", (torch.bfloat16,), 2)
    _need(permuted, "permuted", (torch.int8, torch.uint8))
    _need(scale, "scale", (torch.float32,), 1)
    M, K = A.shape
    N = scale.numel()
    if permuted.numel() != N * (K // 2):
        raise ValueError("permuted must hold N*K/2 bytes")
    if out is None:
        out = torch.empty((M, N), dtype=torch.bfloat16, device=A.device)
    _need(out, "out", (torch.bfloat16,))
    if out.numel() != M * N:
        raise ValueError("out must hold M*N elements")
    st = _lib.load().gemm_w4_permuted(A.data_ptr(), permuted.data_ptr(), scale.data_ptr(), out.data_ptr(), M, N, K,
                                      _stream(stream))
    _lib.check("gemm_w4_permuted", st)
    return out


def quantize_q8_1_pt(x, out=None, stream=None):
    """x bf16 [C, K] (K % 128 == 0) as block_q8_1 in the PT planes: uint8
    [C, 144*K/128] per vector (qs planes 0..7, the (d, s) halves in plane 8)."""
    _need(x, "x", (torch.bfloat16,))
    xx = x if x.dim() == 2 else x.reshape(1, -1)
    C, K = xx.shape
    if out is None:
        out = torch.empty((C, 144 * (K // 128)), dtype=torch.uint8, device=x.device)
    _need(out, "out", (torch.uint8, torch.int8))
    if out.numel() != C * 144 * (K // 128):
        raise ValueError("out must hold C*144*K/128 bytes")
    st = _lib.load().quantize_q8_1_pt(xx.data_ptr(), out.data_ptr(), C, K, _stream(stream))
    _lib.check("quantize_q8_1_pt", st)
    return out


def gemv_w4a8(qweight, scale, zero, pt, out=None, stream=None):
    """d[c, r] = scale[r] * sum_b (d_b * sum_{k in b} q[r, k] qs[c, k] - zero[r] s_b):
    gemv_w4's packed words (int32 [N, K/8]), bf16 scale and zero [N], and x as
    quantize_q8_1_pt's output (uint8 [C, 144*K/128], C <= 8).  Returns bf16 [C, N]."""
    _need(qweight, "qweight", (torch.int32, torch.uint32) if hasattr(torch, "uint32") else (torch.int32,), 2)
    _need(scale, "scale", (torch.bfloat16,), 1)
    _need(zero, "zero", (torch.bfloat16,), 1)
    _need(pt, "pt", (torch.uint8, torch.int8))
    N, K = qweight.shape[0], qweight.shape[1] * 8
    pp = pt if pt.dim() == 2 else pt.reshape(1, -1)
    C = pp.shape[0]
    if K % 128 or pp.shape[1] != 144 * (K // 128) or scale.numel() != N or zero.numel() != N:
        raise ValueError("shape mismatch")
    if out is None:
        out = torch.empty((C, N), dtype=torch.bfloat16, device=qweight.device)
    _need(out, "out", (torch.bfloat16,))
    if out.numel() != C * N:
        raise ValueError("out must hold C*N elements")
    st = _lib.load().gemv_w4a8(qweight.data_ptr(), scale.data_ptr(), zero.data_ptr(), pp.data_ptr(), out.data_ptr(),
                               N, K, C, _stream(stream))
    _lib.check("gemv_w4a8", st)
    return out


def mmvq_ptq1_0(blocks, pt, out=None, stream=None):
    """d[c, r] = sum_k W[r, k] x[c, k] for ternary W in PTQ1_0 blocks (uint8
    [N, K/128, 28], or [N, 28*K/128]) and x as quantize_q8_1_pt's output
    (uint8 [C, 144*K/128], C <= 8).  Returns fp32 [C, N]."""
    _need(blocks, "blocks", (torch.uint8, torch.int8))
    _need(pt, "pt", (torch.uint8, torch.int8))
    N = blocks.shape[0]
    pp = pt if pt.dim() == 2 else pt.reshape(1, -1)
    C = pp.shape[0]
    per_row = blocks.numel() // max(N, 1)
    if N and (blocks.numel() % N or per_row % 28):
        raise ValueError("blocks must hold N rows of 28-byte blocks")
    K = 128 * (per_row // 28) if N else 128 * (pp.shape[1] // 144)
    if pp.shape[1] != 144 * (K // 128):
        raise ValueError("pt must hold 144*K/128 bytes per vector")
    if out is None:
        out = torch.empty((C, N), dtype=torch.float32, device=pt.device)
    _need(out, "out", (torch.float32,))
    if out.numel() != C * N:
        raise ValueError("out must hold C*N elements")
    st = _lib.load().mmvq_ptq1_0(blocks.data_ptr(), pp.data_ptr(), out.data_ptr(), N, K, C, _stream(stream))
    _lib.check("mmvq_ptq1_0", st)
    return out


def mmvq_ptq1_1(sblocks, codebook, esc_idx, esc_patt, pt, K, out=None, stream=None):
    """mmvq_ptq1_0's product over PTQ1_1 superblocks (uint8 [N, ceil(K/1024),
    216]) with their codebook (uint8 [n_code, 8]) and escape table (int64
    [n_esc] ascending superblock indices, uint8 [n_esc, 8]); x as
    quantize_q8_1_pt's output.  Returns fp32 [C, N]."""
    for t, name in ((sblocks, "sblocks"), (codebook, "codebook"), (esc_patt, "esc_patt"), (pt, "pt")):
        _need(t, name, (torch.uint8, torch.int8))
    _need(esc_idx, "esc_idx", (torch.int64,))
    N = sblocks.shape[0]
    pp = pt if pt.dim() == 2 else pt.reshape(1, -1)
    C = pp.shape[0]
    if K % 128 or pp.shape[1] != 144 * (K // 128) or sblocks.numel() != N * -(-K // 1024) * 216:
        raise ValueError("shape mismatch")
    n_code, n_esc = codebook.numel() // 8, esc_idx.numel()
    if codebook.numel() % 8 or esc_patt.numel() != 8 * n_esc:
        raise ValueError("codebook and escape patterns hold 8 exponents each")
    if out is None:
        out = torch.empty((C, N), dtype=torch.float32, device=pt.device)
    _need(out, "out", (torch.float32,))
    if out.numel() != C * N:
        raise ValueError("out must hold C*N elements")
    st = _lib.load().mmvq_ptq1_1(sblocks.data_ptr(), codebook.data_ptr() if n_code else None, n_code,
                                 esc_idx.data_ptr() if n_esc else None, esc_patt.data_ptr() if n_esc else None, n_esc,
                                 pp.data_ptr(), out.data_ptr(), N, K, C, _stream(stream))
    _lib.check("mmvq_ptq1_1", st)
    return out


def ptq1_1_encode(blocks):
    """Convert ternary PTQ1_0 blocks (host uint8 [N, K/128, 28], numpy or a
    CPU tensor) into PTQ1_1 superblocks with the tensor's own codebook.
    Runs on the host.  Returns numpy (sblocks uint8 [N, ceil(K/1024), 216],
    codebook uint8 [n_code, 8], esc_idx int64 [n_esc], esc_patt uint8
    [n_esc, 8])."""
    import ctypes
    import numpy as np
    b = blocks.numpy() if isinstance(blocks, torch.Tensor) else blocks
    b = np.ascontiguousarray(b, dtype=np.uint8)
    if b.ndim != 3 or b.shape[2] != 28:
        raise ValueError("blocks must be [N, K/128, 28] bytes")
    N, bpr = b.shape[:2]
    K = 128 * bpr
    sbpr = -(-bpr // 8)
    lib = _lib.load()
    ptr = lambda a: a.ctypes.data_as(ctypes.c_void_p)
    code = np.zeros((767, 8), np.uint8)
    n_code = ctypes.c_int64(0)
    _lib.check("ptq1_1_codebook", lib.ptq1_1_codebook(ptr(b), N, K, ptr(code), ctypes.byref(n_code)))
    sblocks = np.zeros((N, sbpr, 216), np.uint8)
    cap = max(1, N * sbpr)
    esc_idx = np.zeros(cap, np.int64)
    esc_patt = np.zeros((cap, 8), np.uint8)
    n_esc = ctypes.c_int64(0)
    _lib.check("ptq1_1_encode", lib.ptq1_1_encode(ptr(b), N, K, ptr(code), n_code.value, ptr(sblocks), ptr(esc_idx),
                                                  ptr(esc_patt), cap, ctypes.byref(n_esc)))
    n = n_esc.value
    return sblocks, code[:n_code.value].copy(), esc_idx[:n].copy(), esc_patt[:n].copy()


def device_error(stream=None):
    """Synchronise and return/clear the library's device-side error code."""
    return _lib.load().w4_device_error(_stream(stream))
