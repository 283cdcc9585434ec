"""ctypes loader for libw4.so, the library's C ABI (include/w4.h).

Argument marshalling only: every step of the computation runs in the CUDA
kernels behind these symbols.  If the shared object is missing the import
fails loudly; there is no fallback implementation.
"""
import ctypes
import os

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libw4.so")

W4_OK, W4_ERR_NULL, W4_ERR_SHAPE, W4_ERR_ALIGN, W4_ERR_DTYPE, W4_ERR_CUDA, W4_ERR_DEVICE = 0, -1, -2, -3, -4, -5, -6
W4_ERR_VALUE = -7
W4_F32, W4_BF16 = 0, 1

_lib = None


class W4Error(RuntimeError):
    def __init__(self, fn, status, msg):
        super().__init__("%s failed: %s (status %d)" % (fn, msg, status))
        self.status = status


def load():
    """Load libw4.so (once) and declare every exported signature."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(LIB_PATH):
        raise ImportError(
            "libw4.so is not built (expected at %s); run "
            "`python -c 'import __graft_entry__ as g; g.build()'`" % LIB_PATH)
    lib = ctypes.CDLL(LIB_PATH)
    P, I64, I = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int
    lib.w4_abi_version.argtypes = []
    lib.w4_abi_version.restype = I
    lib.w4_status_string.argtypes = [I]
    lib.w4_status_string.restype = ctypes.c_char_p
    lib.w4_device_error.argtypes = [P]
    lib.w4_device_error.restype = I
    lib.w4_selftest_wait_timeout.argtypes = [P, P]
    lib.w4_selftest_wait_timeout.restype = I
    lib.w4_selftest_configure.argtypes = [ctypes.c_longlong, I]
    lib.w4_selftest_configure.restype = I
    lib.quantize_pack_int4.argtypes = [P, P, P, I64, I64, P]
    lib.quantize_pack_int4.restype = I
    lib.permute_int4.argtypes = [P, P, I64, I64, P]
    lib.permute_int4.restype = I
    lib.quantize_pack_permute_int4.argtypes = [P, P, P, I64, I64, P]
    lib.quantize_pack_permute_int4.restype = I
    lib.gemv_w4.argtypes = [P, P, P, P, P, I64, I64, I64, I, P]
    lib.gemv_w4.restype = I
    lib.gemv_w4_permuted.argtypes = [P, P, P, P, I64, I64, I64, P]
    lib.gemv_w4_permuted.restype = I
    lib.gemm_w4.argtypes = [P, P, P, P, P, I64, I64, I64, P]
    lib.gemm_w4.restype = I
    lib.quantize_int8.argtypes = [P, P, P, I64, I64, P]
    lib.quantize_int8.restype = I
    lib.permute_int8.argtypes = [P, P, I64, I64, P]
    lib.permute_int8.restype = I
    lib.gemv_w8.argtypes = [P, P, P, P, I64, I64, I64, P]
    lib.gemv_w8.restype = I
    lib.gemm_w8.argtypes = [P, P, P, P, I64, I64, I64, P]
    lib.gemm_w8.restype = I
    lib.gemm_w4_permuted.argtypes = [P, P, P, P, I64, I64, I64, P]
    lib.gemm_w4_permuted.restype = I
    lib.quantize_q8_1_pt.argtypes = [P, P, I64, I64, P]
    lib.quantize_q8_1_pt.restype = I
    lib.gemv_w4a8.argtypes = [P, P, P, P, P, I64, I64, I64, P]
    lib.gemv_w4a8.restype = I
    lib.mmvq_ptq1_0.argtypes = [P, P, P, I64, I64, I64, P]
    lib.mmvq_ptq1_0.restype = I
    lib.mmvq_ptq1_1.argtypes = [P, P, I64, P, P, I64, P, P, I64, I64, I64, P]
    lib.mmvq_ptq1_1.restype = I
    lib.ptq1_1_codebook.argtypes = [P, I64, I64, P, P]
    lib.ptq1_1_codebook.restype = I
    lib.ptq1_1_encode.argtypes = [P, I64, I64, P, I64, P, P, P, I64, P]
    lib.ptq1_1_encode.restype = I
    _lib = lib
    return lib


def check(fn, status):
    if status != W4_OK:
        msg = load().w4_status_string(status).decode()
        raise W4Error(fn, status, msg)
