"""Host-only checks of the C ABI: the library builds, loads without a GPU,
exports every symbol include/w4.h declares, and rejects bad arguments on the
host before touching the device (no compute is launched here)."""
import ctypes
import os
import re

import pytest

from helpers import ROOT


def _lib():
    import __graft_entry__
    __graft_entry__._load_builder().build_library()
    from gemm_int4_dequant_gb300 import _lib as L
    return L.load(), L


def _declared_functions():
    src = open(os.path.join(ROOT, "include", "w4.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    names = re.findall(r"^\s*(?:const\s+)?[A-Za-z_][\w]*\s*\**\s+\**(\w+)\s*\(", src, flags=re.M)
    return sorted(set(names))


def test_header_declares_the_hot_path():
    names = _declared_functions()
    for fn in ("quantize_pack_int4", "permute_int4", "quantize_pack_permute_int4", "gemv_w4", "gemv_w4_permuted",
               "gemm_w4", "quantize_int8", "permute_int8", "gemv_w8", "gemm_w8", "gemm_w4_permuted", "quantize_q8_1_pt", "gemv_w4a8", "mmvq_ptq1_0",
               "mmvq_ptq1_1", "ptq1_1_codebook", "ptq1_1_encode",
               "w4_status_string", "w4_abi_version", "w4_device_error", "w4_selftest_wait_timeout",
               "w4_selftest_configure"):
        assert fn in names


def test_library_exports_every_declared_symbol():
    lib, _ = _lib()
    for fn in _declared_functions():
        assert hasattr(lib, fn), "libw4.so does not export %s" % fn
    assert lib.w4_abi_version() == 4
    assert lib.w4_status_string(-2) == b"illegal size or shape"
    assert lib.w4_status_string(-7) == b"input value outside the format's range"


def test_library_has_no_oracle_dependency():
    """The product library neither imports an oracle symbol nor needs the
    oracle's shared object (its dynamic symbol table and NEEDED entries),
    and no product source imports the oracle."""
    import shutil
    import subprocess
    from gemm_int4_dequant_gb300._lib import LIB_PATH
    if not (shutil.which("nm") and shutil.which("readelf")):
        pytest.skip("binutils not installed")
    undefined = subprocess.run(["nm", "-D", "--undefined-only", LIB_PATH], capture_output=True, text=True,
                               check=True).stdout
    defined = subprocess.run(["nm", "-D", "--defined-only", LIB_PATH], capture_output=True, text=True,
                             check=True).stdout
    assert "w4o_" not in undefined and "w4o_" not in defined, "product library references the oracle"
    dyn = subprocess.run(["readelf", "-d", LIB_PATH], capture_output=True, text=True, check=True).stdout
    needed = [l for l in dyn.splitlines() if "(NEEDED)" in l]
    assert needed and not any("oracle" in l for l in needed), needed
    pkg = os.path.join(ROOT, "gemm_int4_dequant_gb300")
    for dirpath, _, files in os.walk(pkg):
        for f in files:
            if f.endswith((".py", ".cu", ".cuh", ".h", ".cpp")):
                text = open(os.path.join(dirpath, f), errors="ignore").read()
                assert "import oracle" not in text and "from oracle" not in text and "w4_oracle" not in text, f


def test_argument_validation_happens_on_host():
    lib, L = _lib()
    A = 0x10000  # 16-byte aligned dummy addresses, never dereferenced
    odd = 0x10008
    # quantize_pack_int4
    assert lib.quantize_pack_int4(A, A, A, 3, 8, None) == L.W4_ERR_SHAPE
    assert lib.quantize_pack_int4(A, A, A, -2, 8, None) == L.W4_ERR_SHAPE
    assert lib.quantize_pack_int4(A, A, A, 4, 0, None) == L.W4_OK  # N == 0: no-op
    assert lib.quantize_pack_int4(None, A, A, 4, 8, None) == L.W4_ERR_NULL
    assert lib.quantize_pack_int4(odd, A, A, 4, 8, None) == L.W4_ERR_ALIGN
    # permute_int4
    assert lib.permute_int4(A, A, 96, 8, None) == L.W4_ERR_SHAPE
    assert lib.permute_int4(A, A, 64, 6, None) == L.W4_ERR_SHAPE
    assert lib.permute_int4(A, A, 0, 8, None) == L.W4_OK
    assert lib.permute_int4(A, None, 64, 8, None) == L.W4_ERR_NULL
    assert lib.permute_int4(A, odd, 64, 8, None) == L.W4_ERR_ALIGN
    # quantize_pack_permute_int4: the permute's K rule, N % 8, the K limit
    assert lib.quantize_pack_permute_int4(A, A, A, 96, 8, None) == L.W4_ERR_SHAPE         # K % 64
    assert lib.quantize_pack_permute_int4(A, A, A, 64, 12, None) == L.W4_ERR_SHAPE        # N % 8
    assert lib.quantize_pack_permute_int4(A, A, A, 26624 + 64, 8, None) == L.W4_ERR_SHAPE
    assert lib.quantize_pack_permute_int4(A, A, A, -64, 8, None) == L.W4_ERR_SHAPE
    assert lib.quantize_pack_permute_int4(A, A, A, 64, 0, None) == L.W4_OK                # N == 0
    assert lib.quantize_pack_permute_int4(None, A, A, 64, 8, None) == L.W4_ERR_NULL
    assert lib.quantize_pack_permute_int4(A, A, None, 64, 8, None) == L.W4_ERR_NULL
    assert lib.quantize_pack_permute_int4(A, odd, A, 64, 8, None) == L.W4_ERR_ALIGN
    # gemv_w4
    assert lib.gemv_w4(A, A, A, A, A, 16, 12, 1, L.W4_BF16, None) == L.W4_ERR_SHAPE
    assert lib.gemv_w4(A, A, A, A, A, 16, 16, 0, L.W4_BF16, None) == L.W4_ERR_SHAPE
    assert lib.gemv_w4(A, A, A, A, A, 16, 16, 9, L.W4_BF16, None) == L.W4_ERR_SHAPE
    assert lib.gemv_w4(A, A, A, A, A, 16, 40960 + 8, 1, L.W4_BF16, None) == L.W4_ERR_SHAPE  # K limit
    assert lib.gemv_w4(A, A, A, A, A, 16, 16, 1, 7, None) == L.W4_ERR_DTYPE
    assert lib.gemv_w4(A, A, None, A, A, 16, 16, 1, L.W4_F32, None) == L.W4_ERR_NULL
    assert lib.gemv_w4(A, A, A, odd, A, 16, 16, 1, L.W4_F32, None) == L.W4_ERR_ALIGN
    assert lib.gemv_w4(A, A, A, A, A, 0, 16, 1, L.W4_F32, None) == L.W4_OK
    # gemv_w4_permuted: the permute's shape rules, C and the K limit
    assert lib.gemv_w4_permuted(A, A, A, A, 16, 96, 1, None) == L.W4_ERR_SHAPE       # K % 64
    assert lib.gemv_w4_permuted(A, A, A, A, 18, 128, 1, None) == L.W4_ERR_SHAPE      # N % 4
    assert lib.gemv_w4_permuted(A, A, A, A, 16, 128, 9, None) == L.W4_ERR_SHAPE
    assert lib.gemv_w4_permuted(A, A, A, A, 16, 40960 + 64, 1, None) == L.W4_ERR_SHAPE
    assert lib.gemv_w4_permuted(A, A, A, A, 0, 128, 1, None) == L.W4_OK
    assert lib.gemv_w4_permuted(A, None, A, A, 16, 128, 1, None) == L.W4_ERR_NULL
    assert lib.gemv_w4_permuted(odd, A, A, A, 16, 128, 1, None) == L.W4_ERR_ALIGN
    # int8 variant
    assert lib.quantize_int8(A, A, A, -1, 8, None) == L.W4_ERR_SHAPE
    assert lib.quantize_int8(A, A, A, 4, 0, None) == L.W4_OK
    assert lib.quantize_int8(A, None, A, 4, 8, None) == L.W4_ERR_NULL
    assert lib.quantize_int8(A, A, odd, 4, 8, None) == L.W4_ERR_ALIGN
    assert lib.permute_int8(A, A, 96, 8, None) == L.W4_ERR_SHAPE        # K % 64
    assert lib.permute_int8(A, A, 64, 7, None) == L.W4_ERR_SHAPE        # N % 2
    assert lib.permute_int8(A, A, 0, 8, None) == L.W4_OK
    assert lib.permute_int8(None, A, 64, 8, None) == L.W4_ERR_NULL
    assert lib.gemv_w8(A, A, A, A, 16, 64, 0, None) == L.W4_ERR_SHAPE
    assert lib.gemv_w8(A, A, A, A, 16, 64, 9, None) == L.W4_ERR_SHAPE
    assert lib.gemv_w8(A, A, A, A, 0, 64, 1, None) == L.W4_OK
    assert lib.gemv_w8(A, A, None, A, 16, 64, 1, None) == L.W4_ERR_NULL
    assert lib.gemv_w8(A, A, A, odd, 16, 64, 1, None) == L.W4_ERR_ALIGN
    # W4A8: the PT layout needs K % 128; x lives in shared memory
    assert lib.quantize_q8_1_pt(A, A, 1, 192, None) == L.W4_ERR_SHAPE
    assert lib.quantize_q8_1_pt(A, A, -1, 128, None) == L.W4_ERR_SHAPE
    assert lib.quantize_q8_1_pt(A, A, 0, 128, None) == L.W4_OK
    assert lib.quantize_q8_1_pt(A, A, 2, 0, None) == L.W4_OK
    assert lib.quantize_q8_1_pt(None, A, 1, 128, None) == L.W4_ERR_NULL
    assert lib.quantize_q8_1_pt(A, odd, 1, 128, None) == L.W4_ERR_ALIGN
    assert lib.gemv_w4a8(A, A, A, A, A, 16, 192, 1, None) == L.W4_ERR_SHAPE        # K % 128
    assert lib.gemv_w4a8(A, A, A, A, A, 16, 128, 0, None) == L.W4_ERR_SHAPE
    assert lib.gemv_w4a8(A, A, A, A, A, 16, 128, 9, None) == L.W4_ERR_SHAPE
    assert lib.gemv_w4a8(A, A, A, A, A, 16, 23168 + 128, 8, None) == L.W4_ERR_SHAPE  # x exceeds shared memory
    assert lib.gemv_w4a8(A, A, A, A, A, 0, 128, 1, None) == L.W4_OK
    assert lib.gemv_w4a8(A, A, None, A, A, 16, 128, 1, None) == L.W4_ERR_NULL
    assert lib.gemv_w4a8(A, A, A, odd, A, 16, 128, 1, None) == L.W4_ERR_ALIGN
    # mmvq_ptq1_0: whole 128-weight blocks; x in shared memory
    assert lib.mmvq_ptq1_0(A, A, A, 16, 192, 1, None) == L.W4_ERR_SHAPE
    assert lib.mmvq_ptq1_0(A, A, A, 16, 128, 0, None) == L.W4_ERR_SHAPE
    assert lib.mmvq_ptq1_0(A, A, A, 16, 128, 9, None) == L.W4_ERR_SHAPE
    assert lib.mmvq_ptq1_0(A, A, A, 16, 23168 + 128, 8, None) == L.W4_ERR_SHAPE
    assert lib.mmvq_ptq1_0(A, A, A, 0, 128, 1, None) == L.W4_OK
    assert lib.mmvq_ptq1_0(None, A, A, 16, 128, 1, None) == L.W4_ERR_NULL
    assert lib.mmvq_ptq1_0(A, A, odd, 16, 128, 1, None) == L.W4_ERR_ALIGN
    # mmvq_ptq1_1: codebook size, escape table, the codebook's share of shared memory
    assert lib.mmvq_ptq1_1(A, A, 768, A, A, 1, A, A, 16, 1024, 1, None) == L.W4_ERR_SHAPE
    assert lib.mmvq_ptq1_1(A, A, -1, A, A, 1, A, A, 16, 1024, 1, None) == L.W4_ERR_SHAPE
    assert lib.mmvq_ptq1_1(A, A, 10, A, A, -1, A, A, 16, 1024, 1, None) == L.W4_ERR_SHAPE
    assert lib.mmvq_ptq1_1(A, A, 10, A, A, 1, A, A, 16, 1000, 1, None) == L.W4_ERR_SHAPE
    assert lib.mmvq_ptq1_1(A, A, 10, A, A, 1, A, A, 16, 22528 + 128, 8, None) == L.W4_ERR_SHAPE
    assert lib.mmvq_ptq1_1(A, None, 10, A, A, 1, A, A, 16, 1024, 1, None) == L.W4_ERR_NULL
    assert lib.mmvq_ptq1_1(A, A, 10, None, A, 1, A, A, 16, 1024, 1, None) == L.W4_ERR_NULL
    assert lib.mmvq_ptq1_1(A, A, 10, odd, A, 1, A, A, 16, 1024, 1, None) == L.W4_ERR_ALIGN
    assert lib.mmvq_ptq1_1(A, A, 10, A, A, 1, A, A, 0, 1024, 1, None) == L.W4_OK
    # gemm_w8: the GEMM's tile rules
    assert lib.gemm_w8(A, A, A, A, 128, 256, 100, None) == L.W4_ERR_SHAPE
    assert lib.gemm_w8(A, A, A, A, 128, 250, 128, None) == L.W4_ERR_SHAPE
    assert lib.gemm_w8(A, None, A, A, 128, 256, 128, None) == L.W4_ERR_NULL
    assert lib.gemm_w8(A, A, odd, A, 128, 256, 128, None) == L.W4_ERR_ALIGN
    assert lib.gemm_w8(A, A, A, A, 0, 256, 128, None) == L.W4_OK
    # gemm_w4_permuted: the GEMM's tile rules
    assert lib.gemm_w4_permuted(A, A, A, A, 128, 256, 100, None) == L.W4_ERR_SHAPE
    assert lib.gemm_w4_permuted(A, A, A, A, 128, 264, 128, None) == L.W4_ERR_SHAPE
    assert lib.gemm_w4_permuted(A, None, A, A, 128, 256, 128, None) == L.W4_ERR_NULL
    assert lib.gemm_w4_permuted(odd, A, A, A, 128, 256, 128, None) == L.W4_ERR_ALIGN
    assert lib.gemm_w4_permuted(A, A, A, A, 0, 256, 128, None) == L.W4_OK
    # gemm_w4
    assert lib.gemm_w4(A, A, A, A, A, 128, 256, 100, None) == L.W4_ERR_SHAPE
    assert lib.gemm_w4(A, A, A, A, A, 128, 250, 128, None) == L.W4_ERR_SHAPE
    assert lib.gemm_w4(A, A, A, A, A, 128, 264, 128, None) == L.W4_ERR_SHAPE
    assert lib.gemm_w4(A, None, A, A, A, 128, 256, 128, None) == L.W4_ERR_NULL
    assert lib.gemm_w4(A, A, A, odd, A, 128, 256, 128, None) == L.W4_ERR_ALIGN
    assert lib.gemm_w4(A, A, A, A, A, 0, 256, 128, None) == L.W4_OK


def test_valid_call_without_gpu_reports_device_error():
    import torch
    if torch.cuda.is_available():
        pytest.skip("a GPU is present")
    lib, L = _lib()
    A = 0x10000
    assert lib.gemv_w4(A, A, A, A, A, 16, 16, 1, L.W4_F32, None) == L.W4_ERR_DEVICE


def test_binding_fails_loudly_without_library(tmp_path, monkeypatch):
    from gemm_int4_dequant_gb300 import _lib as L
    monkeypatch.setattr(L, "_lib", None)
    monkeypatch.setattr(L, "LIB_PATH", str(tmp_path / "missing.so"))
    with pytest.raises(ImportError):
        L.load()
