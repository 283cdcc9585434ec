"""Host-side arithmetic of bench.py (no GPU): algorithmic byte counts, the
roofline record and the source hash that keys the recorded ncu traffic."""
import os
import re
import shutil

import pytest

import bench


def test_gemv_bytes_decode():
    # N*K/2 weights + 2N*2 scale/zero + C*K*2 x + C*N*2 d
    assert bench.gemv_bytes(17280, 5120, 1) == 17280 * 5120 // 2 + 4 * 17280 + 2 * 5120 + 2 * 17280
    assert bench.gemv_bytes(17280, 5120, 1) == 44350720


def test_quant_bytes_one_pass_and_two_calls():
    K = N = 8192
    one = bench.quant_bytes(K, N, fused=True)
    assert one == 2 * K * N + K * N // 2 + 4 * N == 167804928
    # two calls also write the packed matrix and read it back
    assert bench.quant_bytes(K, N, fused=False) == one + K * N


def test_gemm_bytes_and_flops():
    assert bench.gemm_flops(8192, 8192, 8192) == 2 * 8192 ** 3
    assert bench.gemm_bytes(8192, 8192, 8192) == 302022656


def test_workloads_name_known_kinds():
    for name, cfg in bench.WORKLOADS.items():
        assert cfg["kind"] in ("gemv", "quant", "gemm", "gemv8", "quant8", "w4a8", "ptq1", "gemm8", "gemmp"), name
    assert set(bench.COMPONENTS) <= set(bench.WORKLOADS)
    assert bench.WORKLOADS["quant"]["fused"] and not bench.WORKLOADS["quant_2call"]["fused"]


class _Gemv:
    bytes = 44350720
    launches_per_step = 1


def test_roofline_record_hbm():
    peaks = {"hbm_gbs": 6772.5}
    r = bench.roofline(_Gemv(), 10e-6, peaks, "measured", "gemv", "decode")
    assert r["bound"] == "hbm" and r["unit"] == "GB/s"
    assert r["achieved"] == pytest.approx(4435.072)
    assert r["frac"] == pytest.approx(4435.072 / 6772.5)
    assert r["peak_nominal"] == 7900.0 and r["frac_nominal"] == pytest.approx(4435.072 / 7900.0)


def test_source_hash_ignores_comments_but_not_code(tmp_path, monkeypatch):
    src = tmp_path / "k.cu"
    src.write_text("// header\n__global__ void k(int* p) {\n  p[0] = 1; /* one */\n}\n")
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    h0 = bench.source_hash(["k.cu"])
    src.write_text("// another header\n__global__ void k(int* p) {\n    p[0] = 1;   // set\n}\n")
    assert bench.source_hash(["k.cu"]) == h0
    src.write_text("__global__ void k(int* p) {\n  p[0] = 2;\n}\n")
    assert bench.source_hash(["k.cu"]) != h0


def test_recorded_traffic_is_well_formed():
    """Every committed ncu summary records its traffic per launch and the hash
    of the code it measured; the bench reports that traffic while the hash is
    current and null once the code has changed (never a stale figure)."""
    for workload, kind in (("decode", "gemv"), ("c8_perm", "gemv"), ("quant", "quant"), ("gemm", "gemm")):
        text = open(os.path.join(bench.ROOT, "profiles", bench.PROFILE_FILES[workload])).read()
        m1 = re.search(r"traffic_bytes_per_launch:\s*([0-9.eE+]+)", text)
        m2 = re.search(r"kernel_source_sha256_16:\s*([0-9a-f]+)", text)
        assert m1 and float(m1.group(1)) > 0 and m2, workload
        t = bench.recorded_traffic(kind, workload)
        if m2.group(1) == bench.source_hash(bench.KERNEL_SOURCES[kind]):
            assert t == float(m1.group(1)), workload
        else:
            assert t is None, workload


def test_recorded_traffic_drops_on_code_change(tmp_path, monkeypatch):
    root = tmp_path / "repo"
    for rel in bench.KERNEL_SOURCES["gemv"]:
        dst = root / rel
        dst.parent.mkdir(parents=True, exist_ok=True)
        shutil.copy(os.path.join(bench.ROOT, rel), dst)
    monkeypatch.setattr(bench, "ROOT", str(root))
    prof = root / "profiles" / bench.PROFILE_FILES["decode"]
    prof.parent.mkdir(parents=True, exist_ok=True)
    prof.write_text("traffic_bytes_per_launch: 44383232\nkernel_source_sha256_16: %s\n"
                    % bench.source_hash(bench.KERNEL_SOURCES["gemv"]))
    assert bench.recorded_traffic("gemv", "decode") == 44383232
    f = root / bench.KERNEL_SOURCES["gemv"][0]
    f.write_text(f.read_text() + "\nstatic int changed_code = 1;\n")
    assert bench.recorded_traffic("gemv", "decode") is None


def test_w4a8_bytes():
    # weights + scale/zero + x + PT written and read + d
    N, K, C = 17280, 5120, 1
    assert bench.w4a8_bytes(N, K, C) == N * K // 2 + 4 * N + 2 * K + 2 * 144 * 40 + 2 * N


def test_ptq1_bytes():
    # 28-byte blocks + x + PT written and read + fp32 d
    N, K, C = 17280, 5120, 1
    assert bench.ptq1_bytes(N, K, C) == N * 40 * 28 + 2 * K + 2 * 144 * 40 + 4 * N


def test_reference_arm_runs_on_the_host_and_prints_the_contract_line():
    """`bench.py --impl reference` times the oracle on the host cores alone
    (no GPU) and prints one JSON line with the contract's keys."""
    import json
    import subprocess
    import sys
    r = subprocess.run([sys.executable, "bench.py", "--impl", "reference", "--steps", "1", "--warmup", "1",
                        "--cpu-seconds", "1"], cwd=bench.ROOT, capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1
    line = json.loads(lines[0])
    for key in ("impl", "metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better",
                "scaling", "vs_baseline", "dtype", "data", "config", "cpu_baseline", "e2e", "gpu_launches"):
        assert key in line, key
    assert line["impl"] == "reference" and line["gpu_launches"] == 0 and line["value"] > 0
    assert line["cpu_baseline"]["kind"] == "oracle" and line["cpu_baseline"]["cores"] >= 1
    assert line["e2e"]["h2d_bytes_per_step"] == 0 and line["config"]["workload"] == "decode"


def test_all_core_baseline_runs_the_oracle_in_threads():
    r = bench.cpu_baseline_all_cores("decode", budget_s=1.0)
    assert r["kind"] == "oracle" and r["unit"] == "GB/s" and r["value"] > 0
    assert r["cores"] == bench.host_threads() >= 1
    assert bench.cpu_baseline_all_cores("gemm", budget_s=0.1) is None


def test_matmul_context_bar_never_raises():
    """The cuBLAS context bar reports an error note instead of failing the
    run (here: no GPU for its CUDA events)."""
    import types

    import torch
    if torch.cuda.is_available():
        pytest.skip("a GPU is present")
    work = types.SimpleNamespace(B=torch.randint(0, 256, (32, 16), dtype=torch.uint8),
                                 A=torch.zeros((8, 64), dtype=torch.bfloat16),
                                 s=torch.ones(16, dtype=torch.bfloat16), z=torch.full((16,), 8.0, dtype=torch.bfloat16),
                                 M=8, flops=2 * 8 * 16 * 64)
    r = bench.torch_matmul_context(work, 3)
    assert r["value"] is None and "error" in r
