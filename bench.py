"""Benchmark of the int4 weight-only hot path on GB300.

Default workload: the decode GEMV, N=17280 rows, K=5120, C=1 (bf16 x,
scale, zero and output; uint4 weights packed eight per uint32), the
configuration the headline metric "int4 W-only GEMV HBM GB/s" is quoted
on.  One step = one gemv_w4 call on one batch.  The line also carries the
other kernels of the hot path as components: the small-batch GEMVs (C = 4,
8), the same GEMVs over permute_int4's output (gemv_w4_permuted),
quantise+pack+permute of an 8192x8192 bf16 weight (one pass,
quantize_pack_permute_int4; and as the two calls quantize_pack_int4 +
permute_int4), and the 8192^3 bf16 x int4 dequant GEMM (TFLOP/s).

Timing: inputs resident in HBM; weights rotate through enough copies that
the working set is more than twice the L2 (no step reads a weight copy the
L2 still holds); the K timed steps are one CUDA-graph replay bracketed by a
barrier and a device synchronise, timed with CUDA events on the launching
stream; max over ranks.  `e2e` repeats the measurement through the public
Python API with x copied from pinned host memory and d copied back every
step (weights stay resident, as in a decode loop).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                    [--workload decode|c4|c8|c4s|c8s|c4_perm|c8_perm|c4s_perm|c8s_perm|gemm|quant|quant_2call
                                |w8_decode|w8_quant]
                    [--no-components]
"""
import argparse
import hashlib
import json
import os
import re
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402
import torch  # noqa: E402

import synth  # noqa: E402

METRIC = "int4 W-only GEMV HBM GB/s (% of GB300 peak); dequant-GEMM TFLOP/s"
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
# GB300's nominal figures (HBM3e 7.9 TB/s; 2.25 PFLOP/s dense bf16), reported beside the measured peaks
NOMINAL_PEAKS = {"hbm_gbs": 7900.0, "bf16_tflops": 2250.0}

WORKLOADS = {
    "decode": dict(kind="gemv", N=17280, K=5120, C=1),
    "c4": dict(kind="gemv", N=5120, K=17280, C=4),
    "c8": dict(kind="gemv", N=5120, K=17280, C=8),
    "c4s": dict(kind="gemv", N=6144, K=5120, C=4),
    "c8s": dict(kind="gemv", N=6144, K=5120, C=8),
    # quantise + pack + permute of one 8192x8192 weight: the one-pass call,
    # and the two separate calls (packed matrix stored, then permuted)
    "quant": dict(kind="quant", K=8192, N=8192, fused=True),
    "quant_2call": dict(kind="quant", K=8192, N=8192, fused=False),
    "gemm": dict(kind="gemm", M=8192, N=8192, K=8192),
    # the small-batch GEMVs over permute_int4's output (gemv_w4_permuted;
    # fp32 scale per column and no zero point: the same 4N bytes)
    "c4_perm": dict(kind="gemv", N=5120, K=17280, C=4, perm=True),
    "c8_perm": dict(kind="gemv", N=5120, K=17280, C=8, perm=True),
    "c4s_perm": dict(kind="gemv", N=6144, K=5120, C=4, perm=True),
    "c8s_perm": dict(kind="gemv", N=6144, K=5120, C=8, perm=True),
    # the int8 weight-only variant: GEMV over quantize_int8's matrix, and
    # quantize_int8 + permute_int8 of one 8192x8192 weight
    "w8_decode": dict(kind="gemv8", N=17280, K=5120, C=1),
    "w8_quant": dict(kind="quant8", K=8192, N=8192),
    "w8_gemm": dict(kind="gemm8", M=8192, N=8192, K=8192),
    # the GEMM over permute_int4's output (fp32 scale, no zero point)
    "gemm_perm": dict(kind="gemmp", M=8192, N=8192, K=8192),
    # W4A8: x quantised to block_q8_1 in the PT planes, then the int4 GEMV
    # with integer dots (two kernels per step)
    "w4a8_decode": dict(kind="w4a8", N=17280, K=5120, C=1),
    "w4a8_c8": dict(kind="w4a8", N=5120, K=17280, C=8),
    # ternary PTQ1_0 weights: x quantised to block_q8_1 / PT, then the MMVQ
    "ptq1_decode": dict(kind="ptq1", N=17280, K=5120, C=1),
    "ptq1_c8": dict(kind="ptq1", N=5120, K=17280, C=8),
    # the same weights as PTQ1_1 superblocks (the library's host conversion)
    "ptq1_1_decode": dict(kind="ptq1", N=17280, K=5120, C=1, superblocks=True),
}
COMPONENTS = ["c4", "c8", "c4s", "c8s", "c4_perm", "c8_perm", "c4s_perm", "c8s_perm", "quant", "quant_2call", "gemm",
              "w8_decode", "w8_quant", "w8_gemm", "gemm_perm", "w4a8_decode", "w4a8_c8",
              "ptq1_decode", "ptq1_c8", "ptq1_1_decode"]


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return d, "measured"
    return dict(FALLBACK_PEAKS), "fallback"


# ---------------------------------------------------------------------------
# algorithmic bytes / flops per unit of work
# ---------------------------------------------------------------------------

def gemv_bytes(N, K, C, esz=2):
    # packed weights + scale + zero + x + d
    return N * K // 2 + 2 * N * esz + C * K * esz + C * N * esz


def quant_bytes(K, N, fused=True):
    # one pass: read W, write the permuted matrix + scale; two calls add the
    # packed matrix's write and re-read
    one_pass = K * N * 2 + K * N // 2 + 4 * N
    return one_pass if fused else one_pass + 2 * (K * N // 2)


def gemv8_bytes(N, K, C):
    # int8 weights + fp32 scale + x + d
    return N * K + 4 * N + 2 * C * K + 2 * C * N


def quant8_bytes(K, N):
    # quantize_int8: read W, write q + scale; permute_int8: read + write q
    return (2 * K * N + K * N + 4 * N) + 2 * K * N


def w4a8_bytes(N, K, C):
    # weights + bf16 scale and zero + x read by the quantiser + the PT
    # activations written and read back + d
    return N * K // 2 + 4 * N + 2 * C * K + 2 * C * 144 * (K // 128) + 2 * C * N


def ptq1_bytes(N, K, C, superblocks=False):
    # PTQ1_0 blocks (or PTQ1_1 superblocks) + x read by the quantiser + the
    # PT activations written and read back + d (fp32)
    w = N * -(-K // 1024) * 216 if superblocks else N * (K // 128) * 28
    return w + 2 * C * K + 2 * C * 144 * (K // 128) + 4 * C * N


def gemm_bytes(M, N, K):
    return M * K * 2 + K * N // 2 + M * N * 2 + 4 * N


def gemm_flops(M, N, K):
    return 2 * M * N * K


# ---------------------------------------------------------------------------
# distributed plumbing
# ---------------------------------------------------------------------------

def dist_setup(gpus):
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    else:
        torch.cuda.set_device(0)
    return world, rank


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(v, world, device="cuda"):
    """The slowest rank's time (every rank gets it); device is where the
    reduction tensor lives (cuda under NCCL, cpu under gloo)."""
    if world == 1:
        return v
    import torch.distributed as dist
    t = torch.tensor([v], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_rate(per_rank_rate_at_max_time, world):
    """Whole-job throughput: every rank processes the same units (replicas,
    weak scaling), all within the slowest rank's time."""
    return per_rank_rate_at_max_time * world


# ---------------------------------------------------------------------------
# clocks during load
# ---------------------------------------------------------------------------

CLOCK_QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
               "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
               "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")


class ClockSampler:
    def __init__(self, gpu_index):
        self.gpu = gpu_index
        self.proc = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), "--query-gpu=" + CLOCK_QUERY, "--format=csv,noheader,nounits",
                 "-lms", "100"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
        return self

    def __exit__(self, *a):
        self.out = ""
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.out, _ = self.proc.communicate(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
                self.out, _ = self.proc.communicate()

    def summary(self):
        rows = []
        for line in (self.out or "").splitlines():
            f = [x.strip() for x in line.split(",")]
            if len(f) < 9:
                continue
            try:
                rows.append(dict(sm=float(f[1]), smax=float(f[2]), power=float(f[3]), hw=f[5], hwt=f[6], swt=f[7],
                                 pcap=f[8]))
            except ValueError:
                continue
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"], "samples": 0}
        reasons = set()
        for r in rows:
            for key, name in (("hw", "hw_slowdown"), ("hwt", "hw_thermal_slowdown"), ("swt", "sw_thermal_slowdown"),
                              ("pcap", "sw_power_cap")):
                if r[key].lower().startswith("active"):
                    reasons.add(name)
        return {"sm_mhz": statistics.median(r["sm"] for r in rows), "sm_max_mhz": max(r["smax"] for r in rows),
                "reasons": sorted(reasons), "samples": len(rows),
                "power_w_max": max(r["power"] for r in rows)}


# ---------------------------------------------------------------------------
# ncu traffic recorded in profiles/ (valid only while the kernel source is unchanged)
# ---------------------------------------------------------------------------

def source_hash(files):
    """Hash of the kernel sources with comments and whitespace removed, so
    that the recorded counters stay valid across comment edits and are
    dropped when any code changes."""
    h = hashlib.sha256()
    for f in files:
        with open(os.path.join(ROOT, f), encoding="utf-8") as fh:
            text = fh.read()
        text = re.sub(r"/\*.*?\*/", " ", text, flags=re.S)
        text = re.sub(r"//[^\n]*", " ", text)
        h.update(re.sub(r"\s+", "", text).encode("utf-8"))
    return h.hexdigest()[:16]


KERNEL_SOURCES = {
    "gemv": ["gemm_int4_dequant_gb300/csrc/gemv_tma.cu", "gemm_int4_dequant_gb300/csrc/ptx.cuh",
             "gemm_int4_dequant_gb300/csrc/common.cuh"],
    "gemm": ["gemm_int4_dequant_gb300/csrc/gemm_tc.cu", "gemm_int4_dequant_gb300/csrc/ptx.cuh",
             "gemm_int4_dequant_gb300/csrc/common.cuh"],
    "quant": ["gemm_int4_dequant_gb300/csrc/quant_permute.cu", "gemm_int4_dequant_gb300/csrc/ptx.cuh",
              "gemm_int4_dequant_gb300/csrc/common.cuh"],
    "gemv8": ["gemm_int4_dequant_gb300/csrc/int8.cu", "gemm_int4_dequant_gb300/csrc/common.cuh"],
    "w4a8": ["gemm_int4_dequant_gb300/csrc/w4a8.cu", "gemm_int4_dequant_gb300/csrc/common.cuh"],
    "ptq1": ["gemm_int4_dequant_gb300/csrc/ptq1.cu", "gemm_int4_dequant_gb300/csrc/ptx.cuh",
             "gemm_int4_dequant_gb300/csrc/common.cuh"],
    "quant8": ["gemm_int4_dequant_gb300/csrc/quant_permute.cu", "gemm_int4_dequant_gb300/csrc/int8.cu",
               "gemm_int4_dequant_gb300/csrc/ptx.cuh", "gemm_int4_dequant_gb300/csrc/common.cuh"],
}


# ncu summary per workload; for the two-kernel steps (w4a8, ptq1) the traffic
# is that of the GEMV, the step's dominant kernel
PROFILE_FILES = {"decode": "gemv_decode_ncu.md", "gemm": "gemm_8192_ncu.md", "quant": "quant_8192_ncu.md",
                 "c8_perm": "gemv_perm_c8_ncu.md", "c8": "gemv_c8_ncu.md", "c8s": "gemv_c8s_ncu.md",
                 "w8_decode": "gemv_w8_decode_ncu.md", "w4a8_decode": "gemv_w4a8_decode_ncu.md",
                 "ptq1_decode": "mmvq_ptq1_decode_ncu.md", "w4a8_c8": "gemv_w4a8_c8_ncu.md",
                 "ptq1_c8": "mmvq_ptq1_c8_ncu.md", "w8_quant": "quant8_8192_ncu.md"}


def recorded_traffic(kind, workload):
    """dram bytes per launch (per step for the two-kernel quant step) from the
    ncu summary in profiles/, if its recorded source hash matches the current
    kernel source; None otherwise."""
    if workload not in PROFILE_FILES:
        return None
    p = os.path.join(ROOT, "profiles", PROFILE_FILES[workload])
    if not os.path.exists(p):
        return None
    text = open(p).read()
    m1 = re.search(r"traffic_bytes_per_launch:\s*([0-9.eE+]+)", text)
    m2 = re.search(r"kernel_source_sha256_16:\s*([0-9a-f]+)", text)
    if not m1 or not m2 or m2.group(1) != source_hash(KERNEL_SOURCES[kind]):
        return None
    return float(m1.group(1))


# ---------------------------------------------------------------------------
# workloads (our implementation)
# ---------------------------------------------------------------------------

def l2_bytes():
    try:
        return int(torch.cuda.get_device_properties(torch.cuda.current_device()).L2_cache_size)
    except Exception:
        return 128 * 2**20


def copies_for(bytes_per_copy):
    return max(2, int(np.ceil(2.0 * l2_bytes() / bytes_per_copy)) + 1)


class GemvWork:
    def __init__(self, w4, N, K, C, seed=0):
        g = synth.gemv_inputs(N, K, C, act="bf16", seed=seed)
        self.g = g
        dev = torch.device("cuda")
        self.R = copies_for(N * K // 2)
        self.q = [g.qweight.to(dev) for _ in range(self.R)]
        self.s, self.z, self.x = g.scale.to(dev), g.zero.to(dev), g.x.to(dev)
        self.d = torch.empty((C, N), dtype=torch.bfloat16, device=dev)
        self.w4 = w4
        self.i = 0
        self.N, self.K, self.C = N, K, C
        self.bytes = gemv_bytes(N, K, C)
        self.flops = 2 * N * K * C
        self.launches_per_step = 1

    def step(self):
        self.w4.gemv_w4(self.q[self.i % self.R], self.s, self.z, self.x, out=self.d)
        self.i += 1

    def l2_note(self):
        return "rotating %d weight copies (%.0f MB > 2x L2)" % (self.R, self.R * self.N * self.K / 2 / 1e6)


class GemvPermWork:
    """gemv_w4_permuted over weights permuted once at setup (untimed)."""

    def __init__(self, w4, N, K, C, seed=0):
        g = synth.packed_gemv_inputs(N, K, C, seed=seed)
        self.g = g
        dev = torch.device("cuda")
        self.R = copies_for(N * K // 2)
        packed = g.packed.to(dev)
        self.q = [w4.permute_int4(packed) for _ in range(self.R)]
        del packed
        self.s, self.x = g.scale.to(dev), g.x.to(dev)
        self.d = torch.empty((C, N), dtype=torch.bfloat16, device=dev)
        self.w4 = w4
        self.i = 0
        self.N, self.K, self.C = N, K, C
        self.bytes = gemv_bytes(N, K, C)
        self.flops = 2 * N * K * C
        self.launches_per_step = 1

    def step(self):
        self.w4.gemv_w4_permuted(self.q[self.i % self.R], self.s, self.x, out=self.d)
        self.i += 1

    def l2_note(self):
        return "rotating %d permuted weight copies (%.0f MB > 2x L2)" % (self.R, self.R * self.N * self.K / 2 / 1e6)


class Gemv8Work:
    """gemv_w8 over rotating copies of an int8 weight."""

    def __init__(self, w4, N, K, C, seed=0):
        g = synth.int8_gemv_inputs(N, K, C, seed=seed)
        self.g = g
        dev = torch.device("cuda")
        self.R = copies_for(N * K)
        self.q = [g.q.to(dev) for _ in range(self.R)]
        self.s, self.x = g.scale.to(dev), g.x.to(dev)
        self.d = torch.empty((C, N), dtype=torch.bfloat16, device=dev)
        self.w4 = w4
        self.i = 0
        self.N, self.K, self.C = N, K, C
        self.bytes = gemv8_bytes(N, K, C)
        self.flops = 2 * N * K * C
        self.launches_per_step = 1

    def step(self):
        self.w4.gemv_w8(self.q[self.i % self.R], self.s, self.x, out=self.d)
        self.i += 1

    def l2_note(self):
        return "rotating %d int8 weight copies (%.0f MB > 2x L2)" % (self.R, self.R * self.N * self.K / 1e6)


class W4a8Work:
    """quantize_q8_1_pt of x, then gemv_w4a8 over rotating weight copies."""

    def __init__(self, w4, N, K, C, seed=0):
        g = synth.gemv_inputs(N, K, C, act="bf16", seed=seed)
        self.g = g
        dev = torch.device("cuda")
        self.R = copies_for(N * K // 2)
        self.q = [g.qweight.to(dev) for _ in range(self.R)]
        self.s, self.z, self.x = g.scale.to(dev), g.zero.to(dev), g.x.to(dev)
        self.pt = torch.empty((C, 144 * (K // 128)), dtype=torch.uint8, device=dev)
        self.d = torch.empty((C, N), dtype=torch.bfloat16, device=dev)
        self.w4 = w4
        self.i = 0
        self.N, self.K, self.C = N, K, C
        self.bytes = w4a8_bytes(N, K, C)
        self.flops = 2 * N * K * C
        self.launches_per_step = 2

    def run(self, x, i):
        self.w4.quantize_q8_1_pt(x, out=self.pt)
        self.w4.gemv_w4a8(self.q[i % self.R], self.s, self.z, self.pt, out=self.d)

    def step(self):
        self.run(self.x, self.i)
        self.i += 1

    def l2_note(self):
        return "rotating %d weight copies (%.0f MB > 2x L2)" % (self.R, self.R * self.N * self.K / 2 / 1e6)


class Ptq1Work:
    """quantize_q8_1_pt of x, then mmvq_ptq1_0 over rotating copies of a
    PTQ1_0 tensor."""

    def __init__(self, w4, N, K, C, seed=0, superblocks=False):
        dev = torch.device("cuda")
        blocks = synth.ptq1_0_blocks(N, K, seed=seed)
        self.superblocks = superblocks
        if superblocks:
            sb, code, ei, ep = w4.ptq1_1_encode(blocks)   # host conversion, untimed
            blocks = sb
            self.tables = [torch.from_numpy(a).to(dev) for a in (code, ei, ep)]
        self.R = copies_for(blocks.nbytes)
        self.q = [torch.from_numpy(blocks).to(dev) for _ in range(self.R)]
        self.x_cpu = synth.gemv_inputs(1, K, C, act="bf16", seed=seed).x
        self.x = self.x_cpu.to(dev)
        self.pt = torch.empty((C, 144 * (K // 128)), dtype=torch.uint8, device=dev)
        self.d = torch.empty((C, N), dtype=torch.float32, device=dev)
        self.w4 = w4
        self.i = 0
        self.N, self.K, self.C = N, K, C
        self.bytes = ptq1_bytes(N, K, C, superblocks)
        self.flops = 2 * N * K * C
        self.launches_per_step = 2

    def run(self, x, i):
        self.w4.quantize_q8_1_pt(x, out=self.pt)
        if self.superblocks:
            code, ei, ep = self.tables
            self.w4.mmvq_ptq1_1(self.q[i % self.R], code, ei, ep, self.pt, self.K, out=self.d)
        else:
            self.w4.mmvq_ptq1_0(self.q[i % self.R], self.pt, out=self.d)

    def step(self):
        self.run(self.x, self.i)
        self.i += 1

    def l2_note(self):
        per = self.q[0].numel()
        return "rotating %d %s copies (%.0f MB > 2x L2)" % (self.R, "PTQ1_1" if self.superblocks else "PTQ1_0",
                                                          self.R * per / 1e6)


class Quant8Work:
    """quantize_int8 + permute_int8 of one weight."""

    def __init__(self, w4, K, N, seed=0):
        dev = torch.device("cuda")
        self.W = synth.quant_inputs(K, N, seed=seed).to(dev)
        self.q = torch.empty((K, N), dtype=torch.int8, device=dev)
        self.scale = torch.empty((N,), dtype=torch.float32, device=dev)
        self.out = torch.empty((N * K,), dtype=torch.int8, device=dev)
        self.w4 = w4
        self.K, self.N = K, N
        self.bytes = quant8_bytes(K, N)
        self.flops = 0
        self.launches_per_step = 2

    def step(self):
        self.w4.quantize_int8(self.W, q=self.q, scale=self.scale)
        self.w4.permute_int8(self.q, out=self.out)

    def l2_note(self):
        return "W is %.0f MB > L2" % (self.K * self.N * 2 / 1e6)


class QuantWork:
    def __init__(self, w4, K, N, fused=True, seed=0):
        dev = torch.device("cuda")
        W = synth.quant_inputs(K, N, seed=seed).to(dev)
        self.W = W
        self.packed = torch.empty((K // 2, N), dtype=torch.int8, device=dev)
        self.scale = torch.empty((N,), dtype=torch.float32, device=dev)
        self.out = torch.empty((N * K // 2,), dtype=torch.int8, device=dev)
        self.w4 = w4
        self.K, self.N = K, N
        self.fused = fused
        self.bytes = quant_bytes(K, N, fused)
        self.flops = 0
        self.launches_per_step = 1 if fused else 2

    def step(self):
        if self.fused:
            self.w4.quantize_pack_permute_int4(self.W, out=self.out, scale=self.scale)
        else:
            self.w4.quantize_pack_int4(self.W, packed=self.packed, scale=self.scale)
            self.w4.permute_int4(self.packed, out=self.out)

    def l2_note(self):
        return "W is %.0f MB > L2" % (self.K * self.N * 2 / 1e6)


class GemmWork:
    def __init__(self, w4, M, N, K, seed=0):
        dev = torch.device("cuda")
        gi = synth.gemm_inputs(M, N, K, seed=seed)
        self.A, self.B = gi.A.to(dev), gi.B.to(dev)
        self.s, self.z = gi.scale.to(dev), gi.zero.to(dev)
        self.C = torch.empty((M, N), dtype=torch.bfloat16, device=dev)
        self.w4 = w4
        self.M, self.N, self.K = M, N, K
        self.bytes = gemm_bytes(M, N, K)
        self.flops = gemm_flops(M, N, K)
        self.launches_per_step = 1

    def step(self):
        self.w4.gemm_w4(self.A, self.B, self.s, self.z, out=self.C)

    def l2_note(self):
        return "A+C are %.0f MB > L2" % ((self.M * self.K + self.M * self.N) * 2 / 1e6)


class Gemm8Work(GemmWork):
    """gemm_w8: bf16 A times quantize_int8's matrix."""

    def __init__(self, w4, M, N, K, seed=0):
        dev = torch.device("cuda")
        gi = synth.int8_gemv_inputs(N, K, 1, seed=seed)
        self.A = synth.gemm_inputs(M, 16, K, seed=seed + 1).A.to(dev)
        self.B, self.s = gi.q.to(dev), gi.scale.to(dev)
        self.C = torch.empty((M, N), dtype=torch.bfloat16, device=dev)
        self.w4 = w4
        self.M, self.N, self.K = M, N, K
        self.bytes = M * K * 2 + K * N + M * N * 2 + 4 * N
        self.flops = gemm_flops(M, N, K)
        self.launches_per_step = 1

    def step(self):
        self.w4.gemm_w8(self.A, self.B, self.s, out=self.C)


class GemmPermWork(GemmWork):
    """gemm_w4_permuted over weights permuted once at setup (untimed)."""

    def __init__(self, w4, M, N, K, seed=0):
        dev = torch.device("cuda")
        g = synth.packed_gemv_inputs(N, K, 1, seed=seed)
        self.A = synth.gemm_inputs(M, 16, K, seed=seed + 1).A.to(dev)
        self.B = w4.permute_int4(g.packed.to(dev))
        self.s = g.scale.to(dev)
        self.C = torch.empty((M, N), dtype=torch.bfloat16, device=dev)
        self.w4 = w4
        self.M, self.N, self.K = M, N, K
        self.bytes = gemm_bytes(M, N, K)
        self.flops = gemm_flops(M, N, K)
        self.launches_per_step = 1

    def step(self):
        self.w4.gemm_w4_permuted(self.A, self.B, self.s, out=self.C)
def torch_matmul_context(work, steps):
    """Context only, not a product path: the packed B dequantised to bf16 once
    with torch ops (untimed), then torch.matmul (cuBLAS) timed with CUDA
    events over `steps` calls.  Returns TFLOP/s, or an error note (this bar
    never fails the benchmark)."""
    try:
        B = work.B
        K2, N = B.shape
        W = torch.empty((2 * K2, N), dtype=torch.bfloat16, device=B.device)
        W[0::2] = (B & 0x0F).to(torch.bfloat16)   # even k in the low nibble
        W[1::2] = (B >> 4).to(torch.bfloat16)
        W = (W - work.z[None, :]) * work.s[None, :]
        out = torch.empty((work.M, N), dtype=torch.bfloat16, device=B.device)
        for _ in range(3):
            torch.matmul(work.A, W, out=out)
        torch.cuda.synchronize()
        start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        start.record()
        for _ in range(steps):
            torch.matmul(work.A, W, out=out)
        end.record()
        torch.cuda.synchronize()
        sec = start.elapsed_time(end) / 1e3 / steps
        del W, out
        torch.cuda.empty_cache()
        return {"value": work.flops / sec / 1e12, "unit": "TFLOP/s",
                "note": "context: B dequantised to bf16 once (untimed), then torch.matmul (cuBLAS)"}
    except Exception as e:   # noqa: BLE001 -- a context bar must not fail the run
        return {"value": None, "error": "%s: %s" % (type(e).__name__, str(e)[:200])}


def make_work(w4, name):
    cfg = dict(WORKLOADS[name])
    kind = cfg.pop("kind")
    if cfg.pop("perm", False):
        return GemvPermWork(w4, **cfg)
    if kind == "gemv":
        return GemvWork(w4, **cfg)
    if kind == "quant":
        return QuantWork(w4, **cfg)
    if kind == "gemv8":
        return Gemv8Work(w4, **cfg)
    if kind == "quant8":
        return Quant8Work(w4, **cfg)
    if kind == "w4a8":
        return W4a8Work(w4, **cfg)
    if kind == "gemm8":
        return Gemm8Work(w4, **cfg)
    if kind == "gemmp":
        return GemmPermWork(w4, **cfg)
    if kind == "ptq1":
        return Ptq1Work(w4, **cfg)
    return GemmWork(w4, **cfg)


def time_graph(work, steps, warmup, world):
    """Warm up eagerly, capture `steps` steps into one CUDA graph, replay it
    once untimed and once timed.  Returns seconds for the timed replay
    (max over ranks)."""
    stream = torch.cuda.Stream()
    stream.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(stream):
        for _ in range(max(3, warmup)):
            work.step()
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream, capture_error_mode="thread_local"):
        for _ in range(steps):
            work.step()
    g.replay()
    torch.cuda.synchronize()
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    barrier(world)
    torch.cuda.synchronize()
    with torch.cuda.stream(stream):
        start.record(stream)
        g.replay()
        end.record(stream)
    torch.cuda.synchronize()
    barrier(world)
    sec = start.elapsed_time(end) / 1e3
    return max_over_ranks(sec, world), g, stream


def isolated_steps(work, n=50):
    """Mean time of one step launched alone: before each, a 256 MB write
    evicts L2 (cold weights and x) and a short GPU spin keeps the device busy
    while the host prepares the launch, so the event pair brackets the
    step's kernels and not the host; a device synchronise follows every
    step.  The mean, not the median: event timestamps here come in steps of
    about 2 us, and averaging 50 samples resolves below that."""
    stream = torch.cuda.Stream()
    flush = torch.empty(256 * 2**20, dtype=torch.uint8, device="cuda")
    times = []
    with torch.cuda.stream(stream):
        for i in range(n + 3):
            flush.zero_()
            torch.cuda._sleep(2000000)   # about 1 ms of GPU spin, so the launch is queued before e0 runs
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            work.step()
            e1.record(stream)
            e1.synchronize()
            if i >= 3:
                times.append(e0.elapsed_time(e1) / 1e3)
    del flush
    return statistics.fmean(times)


def soak(g, stream, seconds):
    t0 = time.time()
    with torch.cuda.stream(stream):
        while time.time() - t0 < seconds:
            g.replay()
            torch.cuda.synchronize()


def e2e_gemv(w4, work, steps, world):
    """Public API, host buffers: x from pinned host memory in, d back out."""
    x_host = (work.x_cpu if isinstance(work, Ptq1Work) else work.g.x).clone().pin_memory()
    d_host = torch.empty((work.C, work.N), dtype=work.d.dtype).pin_memory()
    x_dev = torch.empty_like(work.x)
    stream = torch.cuda.current_stream()
    perm = isinstance(work, GemvPermWork)
    w8 = isinstance(work, Gemv8Work)
    w4a8 = isinstance(work, (W4a8Work, Ptq1Work))

    def call(i):
        if w4a8:
            work.run(x_dev, i)
        elif perm:
            w4.gemv_w4_permuted(work.q[i % work.R], work.s, x_dev, out=work.d)
        elif w8:
            w4.gemv_w8(work.q[i % work.R], work.s, x_dev, out=work.d)
        else:
            w4.gemv_w4(work.q[i % work.R], work.s, work.z, x_dev, out=work.d)

    for i in range(3):
        x_dev.copy_(x_host, non_blocking=True)
        call(i)
        d_host.copy_(work.d, non_blocking=True)
    torch.cuda.synchronize()
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    barrier(world)
    torch.cuda.synchronize()
    start.record(stream)
    for i in range(steps):
        x_dev.copy_(x_host, non_blocking=True)
        call(i)
        d_host.copy_(work.d, non_blocking=True)
    end.record(stream)
    torch.cuda.synchronize()
    barrier(world)
    sec = max_over_ranks(start.elapsed_time(end) / 1e3, world)
    return sec, x_host.numel() * 2, d_host.numel() * d_host.element_size()


def e2e_generic(work, steps, world):
    """GEMM / quant: every input copied in from pinned host memory and the
    result copied back, each step."""
    if isinstance(work, GemmWork):
        hosts = [work.A.cpu().pin_memory(), work.B.cpu().pin_memory()]
        devs = [work.A, work.B]
        outs = [(work.C, torch.empty_like(work.C, device="cpu").pin_memory())]
    else:
        hosts = [work.W.cpu().pin_memory()]
        devs = [work.W]
        outs = [(work.out, torch.empty_like(work.out, device="cpu").pin_memory()),
                (work.scale, torch.empty_like(work.scale, device="cpu").pin_memory())]
    stream = torch.cuda.current_stream()

    def one():
        for h, d in zip(hosts, devs):
            d.copy_(h, non_blocking=True)
        work.step()
        for d, h in outs:
            h.copy_(d, non_blocking=True)

    for _ in range(2):
        one()
    torch.cuda.synchronize()
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    barrier(world)
    torch.cuda.synchronize()
    start.record(stream)
    for _ in range(steps):
        one()
    end.record(stream)
    torch.cuda.synchronize()
    barrier(world)
    sec = max_over_ranks(start.elapsed_time(end) / 1e3, world)
    hb = sum(h.numel() * h.element_size() for h in hosts)
    ob = sum(h.numel() * h.element_size() for _, h in outs)
    return sec, hb, ob


# ---------------------------------------------------------------------------
# CPU baseline: the oracle as it stands, on a bounded sample
# ---------------------------------------------------------------------------

def cpu_baseline(name, budget_s=10.0):
    import oracle
    from synth import np_bits
    cfg = WORKLOADS[name]
    if cfg["kind"] == "gemv" and cfg.get("perm"):
        g = synth.packed_gemv_inputs(cfg["N"], cfg["K"], cfg["C"], seed=0)
        packed, scale, xb = g.packed.numpy(), g.scale.numpy(), np_bits(g.x)
        N = cfg["N"]
        t0 = time.perf_counter()
        oracle.gemv_packed(packed, scale, xb, cols=(0, min(N, 64)))
        per_col = (time.perf_counter() - t0) / min(N, 64)
        cols = int(max(1, min(N, 1.0 / max(per_col, 1e-9))))
        done, t_total, c0 = 0, 0.0, 0
        while t_total < budget_s:
            c1 = min(N, c0 + cols)
            t0 = time.perf_counter()
            oracle.gemv_packed(packed, scale, xb, cols=(c0, c1))
            t_total += time.perf_counter() - t0
            done += c1 - c0
            c0 = 0 if c1 >= N else c1
        bytes_done = gemv_bytes(cfg["N"], cfg["K"], cfg["C"]) * done / N
        return {"value": bytes_done / t_total / 1e9, "unit": "GB/s", "cores": 1, "kind": "oracle",
                "sample": "%d columns of the %dx%d C=%d GEMV over the packed matrix (fp64 C oracle, single "
                          "thread), %.1f s" % (done, cfg["N"], cfg["K"], cfg["C"], t_total)}
    if cfg["kind"] == "gemv":
        g = synth.gemv_inputs(cfg["N"], cfg["K"], cfg["C"], act="bf16", seed=0)
        args = (np_bits(g.qweight), np_bits(g.scale), np_bits(g.zero), np_bits(g.x), oracle.BF16)
        N = cfg["N"]
        # rows per call sized to ~1 s; repeat until the budget is used
        t0 = time.perf_counter()
        oracle.gemv(*args, rows=(0, min(N, 512)))
        per_row = (time.perf_counter() - t0) / min(N, 512)
        rows = int(max(1, min(N, 1.0 / max(per_row, 1e-9))))
        done_rows, t_total, r0 = 0, 0.0, 0
        while t_total < budget_s:
            r1 = min(N, r0 + rows)
            t0 = time.perf_counter()
            oracle.gemv(*args, rows=(r0, r1))
            t_total += time.perf_counter() - t0
            done_rows += r1 - r0
            r0 = 0 if r1 >= N else r1
        bytes_done = gemv_bytes(cfg["N"], cfg["K"], cfg["C"]) * done_rows / N
        return {"value": bytes_done / t_total / 1e9, "unit": "GB/s", "cores": 1, "kind": "oracle",
                "sample": "%d rows of the %dx%d C=%d GEMV (fp64 C oracle, single thread), %.1f s" %
                          (done_rows, cfg["N"], cfg["K"], cfg["C"], t_total)}
    if cfg["kind"] == "gemm":
        gi = synth.gemm_inputs(cfg["M"], cfg["N"], cfg["K"], seed=0)
        A, B, s, z = np_bits(gi.A), gi.B.numpy(), np_bits(gi.scale), np_bits(gi.zero)
        n_out, t_total = 0, 0.0
        rng = np.random.default_rng(0)
        while t_total < budget_s:
            mi = rng.integers(0, cfg["M"], 4096)
            ni = rng.integers(0, cfg["N"], 4096)
            t0 = time.perf_counter()
            oracle.gemm_at(A, B, s, z, mi, ni)
            t_total += time.perf_counter() - t0
            n_out += 4096
        flops = 2 * cfg["K"] * n_out
        return {"value": flops / t_total / 1e12, "unit": "TFLOP/s", "cores": 1, "kind": "oracle",
                "sample": "%d sampled outputs of the 8192^3 GEMM (fp64 C oracle, single thread), %.1f s" %
                          (n_out, t_total)}
    if cfg["kind"] == "gemmp":
        M, N, K = cfg["M"], cfg["N"], cfg["K"]
        g = synth.packed_gemv_inputs(N, K, 1, seed=0)
        A = np_bits(synth.gemm_inputs(M, 16, K, seed=1).A)
        rng = np.random.default_rng(0)
        n_out, t_total = 0, 0.0
        while t_total < budget_s:
            mi, ni = rng.integers(0, M, 256), rng.integers(0, N, 256)
            t0 = time.perf_counter()
            oracle.gemm_packed_at(A, g.packed.numpy(), g.scale.numpy(), mi, ni)
            t_total += time.perf_counter() - t0
            n_out += 256
        return {"value": 2.0 * K * n_out / t_total / 1e12, "unit": "TFLOP/s", "cores": 1, "kind": "oracle",
                "sample": "%d sampled outputs of the 8192^3 GEMM over the packed matrix (fp64 C oracle, single "
                          "thread), %.1f s" % (n_out, t_total)}
    if cfg["kind"] == "gemm8":
        M, N, K = cfg["M"], cfg["N"], cfg["K"]
        gi = synth.int8_gemv_inputs(N, K, 1, seed=0)
        A = np_bits(synth.gemm_inputs(M, 16, K, seed=1).A)
        rng = np.random.default_rng(0)
        n_out, t_total = 0, 0.0
        while t_total < budget_s:
            mi, ni = rng.integers(0, M, 256), rng.integers(0, N, 256)
            t0 = time.perf_counter()
            oracle.gemm_int8_at(A, gi.q.numpy(), gi.scale.numpy(), mi, ni)
            t_total += time.perf_counter() - t0
            n_out += 256
        flops = 2.0 * K * n_out
        return {"value": flops / t_total / 1e12, "unit": "TFLOP/s", "cores": 1, "kind": "oracle",
                "sample": "%d sampled outputs of the 8192^3 int8 GEMM (fp64 C oracle, single thread), %.1f s" %
                          (n_out, t_total)}
    if cfg["kind"] == "gemv8":
        g = synth.int8_gemv_inputs(cfg["N"], cfg["K"], cfg["C"], seed=0)
        q, scale, xb = g.q.numpy(), g.scale.numpy(), np_bits(g.x)
        N = cfg["N"]
        done, t_total, c0 = 0, 0.0, 0
        cols = 256
        while t_total < budget_s:
            c1 = min(N, c0 + cols)
            t0 = time.perf_counter()
            oracle.gemv_int8(q, scale, xb, cols=(c0, c1))
            t_total += time.perf_counter() - t0
            done += c1 - c0
            c0 = 0 if c1 >= N else c1
        return {"value": gemv8_bytes(cfg["N"], cfg["K"], cfg["C"]) * done / N / t_total / 1e9, "unit": "GB/s",
                "cores": 1, "kind": "oracle",
                "sample": "%d columns of the %dx%d C=%d int8 GEMV (fp64 C oracle, single thread), %.1f s" %
                          (done, cfg["N"], cfg["K"], cfg["C"], t_total)}
    if cfg["kind"] == "w4a8":
        g = synth.gemv_inputs(cfg["N"], cfg["K"], cfg["C"], act="bf16", seed=0)
        qw, s, z, xb = np_bits(g.qweight), np_bits(g.scale), np_bits(g.zero), np_bits(g.x)
        N, K = cfg["N"], cfg["K"]
        done, t_total, r0 = 0, 0.0, 0
        rows = 256
        while t_total < budget_s:
            r1 = min(N, r0 + rows)
            t0 = time.perf_counter()
            pt = oracle.quantize_q8_1_pt(xb)
            oracle.gemv_w4a8(qw, s, z, pt, K, rows=(r0, r1))
            t_total += time.perf_counter() - t0
            done += r1 - r0
            r0 = 0 if r1 >= N else r1
        return {"value": w4a8_bytes(N, K, cfg["C"]) * done / N / t_total / 1e9, "unit": "GB/s", "cores": 1,
                "kind": "oracle",
                "sample": "%d rows of the %dx%d C=%d W4A8 GEMV, x quantised each time (fp64 C oracle, single "
                          "thread), %.1f s" % (done, N, K, cfg["C"], t_total)}
    if cfg["kind"] == "ptq1":
        N, K = cfg["N"], cfg["K"]
        sup = cfg.get("superblocks", False)
        blocks = synth.ptq1_0_blocks(N, K, seed=0)
        wsb = oracle.ptq1_1_encode(blocks) if sup else None
        xb = np_bits(synth.gemv_inputs(1, K, cfg["C"], act="bf16", seed=0).x)
        done, t_total, r0 = 0, 0.0, 0
        rows = 256
        while t_total < budget_s:
            r1 = min(N, r0 + rows)
            t0 = time.perf_counter()
            pt = oracle.quantize_q8_1_pt(xb)
            if sup:
                oracle.mmvq_ptq1_1(wsb, pt, rows=(r0, r1))
            else:
                oracle.mmvq_ptq1_0(blocks, pt, rows=(r0, r1))
            t_total += time.perf_counter() - t0
            done += r1 - r0
            r0 = 0 if r1 >= N else r1
        return {"value": ptq1_bytes(N, K, cfg["C"], sup) * done / N / t_total / 1e9, "unit": "GB/s", "cores": 1,
                "kind": "oracle",
                "sample": "%d rows of the %dx%d C=%d ternary MMVQ, x quantised each time (fp64 C oracle, single "
                          "thread), %.1f s" % (done, N, K, cfg["C"], t_total)}
    if cfg["kind"] == "quant8":
        K, N = cfg["K"], cfg["N"]
        W = np_bits(synth.quant_inputs(K, N, seed=0))
        n_done, t_total = 0, 0.0
        while t_total < budget_s:
            t0 = time.perf_counter()
            s_ref, q_ref = oracle.quantize_int8(W)
            oracle.permute_int8(q_ref, K, N)
            t_total += time.perf_counter() - t0
            n_done += 1
        return {"value": quant8_bytes(K, N) * n_done / t_total / 1e9, "unit": "GB/s", "cores": 1, "kind": "oracle",
                "sample": "%d full int8 quantize+permute of %dx%d (C oracle, single thread), %.1f s" %
                          (n_done, K, N, t_total)}
    K, N = cfg["K"], cfg["N"]
    W = np_bits(synth.quant_inputs(K, N, seed=0))
    n_done, t_total = 0, 0.0
    while t_total < budget_s:
        t0 = time.perf_counter()
        s_ref, p_ref = oracle.quantize_pack(W)
        oracle.permute(p_ref, K, N)
        t_total += time.perf_counter() - t0
        n_done += 1
    return {"value": quant_bytes(K, N, cfg.get("fused", True)) * n_done / t_total / 1e9, "unit": "GB/s", "cores": 1,
            "kind": "oracle",
            "sample": "%d full quantize+pack+permute of %dx%d (C oracle, single thread), %.1f s" %
                      (n_done, K, N, t_total)}


def host_threads():
    """The host cores this process may run on."""
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count() or 1


def cpu_baseline_all_cores(name, budget_s=10.0):
    """The same oracle on every host core: threads take disjoint 64-row
    chunks of the row-layout GEMV (the C oracle runs outside the Python
    lock), until the budget; None for the other workloads."""
    cfg = WORKLOADS[name]
    if cfg["kind"] != "gemv" or cfg.get("perm"):
        return None
    import threading
    from concurrent.futures import ThreadPoolExecutor

    import oracle
    from synth import np_bits
    g = synth.gemv_inputs(cfg["N"], cfg["K"], cfg["C"], act="bf16", seed=0)
    args = (np_bits(g.qweight), np_bits(g.scale), np_bits(g.zero), np_bits(g.x), oracle.BF16)
    N, chunk, threads = cfg["N"], 64, host_threads()
    oracle.gemv(*args, rows=(0, 1))   # load the library before the clock starts
    lock = threading.Lock()
    state = {"next": 0}
    deadline = time.perf_counter() + budget_s

    def worker():
        done = 0
        while time.perf_counter() < deadline:
            with lock:
                r0 = state["next"]
                state["next"] = (r0 + chunk) % N if r0 + chunk < N else 0
            r1 = min(N, r0 + chunk)
            oracle.gemv(*args, rows=(r0, r1))
            done += r1 - r0
        return done

    t0 = time.perf_counter()
    with ThreadPoolExecutor(max_workers=threads) as ex:
        rows = sum(ex.map(lambda _: worker(), range(threads)))
    wall = time.perf_counter() - t0
    return {"value": gemv_bytes(N, cfg["K"], cfg["C"]) * rows / N / wall / 1e9, "unit": "GB/s", "cores": threads,
            "kind": "oracle",
            "sample": "%d rows of the %dx%d C=%d GEMV in 64-row chunks over %d threads (fp64 C oracle), %.1f s" %
                      (rows, N, cfg["K"], cfg["C"], threads, wall)}


# ---------------------------------------------------------------------------
# main
# ---------------------------------------------------------------------------

def dtype_of(name):
    """The arithmetic the workload's kernels compute in."""
    cfg = WORKLOADS[name]
    if cfg["kind"] == "gemv":
        if cfg.get("perm"):
            return "bf16 x / int4 weights (bf16 MMA), fp32 accumulate"
        if cfg["C"] == 1:
            return "fp16 MMA (bf16 x scaled by a power of two) / uint4 weights, fp32 accumulate"
        return "bf16 x / uint4 weights (bf16 MMA), fp32 accumulate"
    if cfg["kind"] == "gemm":
        return "bf16 A / uint4 B (bf16 tcgen05 MMA), fp32 accumulate"
    if cfg["kind"] == "gemm8":
        return "bf16 A / int8 B (bf16 tcgen05 MMA), fp32 accumulate"
    if cfg["kind"] == "gemmp":
        return "bf16 A / permuted int4 B (bf16 tcgen05 MMA), fp32 accumulate"
    if cfg["kind"] == "gemv8":
        return "bf16 x / int8 weights (fp32 FMA)"
    if cfg["kind"] == "quant8":
        return "bf16 in, int8 out (fp32 division)"
    if cfg["kind"] == "w4a8":
        return "x quantised to int8 (block_q8_1) / uint4 weights, int32 dp4a dots, fp32 accumulate"
    if cfg["kind"] == "ptq1":
        fmt = "PTQ1_1" if cfg.get("superblocks") else "PTQ1_0"
        return "x quantised to int8 (block_q8_1) / ternary %s weights, int32 dp4a dots, fp32 accumulate" % fmt
    return "bf16 in, int4 out (fp32 arithmetic)"


def unit_of(work):
    return "TFLOP/s" if isinstance(work, GemmWork) else "GB/s"


def rate(work, sec_per_step):
    if isinstance(work, GemmWork):
        return work.flops / sec_per_step / 1e12
    return work.bytes / sec_per_step / 1e9


def roofline(work, sec_per_launch, peaks, peak_src, kind_name, workload):
    if isinstance(work, GemmWork):
        achieved = work.flops / sec_per_launch / 1e12
        peak = float(peaks.get("bf16_tflops", FALLBACK_PEAKS["bf16_tflops"]))
        return {"bound": "tensor", "achieved": achieved, "peak": peak, "unit": "TFLOP/s",
                "frac": achieved / peak, "peak_source": "%s bf16 burst" % peak_src,
                "peak_nominal": NOMINAL_PEAKS["bf16_tflops"], "frac_nominal": achieved / NOMINAL_PEAKS["bf16_tflops"],
                "traffic": recorded_traffic("gemm", workload)}
    # quant: the two kernels of a step together (bytes of the step / time of the step)
    achieved = work.bytes / work.launches_per_step / sec_per_launch / 1e9
    peak = float(peaks.get("hbm_gbs", FALLBACK_PEAKS["hbm_gbs"]))
    return {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s", "frac": achieved / peak,
            "peak_source": "%s HBM copy" % peak_src,
            "peak_nominal": NOMINAL_PEAKS["hbm_gbs"], "frac_nominal": achieved / NOMINAL_PEAKS["hbm_gbs"],
            "traffic": recorded_traffic(kind_name, workload)}


def run_ours(args, world, rank):
    import gemm_int4_dequant_gb300 as w4
    peaks, peak_src = load_peaks()
    work = make_work(w4, args.workload)
    kind = WORKLOADS[args.workload]["kind"]
    sec, g, stream = time_graph(work, args.steps, args.warmup, world)
    sec_step = sec / args.steps
    value = job_rate(rate(work, sec_step), world)
    with ClockSampler(int(os.environ.get("LOCAL_RANK", "0"))) as cs:
        soak(g, stream, 2.0)
        sec2, _, _ = time_graph(work, args.steps, 0, world)
    clocks = cs.summary()
    iso_sec = isolated_steps(work)
    if kind in ("gemv", "gemv8", "w4a8", "ptq1"):
        e2e_sec, hb, ob = e2e_gemv(w4, work, args.steps, world)
    else:
        e2e_sec, hb, ob = e2e_generic(work, max(2, min(args.steps, 10)), world)
        e2e_sec = e2e_sec * args.steps / max(2, min(args.steps, 10))
    e2e_val = job_rate(rate(work, e2e_sec / args.steps), world)
    line = {
        "metric": METRIC, "value": value, "unit": unit_of(work), "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": sec_step * 1e3, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": dtype_of(args.workload),
        "data": "synthetic (seeded; shapes of the pages' workloads)",
        "config": {"workload": args.workload, **{k: v for k, v in WORKLOADS[args.workload].items() if k != "kind"},
                   "l2": work.l2_note(), "parallelism": "replicas" if world > 1 else "single GPU"},
        "roofline": roofline(work, sec_step / work.launches_per_step, peaks, peak_src, kind, args.workload),
        "isolated": {"value": rate(work, iso_sec), "unit": unit_of(work), "ms_per_step": iso_sec * 1e3,
                     "frac": roofline(work, iso_sec / work.launches_per_step, peaks, peak_src, kind,
                                      args.workload)["frac"],
                     "how": "one step alone after a 256 MB L2-evicting write, device synchronise after it; "
                            "mean of 50"},
        "gpu_launches": args.steps * work.launches_per_step,
        "clocks": clocks,
        "e2e": {"value": e2e_val, "unit": unit_of(work), "h2d_bytes_per_step": hb, "d2h_bytes_per_step": ob},
    }
    line["roofline"]["timing"] = ("CUDA events around one graph replay of the timed steps, launched back to back: "
                                  "a launch may start (programmatic dependent launch) while the previous one "
                                  "finishes; `isolated` is one launch alone")
    if kind == "gemm":
        line["context_torch_matmul"] = torch_matmul_context(work, max(3, min(args.steps, 20)))
    if kind == "quant8" or (kind == "quant" and not WORKLOADS[args.workload].get("fused", True)):
        line["roofline"]["note"] = "two kernels per step (quantise, then permute); achieved = step bytes / step time"
    if kind in ("w4a8", "ptq1"):
        line["roofline"]["note"] = ("two kernels per step (quantise x, then the GEMV); achieved = step bytes / "
                                    "step time")
    if rank == 0 and world == 1:
        line["cpu_baseline"] = cpu_baseline(args.workload, budget_s=args.cpu_seconds)
        every_core = cpu_baseline_all_cores(args.workload, budget_s=args.cpu_seconds)
        if every_core is not None:
            line["cpu_baseline_all_cores"] = every_core
    if args.components and world == 1:
        comps = {}
        for name in [n for n in COMPONENTS if n != args.workload]:
            cfg = WORKLOADS[name]
            wk = make_work(w4, name)
            s, _, _ = time_graph(wk, max(10, args.steps // 4), 3, world)
            per = s / max(10, args.steps // 4)
            rl = roofline(wk, per / wk.launches_per_step, peaks, peak_src, cfg["kind"], name)
            comps[name] = {"value": rate(wk, per), "unit": unit_of(wk), "ms_per_step": per * 1e3,
                           "frac": rl["frac"], "bound": rl["bound"], "traffic": rl["traffic"],
                           "config": {k: v for k, v in cfg.items() if k != "kind"}}
            if cfg["kind"] == "gemm":
                comps[name]["context_torch_matmul"] = torch_matmul_context(wk, 10)
            del wk
            torch.cuda.empty_cache()
        line["components"] = comps
    return line


def run_reference(args, world, rank):
    """The oracle (the plain CPU reference) on the host cores, rank 0 only."""
    if rank != 0:
        return None
    cfg = WORKLOADS[args.workload]
    t_budget = max(1.0, args.cpu_seconds / max(1, args.steps))
    vals = []
    last = None
    for _ in range(args.warmup and 1):
        cpu_baseline(args.workload, budget_s=0.5)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        last = cpu_baseline(args.workload, budget_s=t_budget)
        vals.append(last["value"])
    elapsed = time.perf_counter() - t0
    value = statistics.median(vals)
    unit = last["unit"]
    return {
        "impl": "reference", "metric": METRIC, "value": value, "unit": unit, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": elapsed / args.steps * 1e3, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64 (oracle)", "data": "synthetic (seeded)",
        "config": {"workload": args.workload, **{k: v for k, v in cfg.items() if k != "kind"}},
        "cpu_baseline": {"value": value, "unit": unit, "cores": 1, "kind": "oracle",
                         "sample": "%d steps, each: %s" % (args.steps, last["sample"])},
        "e2e": {"value": value, "unit": unit, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
        "gpu_launches": 0,
    }


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", choices=sorted(WORKLOADS), default="decode")
    ap.add_argument("--cpu-seconds", type=float, default=10.0)
    ap.add_argument("--no-components", dest="components", action="store_false")
    args = ap.parse_args()
    if args.warmup < 3 and args.impl == "ours":
        args.warmup = 3
    if args.impl == "reference":
        rank = int(os.environ.get("RANK", "0"))
        world = int(os.environ.get("WORLD_SIZE", "1"))
        line = run_reference(args, world, rank)
        if line is not None:
            print(json.dumps(line), flush=True)
        return
    world, rank = dist_setup(args.gpus)
    line = run_ours(args, world, rank)
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
