"""Benchmark of the GB300 dense GEMM library.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                    [--workload NAME] [--no-paths] [--no-cpu-baseline] [--no-e2e]

A step is one C = A·B call on one batch of seeded synthetic input.  The
default workload is the pages' main SGEMM: FP32 row-major M = N = K = 4096 (A,
B uniform[-1, 1]), pure FP32 FFMA.  The line printed by rank 0 carries the
throughput in TFLOP/s (2*M*N*K per step, device time by CUDA events on the
launching stream), the roofline of the kernel, the oracle's CPU throughput
on a bounded sample, an end-to-end number through host buffers, the clocks seen
during the timed region and -- under "paths" -- the same measurements for the
tensor-core workloads (FP16 column-major 8192^3 and 3072x5120x6144, BF16 FFN
projection, the fused FFN gate/up projection), the M = 1 decode shapes, and the
general form (gemm_ex: X W^T with W stored [N, K], a strided batch, FP32 with a
transposed B).

--impl reference times the CPU oracle (the reference arm of this build) on
the same workload and prints its line with "impl": "reference".

Under torchrun every rank runs the same workload on its own GPU (replicas, no
collective on the data path): value = FLOPs of all ranks / slowest rank's time.
"""

from __future__ import annotations

import argparse
import csv
import hashlib
import io
import json
import math
import os
import statistics
import subprocess
import sys
import tempfile
import time
from datetime import datetime

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402

import synthetic  # noqa: E402
from dense_matrix_multiply_gb300 import metrics  # noqa: E402

METRIC = "GEMM TFLOP/s (2·M·N·K/t) and % of FP32-SIMT or BF16/FP16 tensor peak"
DEFAULT_WORKLOAD = "sgemm_f32_rm_4096"
# The other workloads measured in the default run ("paths"): every other
# configuration of the five (the FP16 and BF16 tensor-core problems and the
# whole ragged/edge sweep on both the FP32 and the BF16 path, the K = 4100 tail
# beside its K = 4096 control), a decode batch with more 128-column weight
# strips than SMs, then the fused, general-form and FP8 workloads.
DEFAULT_PATHS = ["hgemm_f16_cm_8192", "hgemm_f16_cm_3072x5120x6144", "ffn_bf16_rm_1024x12288x4096",
                 "sgemm_f32_rm_256",
                 "edge_f32_rm_1000x1000x1000", "edge_bf16_rm_1000x1000x1000",
                 "edge_bf16_rm_1x12288x4096", "edge_f32_rm_1x12288x4096", "edge_bf16_rm_32x12288x4096",
                 "decode_bf16_rm_8x28672x4096",
                 "edge_f32_rm_64x64x64", "edge_bf16_rm_64x64x64",
                 "edge_bf16_rm_8192x4096x4100", "edge_bf16_rm_8192x4096x4096",
                 "edge_f32_rm_8192x4096x4100", "edge_f32_rm_8192x4096x4096",
                 "ffn_gate_up_bf16_silu_mul_1024x12288x4096",
                 "gemm_ex_bf16_rm_NT_8192x8192x8192", "gemm_ex_f16_rm_NN_batch32_1024x1024x1024",
                 "gemm_ex_f32_rm_NT_4096x4096x4096", "fp8_rowscale_e4m3_4096x1536x4096",
                 "fp8_rowscale_fused_e4m3_4096x1536x4096", "fp8_rowscale_e4m3_8192x8192x8192",
                 "fp8_rowscale_fused_e4m3_8192x8192x8192"]
# Problems the oracle is also timed on with one host thread (the small
# configurations): whole problems up to ONE_THREAD_FULL_FMAS multiply-adds,
# else a bounded sample of rows.
ONE_THREAD_WORKLOADS = ["sgemm_f32_rm_256", "edge_f32_rm_1000x1000x1000", "edge_bf16_rm_1000x1000x1000",
                        "edge_f32_rm_64x64x64", "edge_bf16_rm_64x64x64"]
ONE_THREAD_FULL_FMAS = 1 << 26
SMS_NOMINAL = 152
FP32_LANES_PER_SM = 128
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0,
                  "sm_max_mhz": 2070.0}
L2_BYTES = 129e6

# DRAM traffic per call (dram__bytes_read.sum + dram__bytes_write.sum, summed over
# the kernels the call launches, the fix-up of a stream-K call excepted) from one
# ncu capture, keyed by workload; valid only while the kernel's source is the one
# captured (sha256 prefix of the .cu file's code, comments and blank lines
# removed: the family's file, or "file" where the kernel lives elsewhere), else
# reported as null.
TRAFFIC = {
    "decode_bf16_rm_8x28672x4096": {"bytes": 238219008, "source": "58dc7414ad7d", "file": "skinny_wide.cu"},
    "edge_bf16_rm_1000x1000x1000": {"bytes": 4047360, "source": "2f4b56551425"},
    "edge_bf16_rm_1x12288x4096": {"bytes": 103672576, "source": "2f4b56551425"},
    "edge_bf16_rm_32x12288x4096": {"bytes": 103931136, "source": "2f4b56551425"},
    "edge_bf16_rm_64x64x64": {"bytes": 55552, "source": "2f4b56551425"},
    "edge_bf16_rm_8192x4096x4096": {"bytes": 209809152, "source": "2f4b56551425"},
    # the A rows staged into aligned rows (pad_rows_kernel), then the CTA pairs
    "edge_bf16_rm_8192x4096x4100": {"bytes": 87304704 + 206491392, "source": "2f4b56551425"},
    "edge_f32_rm_1000x1000x1000": {"bytes": 8025856, "source": "61cf656ecb0d"},
    "edge_f32_rm_1x12288x4096": {"bytes": 204522240, "source": "a821897d27f4"},
    "edge_f32_rm_64x64x64": {"bytes": 52480, "source": "61cf656ecb0d"},
    "edge_f32_rm_8192x4096x4096": {"bytes": 723894528 + 78944000, "source": "61cf656ecb0d"},
    "edge_f32_rm_8192x4096x4100": {"bytes": 724274432 + 79040768, "source": "61cf656ecb0d"},
    "ffn_bf16_rm_1024x12288x4096": {"bytes": 121778176, "source": "2f4b56551425"},
    "ffn_gate_up_bf16_silu_mul_1024x12288x4096": {"bytes": 230824960, "source": "2f4b56551425"},  # the fix-up kernel adds 4.2 MB
    "fp8_rowscale_e4m3_4096x1536x4096": {"bytes": 23120896, "source": "2f4b56551425"},  # the quantiser moves 33.6 MB
    "fp8_rowscale_e4m3_8192x8192x8192": {"bytes": 455611264, "source": "2f4b56551425"},  # the quantiser moves 166.2 MB
    "fp8_rowscale_fused_e4m3_4096x1536x4096": {"bytes": 33559808 + 39924224, "source": "2f4b56551425"},  # the row amax pass, then the product
    "fp8_rowscale_fused_e4m3_8192x8192x8192": {"bytes": 137113856 + 729919488, "source": "2f4b56551425"},  # the row amax pass, then the product
    "gemm_ex_bf16_rm_NT_8192x8192x8192": {"bytes": 1194888448, "source": "2f4b56551425"},
    "gemm_ex_f16_rm_NN_batch32_1024x1024x1024": {"bytes": 172421632, "source": "2f4b56551425"},
    "gemm_ex_f32_rm_NT_4096x4096x4096": {"bytes": 387815680, "source": "61cf656ecb0d"},
    "gemv_bf16_rm_1x12288x4100": {"bytes": 103579904, "source": "a821897d27f4"},
    "hgemm_f16_cm_3072x5120x6144": {"bytes": 207828736, "source": "2f4b56551425"},  # the fix-up kernel adds 12.6 MB
    "hgemm_f16_cm_8192": {"bytes": 1171736320, "source": "2f4b56551425"},
    "sgemm_f32_rm_256": {"bytes": 543744, "source": "61cf656ecb0d"},
    # both grids of the call: the whole rounds and the half-K last round
    "sgemm_f32_rm_4096": {"bytes": 353438976 + 46182912, "source": "61cf656ecb0d"},
    "single_cta_bf16_rm_128x12288x4096": {"bytes": 104717824, "source": "2f4b56551425"},
    "unaligned_f32_rm_4096x4096x4095": {"bytes": 384094976, "source": "61cf656ecb0d"},
}

KERNEL_SOURCE = {
    "simt": "simt_gemm.cu",
    "umma": "umma_gemm.cu",
    "gemv": "gemv.cu",
}


def all_workloads():
    out = {}
    for name, (cfg, probs) in synthetic.WORKLOADS.items():
        out[name] = (cfg, probs[0])
    for (M, N, K) in synthetic.EDGE_SHAPES:
        for v in ("f32_rm", "bf16_rm"):
            out[f"edge_{v}_{M}x{N}x{K}"] = (synthetic.EDGE_CONFIG_ID, (v, M, N, K, "uniform", 1.0, "uniform", 1.0))
    # kernels of the dispatch table that no configuration above reaches, for
    # their profiles: the single-CTA tensor-core kernel (M = 128) and the
    # scalar-FFMA SIMT kernel (FP32 rows not 16-byte aligned: K = 4095)
    out["single_cta_bf16_rm_128x12288x4096"] = (synthetic.EDGE_CONFIG_ID, ("bf16_rm", 128, 12288, 4096, "uniform",
                                                                         1.0, "uniform", 1.0))
    out["unaligned_f32_rm_4096x4096x4095"] = (synthetic.EDGE_CONFIG_ID, ("f32_rm", 4096, 4096, 4095, "uniform", 1.0,
                                                                       "uniform", 1.0))
    # a decode batch whose 128-column strips outnumber the SMs (the 256-column
    # skinny kernel), and the GEMV's bf16 instance (A rows of 8200 bytes, which
    # TMA cannot describe, keep M = 1 off the tensor cores)
    out["decode_bf16_rm_8x28672x4096"] = (synthetic.EDGE_CONFIG_ID, ("bf16_rm", 8, 28672, 4096, "uniform", 1.0,
                                                                   "uniform", 1.0))
    out["gemv_bf16_rm_1x12288x4100"] = (synthetic.EDGE_CONFIG_ID, ("bf16_rm", 1, 12288, 4100, "uniform", 1.0,
                                                                 "uniform", 1.0))
    # the FFN gate/up projection with its SiLU * U epilogue fused (two GEMMs)
    out["ffn_gate_up_bf16_silu_mul_1024x12288x4096"] = (3, ("bf16_silu_mul", 1024, 12288, 4096, "normal", 1.0,
                                                             "normal", 1.0 / 64.0))
    # the row-scaled FP8 projection of example 5-8: A [4096,4096] half quantised
    # row-wise to E4M3, times E4M3 weights [4096,1536], half output
    out["fp8_rowscale_e4m3_4096x1536x4096"] = (5, ("e4m3_rowscale", 4096, 1536, 4096, "normal", 1.0,
                                                    "uniform", 1.0))
    # the same step with the quantisation fused into the product's load path
    # (example 5-8's second scheme), and both schemes on a large square problem
    out["fp8_rowscale_fused_e4m3_4096x1536x4096"] = (5, ("e4m3_fused", 4096, 1536, 4096, "normal", 1.0,
                                                          "uniform", 1.0))
    out["fp8_rowscale_e4m3_8192x8192x8192"] = (5, ("e4m3_rowscale", 8192, 8192, 8192, "normal", 1.0,
                                                    "uniform", 1.0))
    out["fp8_rowscale_fused_e4m3_8192x8192x8192"] = (5, ("e4m3_fused", 8192, 8192, 8192, "normal", 1.0,
                                                          "uniform", 1.0))
    # the general form (gemm_ex): a linear layer's X W^T with W stored [N, K],
    # a strided batch, and FP32 with a transposed B on the SIMT kernel
    for dtype, ops, batch, (M, N, K) in (("bf16", "NT", 1, (8192, 8192, 8192)),
                                         ("f16", "NN", 32, (1024, 1024, 1024)),
                                         ("f32", "NT", 1, (4096, 4096, 4096))):
        tag = f"gemm_ex_{dtype}_rm_{ops}" + (f"_batch{batch}" if batch > 1 else "") + f"_{M}x{N}x{K}"
        out[tag] = (synthetic.EDGE_CONFIG_ID, (f"ex:{dtype}:rm:{ops[0]}:{ops[1]}:{batch}", M, N, K,
                                               "uniform", 1.0, "uniform", 1.0))
    return out


def ex_parse(variant: str):
    """'ex:<dtype>:<layout>:<op_a>:<op_b>:<batch>' -> its fields (batch as int)."""
    _, dtype, layout, op_a, op_b, batch = variant.split(":")
    return dtype, layout, op_a, op_b, int(batch)


def read_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            d = json.load(f)
        return d, "measured"
    return dict(FALLBACK_PEAKS), "fallback"


def code_text(src: str) -> str:
    """C/C++/CUDA source without its comments and blank lines, each line stripped:
    what the compiler sees, so that editing a comment keeps a capture valid."""
    out, i, n = [], 0, len(src)
    in_str = in_chr = False
    while i < n:
        c = src[i]
        if in_str or in_chr:
            out.append(c)
            if c == "\\" and i + 1 < n:
                out.append(src[i + 1])
                i += 2
                continue
            if (in_str and c == '"') or (in_chr and c == "'"):
                in_str = in_chr = False
            i += 1
        elif src.startswith("//", i):
            j = src.find("\n", i)
            i = n if j < 0 else j
        elif src.startswith("/*", i):
            j = src.find("*/", i + 2)
            i = n if j < 0 else j + 2
        else:
            in_str, in_chr = c == '"', c == "'"
            out.append(c)
            i += 1
    return "\n".join(line.strip() for line in "".join(out).splitlines() if line.strip())


def file_hash(name: str) -> str:
    """sha256 prefix of a kernel file's code (comments and blank lines removed)."""
    path = os.path.join(ROOT, "dense_matrix_multiply_gb300", "csrc", name)
    with open(path, encoding="utf-8") as f:
        return hashlib.sha256(code_text(f.read()).encode()).hexdigest()[:12]


def source_hash(kind: str) -> str:
    """Code hash of the file that holds a kernel family."""
    return file_hash(KERNEL_SOURCE[kind])


# ------------------------------------------------------------------ clocks
class ClockSampler:
    """nvidia-smi sampling of SM clock and throttle reasons in the background."""

    FIELDS = ["timestamp", "uuid", "clocks.sm", "clocks.max.sm", "power.draw",
              "clocks_event_reasons.active", "clocks_event_reasons.hw_slowdown",
              "clocks_event_reasons.hw_thermal_slowdown", "clocks_event_reasons.sw_thermal_slowdown",
              "clocks_event_reasons.sw_power_cap"]

    def __init__(self, uuid: str | None, period_ms: int = 50):
        self.uuid = uuid
        self.proc = None
        self.file = tempfile.NamedTemporaryFile("w+", suffix=".csv", delete=False)
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "--query-gpu=" + ",".join(self.FIELDS), "--format=csv,noheader,nounits",
                 "-lms", str(period_ms)], stdout=self.file, stderr=subprocess.DEVNULL)
        except OSError:
            self.proc = None

    def stop(self):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
        self.file.flush()

    def summary(self, t0: float, t1: float):
        """Median SM MHz and the throttle reasons seen between host times t0 and t1."""
        self.file.seek(0)
        rows = list(csv.reader(io.StringIO(self.file.read())))
        try:
            os.unlink(self.file.name)
        except OSError:
            pass
        mhz, maxmhz, reasons, power = [], [], set(), []
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for r in rows:
            if len(r) < len(self.FIELDS):
                continue
            r = [x.strip() for x in r]
            try:
                ts = datetime.strptime(r[0], "%Y/%m/%d %H:%M:%S.%f").timestamp()
            except ValueError:
                continue
            if self.uuid and r[1] != self.uuid:
                continue
            if not (t0 - 0.05 <= ts <= t1 + 0.05):
                continue
            try:
                mhz.append(float(r[2]))
                maxmhz.append(float(r[3]))
                power.append(float(r[4]))
            except ValueError:
                continue
            for name, val in zip(names, r[6:10]):
                if val.lower() == "active":
                    reasons.add(name)
        if not mhz:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        return {"sm_mhz": statistics.median(mhz), "sm_max_mhz": max(maxmhz), "reasons": sorted(reasons),
                "samples": len(mhz), "power_w_max": max(power) if power else None}


# ------------------------------------------------------------------ helpers
def device_inputs(variant, A, B, M, N):
    import torch
    if variant.startswith("f32"):
        dA, dB = torch.from_numpy(A).cuda(), torch.from_numpy(B).cuda()
        dC = torch.empty(M * N, dtype=torch.float32, device="cuda")
    else:
        dA = torch.from_numpy(A.view(np.int16)).cuda()
        dB = torch.from_numpy(B.view(np.int16)).cuda()
        dC = torch.empty(M * N, dtype=torch.int16, device="cuda")
    return dA, dB, dC


ENTRY = {"f32_rm": "gemm_f32_rm", "f16_cm": "gemm_f16_cm", "bf16_rm": "gemm_bf16_rm"}


def kernel_kind(name: str) -> str:
    return name.split("_")[0]


def roofline_for(kind: str, variant: str, M, N, K, seconds_per_launch: float, peaks: dict, peaks_src: str,
                 sm_mhz: float | None, sms: int, workload: str, prop_mhz: float | None = None):
    es = 4 if variant.startswith("f32") or variant.startswith("ex:f32") else 2
    if variant == "bf16_silu_mul":  # two products, X read once: X, W_g, W_u, Z
        flops = 2 * metrics.gemm_flops(M, N, K)
        algo_bytes = es * (M * K + 2 * K * N + M * N)
    elif variant == "e4m3_rowscale":  # the product kernel: Q, W codes, the row scales, half C
        flops = metrics.gemm_flops(M, N, K)
        algo_bytes = M * K + K * N + 4 * M + 2 * M * N
    elif variant == "e4m3_fused":  # the whole fused step: half A once, W codes, half C
        flops = metrics.gemm_flops(M, N, K)
        algo_bytes = 2 * M * K + K * N + 2 * M * N
    elif variant.startswith("ex:"):  # batch independent products, beta = 0 (C not read)
        batch = ex_parse(variant)[4]
        flops = batch * metrics.gemm_flops(M, N, K)
        algo_bytes = batch * metrics.min_bytes(M, N, K, es)
    else:
        flops = metrics.gemm_flops(M, N, K)
        algo_bytes = metrics.min_bytes(M, N, K, es)
    tr = TRAFFIC.get(workload)
    traffic = None
    src_file = tr.get("file") if tr else None
    if tr and tr.get("source") == (file_hash(src_file) if src_file else
                                   source_hash(kind if kind in KERNEL_SOURCE else "simt")):
        traffic = tr["bytes"]
    if kind == "gemv":
        achieved = algo_bytes / seconds_per_launch / 1e9
        peak = float(peaks["hbm_gbs"])
        return {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s", "frac": achieved / peak,
                "traffic": traffic, "algorithmic_bytes": algo_bytes, "peak_source": peaks_src}
    if kind == "umma":
        # below the ridge point (FLOPs per byte at which the measured tensor and
        # HBM peaks meet) the tensor-core kernel is bound by HBM: skinny M
        tpeak = float(peaks["bf16_tflops"]) * (2.0 if variant in ("e4m3_rowscale", "e4m3_fused") else 1.0)
        if flops / algo_bytes < tpeak * 1e12 / (float(peaks["hbm_gbs"]) * 1e9):
            achieved = algo_bytes / seconds_per_launch / 1e9
            peak = float(peaks["hbm_gbs"])
            return {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s", "frac": achieved / peak,
                    "traffic": traffic, "algorithmic_bytes": algo_bytes, "algorithmic_flops": flops,
                    "peak_source": peaks_src}
    achieved = flops / seconds_per_launch / 1e12
    if kind == "umma" and variant in ("e4m3_rowscale", "e4m3_fused"):
        # dense FP8 rate = 2 x the dense BF16 rate (4.5 vs 2.25 PFLOP/s nominal)
        peak = 2.0 * float(peaks["bf16_tflops"])
        return {"bound": "tensor", "achieved": achieved, "peak": peak, "unit": "TFLOP/s",
                "frac": achieved / peak, "traffic": traffic, "algorithmic_flops": flops,
                "algorithmic_bytes": algo_bytes,
                "peak_source": f"{peaks_src} cuBLAS bf16 burst x 2 (nominal FP8/BF16 dense ratio)"}
    if kind == "umma":
        peak = float(peaks["bf16_tflops"])
        return {"bound": "tensor", "achieved": achieved, "peak": peak, "unit": "TFLOP/s",
                "frac": achieved / peak, "traffic": traffic, "algorithmic_flops": flops,
                "algorithmic_bytes": algo_bytes, "peak_source": f"{peaks_src} cuBLAS bf16 burst"
                + (" (f16 dense rate equals bf16)" if variant.startswith("f16") else "")}
    # SIMT FP32: SMs x 128 lanes x 2 FLOP x clock
    max_mhz = float(peaks.get("sm_max_mhz", FALLBACK_PEAKS["sm_max_mhz"]))
    peak = metrics.simt_fp32_peak(sms, max_mhz * 1e6, FP32_LANES_PER_SM) / 1e12
    out = {"bound": "alu", "achieved": achieved, "peak": peak, "unit": "TFLOP/s", "frac": achieved / peak,
           "traffic": traffic, "algorithmic_flops": flops, "algorithmic_bytes": algo_bytes,
           "peak_source": f"{sms} SMs x {FP32_LANES_PER_SM} FP32 lanes x 2 x {max_mhz:.0f} MHz (max SM clock)"}
    if prop_mhz:
        # the pages' main convention: the clock the device reports (cudaDevAttrClockRate)
        p1 = metrics.simt_fp32_peak(sms, prop_mhz * 1e6, FP32_LANES_PER_SM) / 1e12
        out["peak_at_device_prop_clock"] = p1
        out["frac_at_device_prop_clock"] = achieved / p1
        out["device_prop_clock_mhz"] = prop_mhz
    if sm_mhz:
        # numerator and denominator at the clock sampled during the timed region
        p2 = metrics.simt_fp32_peak(sms, sm_mhz * 1e6, FP32_LANES_PER_SM) / 1e12
        out["peak_at_measured_clock"] = p2
        out["frac_at_measured_clock"] = achieved / p2
        out["measured_clock_mhz"] = sm_mhz
    return out


def time_device(fn, steps: int, warmup: int, stream):
    """CUDA-event time of `steps` calls on `stream` after `warmup` calls: ms total."""
    import torch
    for _ in range(warmup):
        fn()
    torch.cuda.synchronize()
    start = torch.cuda.Event(enable_timing=True)
    end = torch.cuda.Event(enable_timing=True)
    start.record(stream)
    for _ in range(steps):
        fn()
    end.record(stream)
    torch.cuda.synchronize()
    return start.elapsed_time(end)


_FLUSH = None


def time_device_flushed(fn, steps: int, warmup: int, stream):
    """CUDA-event time of `steps` calls on `stream`, each timed on its own with
    the L2 flushed before it (a read of a 512 MiB buffer, four times the L2,
    leaving clean lines so that the timed call pays no write-backs): ms total,
    launch latency of every call included.  For problems that fit in L2."""
    import torch
    global _FLUSH
    if _FLUSH is None:
        _FLUSH = (torch.ones(512 * 1024 * 1024 // 4, device="cuda"), torch.empty(1, device="cuda"))
    buf, sink = _FLUSH
    for _ in range(warmup):
        fn()
    torch.cuda.synchronize()
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(steps)]
    for e0, e1 in evs:
        with torch.cuda.stream(stream):
            torch.sum(buf, dim=0, out=sink)
        e0.record(stream)
        fn()
        e1.record(stream)
    torch.cuda.synchronize()
    return sum(e0.elapsed_time(e1) for e0, e1 in evs)


def spread_stats(times_ms):
    """Median, 10th and 90th percentiles and coefficient of variation of
    per-call times (ms); `noisy` when the variation exceeds 2 %."""
    t = np.sort(np.asarray(times_ms, dtype=np.float64))
    mean = float(t.mean())
    cv = float(t.std() / mean) if mean > 0 else 0.0
    return {"calls": int(t.size), "median_ms": float(np.median(t)), "p10_ms": float(np.percentile(t, 10)),
            "p90_ms": float(np.percentile(t, 90)), "cv": cv, "noisy": cv > 0.02}


def per_call_times(fn, calls: int, stream, flushed: bool):
    """Each of `calls` calls between its own pair of CUDA events on `stream`
    (after the L2 flush when `flushed`): ms per call.  A pass of its own after
    the timed region, whose back-to-back calls overlap one another."""
    import torch
    global _FLUSH
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(calls)]
    sink = None
    if flushed:
        if _FLUSH is None:
            _FLUSH = (torch.ones(512 * 1024 * 1024 // 4, device="cuda"), torch.empty(1, device="cuda"))
        buf, sink = _FLUSH
    torch.cuda.synchronize()
    for e0, e1 in evs:
        if sink is not None:
            with torch.cuda.stream(stream):
                torch.sum(buf, dim=0, out=sink)
        e0.record(stream)
        fn()
        e1.record(stream)
    torch.cuda.synchronize()
    return [e0.elapsed_time(e1) for e0, e1 in evs]


def host_inputs(variant, cfg, M, N, K, da, sa, db, sb):
    """Seeded host buffers of a workload: (A, B, extra)."""
    if variant == "bf16_silu_mul":
        A = synthetic.matrix("bf16", M, K, synthetic.seed_for(cfg, 1), da, sa)
        B = synthetic.matrix("bf16", K, N, synthetic.seed_for(cfg, 2), db, sb)
        return A, B, (synthetic.matrix("bf16", K, N, synthetic.seed_for(cfg, 3), db, sb),)
    if variant in ("e4m3_rowscale", "e4m3_fused"):
        A = synthetic.matrix("f16", M, K, synthetic.seed_for(cfg, 1), da, sa)
        return A, synthetic.e4m3_codes(N, K, synthetic.seed_for(cfg, 2)), ()
    if variant.startswith("ex:"):
        dtype, _, _, _, batch = ex_parse(variant)
        A = synthetic.matrix(dtype, batch * M, K, synthetic.seed_for(cfg, 5), da, sa)
        B = synthetic.matrix(dtype, batch * K, N, synthetic.seed_for(cfg, 6), db, sb)
        return A, B, ()
    A, B = synthetic.problem_inputs(variant, M, N, K, cfg, da, sa, db, sb)
    return A, B, ()


def oracle_rows(variant, A, B, M, N, K, rows, extra=()):
    """The oracle on output rows `rows` (for a batched workload: rows 0..len-1
    of the first batch entry).  Returns (the FLOPs that took, (C_ref, S) of
    those rows for the three plain variants, else None)."""
    import oracle
    if variant == "bf16_silu_mul":
        oracle.silu_mul(A, B, extra[0], M, N, K, rows=rows)
        return 4.0 * len(rows) * N * K, None
    if variant in ("e4m3_rowscale", "e4m3_fused"):  # quantise the rows, then their products
        a = np.ascontiguousarray(A.reshape(M, K)[rows])
        Q, S = oracle.quantize_rows_e4m3(a, len(rows), K)
        oracle.gemm_e4m3_rowscale(Q, S, B, len(rows), N, K)
        return 2.0 * len(rows) * N * K, None
    if variant.startswith("ex:"):
        dtype, layout, op_a, op_b, _ = ex_parse(variant)
        m = len(rows)
        lda = M if op_a == "T" else K
        ldb = K if op_b == "T" else N
        oracle.gemm_ex(dtype, layout, op_a, op_b, m, N, K, 1.0, A[:M * K], lda, 0, B[:K * N], ldb, 0, 0.0,
                       None, N, 0, 1)
        return 2.0 * m * N * K, None
    ref = oracle.gemm_rows(variant, A, B, M, N, K, rows)
    return 2.0 * len(rows) * N * K, ref


def sample_rows(M: int, n: int) -> np.ndarray:
    """n distinct output rows spread evenly over 0..M-1, first and last included."""
    n = max(1, min(int(n), M))
    if n == 1:
        return np.zeros(1, dtype=np.int64)
    return (np.arange(n, dtype=np.int64) * (M - 1)) // (n - 1)


def cpu_sample(variant, A, B, M, N, K, budget_s: float, extra=()):
    """Times the oracle on a bounded sample of output rows of the same problem,
    spread over all of M.  Returns (flop/s, rows, seconds, threads, the rows,
    their (C_ref, S) or None)."""
    import oracle
    threads = oracle.num_threads()
    # calibrate on one row per thread
    rows = np.arange(min(threads, M), dtype=np.int64)
    t0 = time.perf_counter()
    oracle_rows(variant, A, B, M, N, K, rows, extra)
    dt = time.perf_counter() - t0
    per_round = max(dt, 1e-6)
    rounds = max(1, int(budget_s / per_round))
    nrows = int(min(M, rows.size * rounds))
    sel = sample_rows(M, nrows)
    t0 = time.perf_counter()
    fl, ref = oracle_rows(variant, A, B, M, N, K, sel, extra)
    dt = time.perf_counter() - t0
    return fl / dt, nrows, dt, threads, sel, ref


def sample_parity(variant, host_c, M, N, K, rows, ref):
    """The library's C (host copy of the timed output buffer: float32, or half /
    bf16 bits as int16) on the oracle's sampled rows, against the oracle within
    the variant's tolerance."""
    from oracle import compare
    C_ref, S = ref
    c = np.asarray(host_c)
    if variant == "f32_rm":
        got = c.astype(np.float64).reshape(M, N)[rows]
    elif variant == "bf16_rm":
        got = (c.view(np.uint16).astype(np.uint32) << 16).view(np.float32).astype(np.float64).reshape(M, N)[rows]
    elif variant == "f16_cm":  # column-major: element (i, j) at i + j*M
        got = c.view(np.float16).astype(np.float64).reshape(N, M).T[rows]
    else:
        raise ValueError(variant)
    r = compare.check(variant, got, C_ref, S, K)
    return {"rows": int(len(rows)), "elements": int(got.size), "ok": bool(r["ok"]),
            "max_err_over_tol": float(r["max_err_over_tol"])}


def e2e_pipelined(fn, h_in, d_in, dC, hC, M, N, K, stream, steps, flops):
    """End-to-end throughput with copies overlapped across steps: step i copies
    its inputs from pinned host memory into buffer set i % 2 (its own stream),
    computes on the library's stream once they have landed, and copies its
    result back to pinned host memory (a third stream).  Every step's copies are
    inside the timed region."""
    import torch
    sets = [list(d_in) + [dC], [t.clone() for t in d_in] + [torch.empty_like(dC)]]
    hCs = [hC, torch.empty_like(hC).pin_memory()]
    s_h2d, s_d2h = torch.cuda.Stream(), torch.cuda.Stream()
    ev_in = [torch.cuda.Event(), torch.cuda.Event()]
    ev_done = [torch.cuda.Event(), torch.cuda.Event()]
    ev_out = [torch.cuda.Event(), torch.cuda.Event()]

    def run(n):
        for i in range(n):
            k = i % 2
            if i >= 2:
                s_h2d.wait_event(ev_done[k])          # set k's inputs are no longer read
            with torch.cuda.stream(s_h2d):
                for h, d in zip(h_in, sets[k][:-1]):
                    d.copy_(h, non_blocking=True)
                ev_in[k].record(s_h2d)
            stream.wait_event(ev_in[k])
            if i >= 2:
                stream.wait_event(ev_out[k])          # set k's previous result was read out
            st = fn(*[t.data_ptr() for t in sets[k]], M, N, K)
            if st != 0:
                raise RuntimeError(f"library status {st}")
            ev_done[k].record(stream)
            s_d2h.wait_event(ev_done[k])
            with torch.cuda.stream(s_d2h):
                hCs[k].copy_(sets[k][-1], non_blocking=True)
                ev_out[k].record(s_d2h)

    run(2)
    torch.cuda.synchronize()
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    start.record(s_h2d)
    run(steps)
    end.record(s_d2h)
    torch.cuda.synchronize()
    ms = start.elapsed_time(end)
    return {"value": flops * steps / (ms / 1e3) / 1e12, "unit": "TFLOP/s", "ms_per_step": ms / steps,
            "steps": steps, "overlap": "host->device copy of step i+1 and device->host copy of step i-1 "
                                       "run during step i (three streams, two buffer sets)"}


# ------------------------------------------------------------------ cuBLAS column
class Cublas:
    """cuBLAS, timed beside the library as a reference column (outside the
    library, never on its path): FP32 SGEMM in pedantic math (no TF32, as the
    pages' cuBLAS baseline), half and bf16 through cublasGemmEx with FP32
    compute and default math.  Row-major problems use the identity C^T = B^T A^T
    ("SGEMM measured and the three ledgers", section 2)."""

    OP_N, R_32F, R_16F, R_16BF, COMPUTE_32F, GEMM_DEFAULT = 0, 0, 2, 14, 68, -1
    DEFAULT_MATH, PEDANTIC_MATH = 0, 2

    def __init__(self):
        import ctypes
        import glob
        self.ct = ctypes
        cands = glob.glob("/usr/local/cuda/lib64/libcublas.so*")
        try:
            import nvidia
            for d in nvidia.__path__:
                cands += glob.glob(os.path.join(d, "cublas", "lib", "libcublas.so*"))
        except ImportError:
            pass
        self.lib, err = None, "libcublas not found"
        for c in sorted(cands, key=len):
            try:
                self.lib = ctypes.CDLL(c)
                break
            except OSError as e:
                err = str(e)
        if self.lib is None:
            raise RuntimeError(err)
        self.handle = ctypes.c_void_p()
        if self.lib.cublasCreate_v2(ctypes.byref(self.handle)) != 0:
            raise RuntimeError("cublasCreate failed")
        vp, i, ll = ctypes.c_void_p, ctypes.c_int, ctypes.c_longlong
        self.lib.cublasSgemm_v2.argtypes = [vp, i, i, i, i, i, vp, vp, i, vp, i, vp, vp, i]
        self.lib.cublasGemmEx.argtypes = [vp, i, i, i, i, i, vp, vp, i, i, vp, i, i, vp, vp, i, i, i, i]
        self.lib.cublasSetStream_v2.argtypes = [vp, vp]
        self.lib.cublasSetMathMode.argtypes = [vp, i]
        self.one = ctypes.c_float(1.0)
        self.zero = ctypes.c_float(0.0)

    def call(self, variant, M, N, K, pa, pb, pc):
        ct, lib, h = self.ct, self.lib, self.handle
        one, zero = ct.byref(self.one), ct.byref(self.zero)
        if variant == "f32_rm":
            lib.cublasSetMathMode(h, self.PEDANTIC_MATH)
            return lib.cublasSgemm_v2(h, self.OP_N, self.OP_N, N, M, K, one, pb, N, pa, K, zero, pc, N)
        lib.cublasSetMathMode(h, self.DEFAULT_MATH)
        if variant == "f16_cm":
            return lib.cublasGemmEx(h, self.OP_N, self.OP_N, M, N, K, one, pa, self.R_16F, M, pb, self.R_16F, K,
                                    zero, pc, self.R_16F, M, self.COMPUTE_32F, self.GEMM_DEFAULT)
        # bf16 row-major
        return lib.cublasGemmEx(h, self.OP_N, self.OP_N, N, M, K, one, pb, self.R_16BF, N, pa, self.R_16BF, K,
                                zero, pc, self.R_16BF, N, self.COMPUTE_32F, self.GEMM_DEFAULT)

    def measure(self, variant, M, N, K, dA, dB, dC_like, stream, steps, flushed=False, sets=None):
        """{"tflops", "ms_per_step", "mode", "max_abs_diff_vs_library"}: cuBLAS on the
        same device inputs, timed like the library (CUDA events, same stream)."""
        import torch
        self.lib.cublasSetStream_v2(self.handle, self.ct.c_void_p(stream.cuda_stream))
        out = torch.empty_like(dC_like)
        pc = out.data_ptr()
        ab = sets or [(dA.data_ptr(), dB.data_ptr())]   # rotated like the library's calls
        i = [0]

        def step():
            pa, pb = ab[i[0] % len(ab)]
            i[0] += 1
            st = self.call(variant, M, N, K, pa, pb, pc)
            if st != 0:
                raise RuntimeError(f"cuBLAS status {st}")

        ms = (time_device_flushed if flushed else time_device)(step, steps, 3, stream)
        torch.cuda.synchronize()
        if variant == "f32_rm":
            diff = (out - dC_like).abs().max().item()
        else:
            dt = torch.float16 if variant.startswith("f16") else torch.bfloat16
            diff = (out.view(dt).float() - dC_like.view(dt).float()).abs().max().item()
        mode = "FP32, CUBLAS_PEDANTIC_MATH" if variant == "f32_rm" else "cublasGemmEx, FP32 compute, default math"
        return {"tflops": metrics.gemm_flops(M, N, K) / (ms / 1e3 / steps) / 1e12, "ms_per_step": ms / steps,
                "mode": mode, "max_abs_diff_vs_library": diff}


_CUBLAS = None


def cublas_column(variant, M, N, K, dA, dB, dC, stream, steps, flushed=False, sets=None):
    global _CUBLAS
    if variant not in ("f32_rm", "f16_cm", "bf16_rm"):
        return None
    try:
        if _CUBLAS is None:
            _CUBLAS = Cublas()
        return _CUBLAS.measure(variant, M, N, K, dA, dB, dC, stream, steps, flushed, sets)
    except Exception as e:  # a reference column only: report why it is missing
        return {"unavailable": str(e)[:200]}


# ------------------------------------------------------------------ replicas
def slowest_rank_ms(ms: float, world: int, device: str = "cpu") -> float:
    """The timed region's length on the slowest rank (every rank gets it)."""
    if world <= 1:
        return ms
    import torch
    import torch.distributed as dist
    t = torch.tensor([ms], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def replica_throughput(flops_per_step: float, steps: int, world: int, ms_slowest: float) -> float:
    """Whole-job TFLOP/s of `world` independent replicas (weak scaling): the FLOPs
    of all ranks divided by the slowest rank's time."""
    return flops_per_step * steps * world / (ms_slowest / 1e3) / 1e12


# ------------------------------------------------------------------ our arm
def measure_workload(name, steps, warmup, peaks, peaks_src, sms, stream, sampler_uuid=None, e2e=True,
                     cpu_budget=0.0, clocks=True, prop_mhz=None, cublas=True):
    import torch
    import dense_matrix_multiply_gb300 as g

    cfg, (variant, M, N, K, da, sa, db, sb) = all_workloads()[name]
    g.gemm_set_stream(stream)
    extra = []
    if variant == "bf16_silu_mul":
        A = synthetic.matrix("bf16", M, K, synthetic.seed_for(cfg, 1), da, sa)
        B = synthetic.matrix("bf16", K, N, synthetic.seed_for(cfg, 2), db, sb)
        Wu = synthetic.matrix("bf16", K, N, synthetic.seed_for(cfg, 3), db, sb)
        dA, dB, dC = device_inputs("bf16_rm", A, B, M, N)
        dWu = torch.from_numpy(Wu.view(np.int16)).cuda()
        extra = [Wu]
        fn = g.load().gemm_bf16_rm_silu_mul
        pa, pb, pu, pc = dA.data_ptr(), dB.data_ptr(), dWu.data_ptr(), dC.data_ptr()

        def call():
            return fn(pa, pb, pu, pc, M, N, K)
    elif variant == "e4m3_rowscale":
        # one step: quantise A row-wise (E4M3 codes + row scales), then the FP8 product
        A, B, _ = host_inputs(variant, cfg, M, N, K, da, sa, db, sb)
        dA = torch.from_numpy(A.view(np.int16)).cuda()
        dB = torch.from_numpy(B).cuda()
        dQ = torch.empty(M * K, dtype=torch.uint8, device="cuda")
        dS = torch.empty(M, dtype=torch.float32, device="cuda")
        dC = torch.empty(M * N, dtype=torch.int16, device="cuda")
        lib = g.load()
        pa, pb, pq, ps, pc = dA.data_ptr(), dB.data_ptr(), dQ.data_ptr(), dS.data_ptr(), dC.data_ptr()

        e4_sets = [(pa, pb, pq, ps, pc)]
        e4_i = [0, 0]  # rotation counters of quantize() and product()

        def quantize():
            a, _, q, sc, _ = e4_sets[e4_i[0] % len(e4_sets)]
            e4_i[0] += 1
            return lib.gemm_quantize_rows_e4m3(a, q, sc, M, K)

        def product():
            _, b, q, sc, c = e4_sets[e4_i[1] % len(e4_sets)]
            e4_i[1] += 1
            return lib.gemm_e4m3_rowscale(q, sc, b, c, M, N, K)

        def call():
            return quantize() or product()
    elif variant == "e4m3_fused":
        # one step: the row amax pass and the product that quantises A as it loads it
        A, B, _ = host_inputs(variant, cfg, M, N, K, da, sa, db, sb)
        dA = torch.from_numpy(A.view(np.int16)).cuda()
        dB = torch.from_numpy(B).cuda()
        dC = torch.empty(M * N, dtype=torch.int16, device="cuda")
        fused_fn = g.load().gemm_e4m3_rowscale_fused
        plain_sets = [(dA.data_ptr(), dB.data_ptr(), dC.data_ptr())]
        plain_i = [0]

        def call():
            pa_, pb_, pc_ = plain_sets[plain_i[0] % len(plain_sets)]
            plain_i[0] += 1
            return fused_fn(pa_, pb_, pc_, M, N, K)
    elif variant.startswith("ex:"):
        # tight strides: A stored [M,K] or [K,M], B [K,N] or [N,K], batch matrices back to back
        dtype, layout, op_a, op_b, batch = ex_parse(variant)
        A, B, _ = host_inputs(variant, cfg, M, N, K, da, sa, db, sb)
        dA, dB, dC = device_inputs(dtype + "_rm", A, B, batch * M, N)
        lda = M if op_a == "T" else K
        ldb = K if op_b == "T" else N
        fn = g.load().gemm_ex
        args_ex = (g.DTYPES[dtype], g.LAYOUTS[layout], g.OPS[op_a], g.OPS[op_b], M, N, K, 1.0,
                   dA.data_ptr(), lda, M * K, dB.data_ptr(), ldb, K * N, 0.0, dC.data_ptr(), N, M * N, batch)

        def call():
            return fn(*args_ex)
    else:
        A, B = synthetic.problem_inputs(variant, M, N, K, cfg, da, sa, db, sb)
        dA, dB, dC = device_inputs(variant, A, B, M, N)
        fn = getattr(g.load(), ENTRY[variant])
        plain_sets = [(dA.data_ptr(), dB.data_ptr(), dC.data_ptr())]
        plain_i = [0]

        def call():
            pa_, pb_, pc_ = plain_sets[plain_i[0] % len(plain_sets)]
            plain_i[0] += 1
            return fn(pa_, pb_, pc_, M, N, K)

    def step():
        st = call()
        if st != 0:
            raise RuntimeError(f"{name} failed: {g.gemm_status_string(st)} {g.gemm_last_error()}")

    step()
    g.gemm_synchronize()
    kernel = g.gemm_last_kernel()
    kind = kernel_kind(kernel)

    footprint = sum(t.numel() * t.element_size() for t in [dA, dB, dC] + ([dWu] if extra else [])
                    + ([dQ, dS] if variant == "e4m3_rowscale" else []))
    # Operands that fit in L2 would stay there between calls.  Then the calls
    # rotate over R copies of them, R x footprint > 3 x L2, so that every call
    # reads its operands from DRAM (as consecutive layers of a model would),
    # timed back to back.
    rotated = 1
    keep = []
    if footprint <= L2_BYTES and (variant in ENTRY or variant in ("e4m3_rowscale", "e4m3_fused")):
        rotated = int(min(512, -(-3 * int(L2_BYTES) // max(1, footprint))))
        for _ in range(rotated - 1):
            if variant in ENTRY or variant == "e4m3_fused":
                a2, b2, c2 = dA.clone(), dB.clone(), torch.empty_like(dC)
                keep += [a2, b2, c2]
                plain_sets.append((a2.data_ptr(), b2.data_ptr(), c2.data_ptr()))
            else:
                a2, b2, q2, s2, c2 = dA.clone(), dB.clone(), torch.empty_like(dQ), torch.empty_like(dS), \
                    torch.empty_like(dC)
                keep += [a2, b2, q2, s2, c2]
                e4_sets.append((a2.data_ptr(), b2.data_ptr(), q2.data_ptr(), s2.data_ptr(), c2.data_ptr()))
    flushed = footprint <= L2_BYTES and rotated == 1
    split = {}
    if variant == "e4m3_rowscale":
        # each kernel of the step timed on its own: the product is the dominant
        # (tensor-bound) kernel, the quantisation is HBM-bound
        for nm, fn1 in (("quantize", quantize), ("product", product)):
            ms1 = (time_device_flushed if flushed else time_device)(fn1, steps, 3, stream)
            split[nm] = ms1 / steps
    sampler = ClockSampler(sampler_uuid) if clocks else None
    for _ in range(warmup):
        step()
    torch.cuda.synchronize()
    time.sleep(0.2 if clocks else 0)
    t_host0 = time.time()
    launches0 = g.gemm_kernel_launches()
    ms = (time_device_flushed if flushed else time_device)(step, steps, 0, stream)
    launches = g.gemm_kernel_launches() - launches0  # the library's own count of its launches
    t_host1 = time.time()
    g.gemm_synchronize()
    clk = None
    if sampler:
        time.sleep(0.1)
        sampler.stop()
        clk = sampler.summary(t_host0, t_host1)

    flops = metrics.gemm_flops(M, N, K) * (2 if variant == "bf16_silu_mul" else
                                           ex_parse(variant)[4] if variant.startswith("ex:") else 1)
    s_per = ms / 1e3 / steps
    s_kernel = split["product"] / 1e3 if split else s_per
    res = {
        "workload": name, "variant": variant, "M": M, "N": N, "K": K, "kernel": kernel, "flops_per_step": flops,
        "ms_per_step": ms / steps, "tflops": flops / s_per / 1e12, "steps": steps, "ms_total": ms,
        "roofline": roofline_for(kind, variant, M, N, K, s_kernel, peaks, peaks_src,
                                 clk["sm_mhz"] if clk else None, sms, name, prop_mhz),
        "clocks": clk, "footprint_bytes": int(footprint), "gpu_launches": int(launches),
        "l2": (f"{footprint / 2**20:.1f} MiB of operands fit in the 129 MB L2: calls rotate over {rotated} "
               f"copies ({rotated * footprint / 2**20:.0f} MiB), each read from DRAM, back to back"
               if rotated > 1 else
               f"flushed before every timed call (read of a 512 MiB buffer): {footprint / 2**20:.0f} MiB of "
               f"operands fit in the 129 MB L2" if flushed else
               f"no flush: {footprint / 2**20:.0f} MiB of operands > 129 MB L2"),
    }

    try:
        res["per_call"] = spread_stats(per_call_times(step, min(steps, 100), stream, flushed))
    except Exception as exc:  # the line is still printed; the failure is named in it
        res["per_call"] = {"error": f"{type(exc).__name__}: {exc}"[:200]}

    if cublas and variant in ("f32_rm", "f16_cm", "bf16_rm"):
        res["cublas"] = cublas_column(variant, M, N, K, dA, dB, dC, stream, steps, flushed,
                                      [(p_[0], p_[1]) for p_ in plain_sets] if variant in ENTRY else None)
    if split:
        q_bytes = 2 * M * K + M * K + 4 * M  # read A once, write the codes and the scales
        res["kernels"] = {
            "quantize_e4m3": {"ms": split["quantize"], "GB/s": q_bytes / (split["quantize"] / 1e3) / 1e9,
                              "frac_hbm": q_bytes / (split["quantize"] / 1e3) / 1e9 / float(peaks["hbm_gbs"]),
                              "algorithmic_bytes": q_bytes},
            "umma_e4m3_rowscale": {"ms": split["product"], "TFLOP/s": flops / (split["product"] / 1e3) / 1e12},
        }
    if e2e and (variant in ENTRY or variant == "bf16_silu_mul"):
        hA = torch.from_numpy(A.view(np.int16) if A.dtype != np.float32 else A).pin_memory()
        hB = torch.from_numpy(B.view(np.int16) if B.dtype != np.float32 else B).pin_memory()
        hC = torch.empty_like(dC, device="cpu").pin_memory()
        hX = [torch.from_numpy(x.view(np.int16)).pin_memory() for x in extra]
        dX = [dWu] if extra else []

        def e2e_step():
            with torch.cuda.stream(stream):
                dA.copy_(hA, non_blocking=True)
                dB.copy_(hB, non_blocking=True)
                for h, d in zip(hX, dX):
                    d.copy_(h, non_blocking=True)
                step()
                hC.copy_(dC, non_blocking=True)

        n_e2e = max(3, min(steps, 20))
        h2d_bytes = int(hA.numel() * hA.element_size() + hB.numel() * hB.element_size()
                        + sum(h.numel() * h.element_size() for h in hX))
        d2h_bytes = int(hC.numel() * hC.element_size())
        # serial: every step copies its inputs in, computes and copies its result
        # out on one stream, nothing overlapped
        ms_serial = time_device(e2e_step, n_e2e, 2, stream)
        serial = {"value": flops * n_e2e / (ms_serial / 1e3) / 1e12, "unit": "TFLOP/s",
                  "h2d_bytes_per_step": h2d_bytes, "d2h_bytes_per_step": d2h_bytes,
                  "ms_per_step": ms_serial / n_e2e, "steps": n_e2e}
        # pipelined: the same copies and calls, with two device buffer sets and
        # three streams, so that the host->device copy of step i+1 and the
        # device->host copy of step i-1 run while step i computes
        res["e2e"] = dict(e2e_pipelined(fn, [hA, hB] + hX, [dA, dB] + dX, dC, hC, M, N, K, stream, n_e2e,
                                        flops), h2d_bytes_per_step=h2d_bytes, d2h_bytes_per_step=d2h_bytes)
        res["e2e_serial"] = serial

    if cpu_budget > 0:
        fps, nrows, dt, threads, sel, ref = cpu_sample(variant, A, B, M, N, K, cpu_budget, extra)
        res["cpu_baseline"] = {"value": fps / 1e12, "unit": "TFLOP/s", "cores": threads, "kind": "oracle",
                               "sample": f"{nrows} of {M} output rows spread over M ({nrows}x{N}x{K} FMAs, "
                                         f"FP64 oracle) in {dt:.1f} s"}
        if ref is not None:
            # the same rows of the timed output buffer, against the oracle
            try:
                res["cpu_baseline"]["parity"] = sample_parity(variant, dC.cpu().numpy(), M, N, K, sel, ref)
            except Exception as exc:  # the line is still printed; the failure is named in it
                res["cpu_baseline"]["parity"] = {"error": f"{type(exc).__name__}: {exc}"[:200]}
    del dA, dB, dC, keep
    torch.cuda.empty_cache()
    return res


def add_k4096_controls(paths):
    """Beside each K = 4100 workload measured with its K = 4096 control (same M,
    N and path), the control's time and throughput and the slowdown of the odd K:
    throughput at K = 4096 over throughput at K = 4100 (> 1: the tail costs more
    than its extra 0.1 % of FLOPs)."""
    by_name = {p["workload"]: p for p in paths}
    for p in paths:
        name = p["workload"]
        if not name.endswith("x4100"):
            continue
        ctrl = by_name.get(name[:-len("4100")] + "4096")
        if ctrl is None:
            continue
        p["k4096_control"] = {"workload": ctrl["workload"], "ms_per_step": ctrl["ms_per_step"],
                              "tflops": ctrl["tflops"], "kernel": ctrl["kernel"],
                              "slowdown_vs_k4096": ctrl["tflops"] / p["tflops"]}


def compact_paths(paths):
    """One short record per path: kernel, microseconds per call, TFLOP/s, the
    roofline fraction and its bound, DRAM traffic over the algorithmic bytes
    (when captured), cuBLAS's TFLOP/s on the same inputs, and the K = 4096
    control's slowdown for the K = 4100 rows."""
    out = {}
    for p in paths:
        rf = p.get("roofline") or {}
        rec = {"kernel": p["kernel"], "us": round(1e3 * p["ms_per_step"], 2), "tflops": round(p["tflops"], 2),
               "frac": round(rf.get("frac", 0.0), 3), "bound": rf.get("bound")}
        if rf.get("traffic") and rf.get("algorithmic_bytes"):
            rec["traffic_x"] = round(rf["traffic"] / rf["algorithmic_bytes"], 2)
        cb = p.get("cublas") or {}
        if cb.get("tflops"):
            rec["cublas_tflops"] = round(cb["tflops"], 2)
        if "k4096_control" in p:
            rec["slowdown_vs_k4096"] = round(p["k4096_control"]["slowdown_vs_k4096"], 3)
        out[p["workload"]] = rec
    return out


def cpu_one_thread(names, budget_s: float):
    """The oracle on one host thread for the small configurations: the whole
    problem when it holds at most ONE_THREAD_FULL_FMAS multiply-adds, else rows
    spread over M for about budget_s seconds.  TFLOP/s on the 2*M*N*K convention."""
    import oracle
    threads = oracle.num_threads()
    out = {}
    oracle.set_num_threads(1)
    try:
        for name in names:
            cfg, (variant, M, N, K, da, sa, db, sb) = all_workloads()[name]
            A, B, extra = host_inputs(variant, cfg, M, N, K, da, sa, db, sb)
            if M * N * K <= ONE_THREAD_FULL_FMAS:
                sel = np.arange(M, dtype=np.int64)
            else:
                t0 = time.perf_counter()
                oracle_rows(variant, A, B, M, N, K, np.zeros(1, dtype=np.int64), extra)
                per_row = max(time.perf_counter() - t0, 1e-6)
                sel = sample_rows(M, max(1, int(budget_s / per_row)))
            t0 = time.perf_counter()
            fl, _ = oracle_rows(variant, A, B, M, N, K, sel, extra)
            dt = time.perf_counter() - t0
            out[name] = {"tflops": fl / dt / 1e12, "seconds": dt, "cores": 1,
                         "sample": "whole problem" if sel.size == M else f"{sel.size} of {M} rows"}
    finally:
        oracle.set_num_threads(threads)
    return out


def bench_line(res, workload, steps, warmup, world, ms_total, e2e_ms, paths):
    """The JSON line of our arm from rank 0's measurement `res`, the slowest
    rank's timed-region length `ms_total` and per-step end-to-end times `e2e_ms`
    (slowest rank, keyed "e2e" / "e2e_serial"): whole-job figures over `world`
    replicas."""
    M, N, K = res["M"], res["N"], res["K"]
    value = replica_throughput(res["flops_per_step"], steps, world, ms_total)
    clk = res["clocks"] or {}
    line = {
        "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": world, "steps": steps,
        "warmup": warmup, "ms_per_step": ms_total / steps, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None,
        "dtype": "f32" if res["variant"].startswith("f32") else res["variant"].split("_")[0],
        "data": "synthetic",
        "config": {"workload": workload, "M": M, "N": N, "K": K,
                   "layout": "column-major" if res["variant"].endswith("_cm") else "row-major",
                   "inputs": "uniform[-1,1] seeded SplitMix64" if "ffn" not in workload
                   else "X~N(0,1), W~N(0,1/4096) seeded SplitMix64",
                   "l2": res["l2"],
                   "parallelism": f"replicas x{world}"},
        "kernel": res["kernel"],
        "roofline": res["roofline"],
        # counted by the library over rank 0's timed steps; every replica runs the same calls
        "gpu_launches": res["gpu_launches"] * world,
        "clocks": {"sm_mhz": clk.get("sm_mhz"), "sm_max_mhz": clk.get("sm_max_mhz"),
                   "reasons": clk.get("reasons", []), "samples": clk.get("samples", 0)},
    }
    for key in ("e2e", "e2e_serial"):
        if key in res:
            e = dict(res[key])
            ms = e2e_ms.get(key, e["ms_per_step"])
            e["value"] = replica_throughput(res["flops_per_step"], 1, world, ms)
            e["ms_per_step"] = ms
            line[key] = e
    if "per_call" in res:
        line["per_call"] = res["per_call"]
    if "cpu_baseline" in res:
        line["cpu_baseline"] = res["cpu_baseline"]
    if res.get("cublas"):
        line["cublas"] = res["cublas"]
    if paths:
        # the full records first, then a compact summary as the line's last key
        line["paths_detail"] = paths
        line["paths"] = compact_paths(paths)
    return line


def run_ours(args):
    import torch
    import torch.distributed as dist
    import dense_matrix_multiply_gb300 as g

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    torch.cuda.set_device(local)
    if world == 1:
        g.ensure_built()
    g.load()
    peaks, peaks_src = read_peaks()
    props = torch.cuda.get_device_properties(local)
    sms = props.multi_processor_count
    prop_mhz = getattr(props, "clock_rate", 0) / 1000.0 or None  # kHz -> MHz
    uuid = None
    try:
        uuid = "GPU-" + str(torch.cuda.get_device_properties(local).uuid)
    except Exception:
        uuid = None
    stream = torch.cuda.Stream()

    # CPU baseline first (before heavy GPU use), rank 0 at N=1 only.
    res = measure_workload(args.workload, args.steps, args.warmup, peaks, peaks_src, sms, stream,
                           sampler_uuid=uuid, e2e=not args.no_e2e,
                           cpu_budget=(args.cpu_seconds if (rank == 0 and world == 1
                                                            and not args.no_cpu_baseline) else 0.0),
                           clocks=(rank == 0), prop_mhz=prop_mhz)
    ms_total = res["ms_total"]
    ms_total = slowest_rank_ms(ms_total, world, device="cuda")

    # end to end, whole job: every rank's replica through its slowest rank's time
    e2e_ms = {}
    for key in ("e2e", "e2e_serial"):
        if key in res:
            e2e_ms[key] = slowest_rank_ms(res[key]["ms_per_step"], world, device="cuda")

    paths = []
    if not args.no_paths and rank == 0:
        for wl in args.paths:
            if wl == args.workload:
                continue
            r = measure_workload(wl, max(5, args.path_steps), 3, peaks, peaks_src, sms, stream,
                                 sampler_uuid=uuid, e2e=False, cpu_budget=0.0, clocks=True, prop_mhz=prop_mhz)
            paths.append({k: r[k] for k in ("workload", "kernel", "M", "N", "K", "ms_per_step", "tflops",
                                            "roofline", "clocks", "kernels", "cublas", "l2", "gpu_launches",
                                            "per_call")
                          if k in r})
        add_k4096_controls(paths)

    one_thread = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        one_thread = cpu_one_thread(ONE_THREAD_WORKLOADS, args.one_thread_seconds)

    if rank == 0:
        line = bench_line(res, args.workload, args.steps, args.warmup, world, ms_total, e2e_ms, paths)
        if one_thread:
            line["cpu_baseline"]["one_thread"] = one_thread
        print(json.dumps(line), flush=True)
    if world > 1:
        dist.barrier()
        dist.destroy_process_group()


# ------------------------------------------------------------------ reference arm
def run_reference(args):
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    import oracle
    cfg, (variant, M, N, K, da, sa, db, sb) = all_workloads()[args.workload]
    A, B, extra = host_inputs(variant, cfg, M, N, K, da, sa, db, sb)
    threads = oracle.num_threads()
    # size each step so that warmup + steps take about args.ref_seconds in total
    rows = np.arange(min(threads, M), dtype=np.int64)
    t0 = time.perf_counter()
    oracle_rows(variant, A, B, M, N, K, rows, extra)
    per_round = max(time.perf_counter() - t0, 1e-6)
    per_step = args.ref_seconds / max(1, args.steps + args.warmup)
    nrows = int(min(M, max(1, round(per_step / per_round)) * rows.size))
    sel = np.arange(nrows, dtype=np.int64) % M
    for _ in range(args.warmup):
        oracle_rows(variant, A, B, M, N, K, sel, extra)
    t0 = time.perf_counter()
    flops = 0.0
    for _ in range(args.steps):
        flops += oracle_rows(variant, A, B, M, N, K, sel, extra)[0]
    dt = time.perf_counter() - t0
    value = flops / dt / 1e12
    sample = f"{nrows} of {M} output rows per step ({nrows}x{N}x{K} FMAs, FP64 oracle)"
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": dt * 1e3 / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic",
        "config": {"workload": args.workload, "M": M, "N": N, "K": K,
                   "layout": "column-major" if variant.endswith("_cm") else "row-major",
                   "parallelism": "host cores (CPU oracle)"},
        "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": threads, "kind": "oracle", "sample": sample},
        "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def main(argv=None):
    p = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=200)
    p.add_argument("--warmup", type=int, default=10)
    p.add_argument("--impl", choices=["ours", "reference"], default="ours")
    p.add_argument("--workload", default=DEFAULT_WORKLOAD, choices=sorted(all_workloads()))
    p.add_argument("--paths", nargs="*", default=DEFAULT_PATHS)
    p.add_argument("--path-steps", type=int, default=50)
    p.add_argument("--no-paths", action="store_true")
    p.add_argument("--no-cpu-baseline", action="store_true")
    p.add_argument("--no-e2e", action="store_true")
    p.add_argument("--cpu-seconds", type=float, default=12.0)
    p.add_argument("--ref-seconds", type=float, default=60.0)
    p.add_argument("--one-thread-seconds", type=float, default=2.0)
    args = p.parse_args(argv)
    if args.impl == "ours":
        args.warmup = max(3, args.warmup)  # timing rule: at least 3 untimed warm-up steps
    if args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
