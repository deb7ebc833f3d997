"""Benchmark of the block-scaled fused dequantizing matmul on GB300.

Headline workload (one "step"): a decode pass over a stack of L distinct
mxfp4 weight matrices, N = K = 4096 (E2M1 codes + E8M0 scale per 32-block,
W ~ N(0, 0.02), seed 0), one qmm per layer with M = 1 bf16 activation row
(X ~ N(0, 1)).  The L copies together exceed 3x the 129 MB L2, so every
layer's weights come from HBM; the L launches of a step are captured in one
CUDA graph.  value = algorithmic bytes (codes + scales + X + out, each once)
per second, whole job.

Also reported (``breakdown``): the other workloads of the method at their
stated shapes -- the nvfp4 batch GEMV (M = 1, 8; N = 14336), the mxfp8 E4M3
prefill GEMM (M = 2048, N = K = 4096) and the int4-affine / mxfp8 E5M2 /
nvfp8 sweep (M = 1, 16, 128, 4096; N = 11008, K = 4096), mxint8, int8 and
int4 at M = 1 and 4096 and the fp16-scale int8 / int4 twins at M = 1 on the
same N, K, the two-level residual mxfp4x2 and mxint4 at M = 1 and 2048
(N = K = 4096), the legacy float fp4 (M = 1), fp8 E5M2 (M = 1, N = 11008) and
fp8 E4M3 (M = 2048) -- GEMV rows in GB/s,
GEMM rows in TFLOP/s, each against its roofline.

``--impl reference`` times the CPU oracle (numpy decode -> float64 W ->
float64 matmul) on a bounded sample of the same workload.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "qGEMV HBM GB/s (M=1) & qGEMM TFLOP/s (M≥128), % of GB300 roofline"
L2_BYTES = 129 * 2 ** 20
HEADLINE = ("mxfp4", 1, 4096, 4096)


def parse():
    p = argparse.ArgumentParser()
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=20)
    p.add_argument("--warmup", type=int, default=5)
    p.add_argument("--impl", default="ours", choices=["ours", "reference"])
    p.add_argument("--no-breakdown", action="store_true")
    p.add_argument("--only", default=None, help="run one breakdown row: fmt:M:N:K[:A|:A8|:A4], gather:fmt:M:N:K:E, batched:fmt:M:N1,N2:K, "
                   "rmsnorm:fmt:M:N:K, gated_rmsnorm:fmt:M:N:K or dequant:fmt:N:K:f32|bf16")
    return p.parse_args()


def sizes(fmt, m, n, k):
    """Algorithmic bytes of one qmm: codes + scales + global + X (bf16) + out (bf16)."""
    import block_scaled_quantized_spec_gb300 as q
    b = q.qfmt_codes_bytes(fmt, n, k) + q.qfmt_scales_bytes(fmt, n, k) + 2 * m * k + 2 * m * n
    if fmt == "nvfp4":
        b += 4
    return b


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        d = json.load(open(path))
        return d["hbm_gbs"], d["bf16_tflops"], d.get("bf16_tflops_sustained", d["bf16_tflops"]), "measured"
    return 6800.0, 1900.0, 1700.0, "fallback"


class Clocks:
    """Samples nvidia-smi during the timed region."""

    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        self.index = index
        self.proc = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.Q}", "--format=csv,noheader,nounits",
                 "-lms", "100"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except (OSError, FileNotFoundError):
            self.proc = None
        return self

    def __exit__(self, *a):
        self.lines = []
        if self.proc is not None:
            self.proc.terminate()
            try:
                out, _ = self.proc.communicate(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
                out, _ = self.proc.communicate()
            self.lines = [ln for ln in out.splitlines() if ln.strip()]

    def summary(self):
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in getattr(self, "lines", []):
            f = [x.strip() for x in ln.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                mx = float(f[2])
            except ValueError:
                continue
            for nm, v in zip(names, f[5:9]):
                if v.lower() == "active":
                    reasons.add(nm)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": mx, "reasons": sorted(reasons),
                "samples": len(sm)}


def dist_init(args):
    import torch
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    else:
        torch.cuda.set_device(0)
    return rank, world, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(x, world):
    """Max of a per-rank float over all ranks (CUDA tensor under NCCL, CPU under gloo)."""
    if world == 1:
        return x
    import torch
    import torch.distributed as dist
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([x], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_throughput(per_rank_bytes, per_rank_ms, world):
    """Whole-job bytes/s: every rank's units over the slowest rank's time (weak scaling)."""
    total = per_rank_bytes * world
    slowest = max_over_ranks(per_rank_ms, world)
    return total / (slowest * 1e-3), slowest


class Problem:
    """L copies of one packed weight in HBM, their activations and outputs.

    path "auto": a workspace when the call can use one (the block-scaled
    tensor-core GEMM of the MX formats, M > 16), the call a user makes with
    one; "A": no workspace (the bf16-decode GEMM); "A8": both operands
    quantized (qmm_a8: the activations packed to MXFP8 E4M3, one
    block-scaled MMA per block); "A4": the all-FP4 product (qmm_a4: the
    activations packed to MXFP4, kind::mxf4).
    """

    def __init__(self, fmt, m, n, k, copies, seed=0, path="auto"):
        import numpy as np
        import torch
        import block_scaled_quantized_spec_gb300 as q
        from block_scaled_quantized_spec_gb300 import synth
        self.fmt, self.m, self.n, self.k = fmt, m, n, k
        rng = np.random.default_rng(seed)
        w = synth.weights(n, k, rng=rng, outliers=(fmt == "nvfp4"))
        xb = synth.activations_bf16(m, k, rng=rng)
        c, s, g = q.qfmt_pack(fmt, w)
        del w
        self.g = g
        dc = torch.from_numpy(c).cuda()
        ds = torch.from_numpy(s).cuda()
        self.codes = [dc] + [dc.clone() for _ in range(copies - 1)]
        self.scales = [ds] + [ds.clone() for _ in range(copies - 1)]
        self.x_host = torch.from_numpy(xb.view(np.int16)).view(torch.bfloat16)
        x = self.x_host.cuda()
        self.x = [x] + [x.clone() for _ in range(copies - 1)]
        self.out = [torch.empty((m, n), dtype=torch.bfloat16, device="cuda") for _ in range(copies)]
        self.copies = copies
        self.bytes = sizes(fmt, m, n, k)
        self.flops = 2.0 * m * n * k
        self.a8 = path == "A8"
        self.a4 = path == "A4"
        if self.a8:
            wsb = q.qmm_a8_workspace_bytes(fmt, m, k)
        elif self.a4:
            wsb = q.qmm_a4_workspace_bytes(fmt, m, k)
        else:
            wsb = q.qmm_workspace_bytes(fmt, m, k) if path == "auto" else 0
        # one workspace serves every layer: each call's activation split waits
        # for the previous call to finish before it writes
        self.ws = torch.empty(wsb, dtype=torch.uint8, device="cuda") if wsb else None
        self.path = ("A8" if self.a8 else "A4" if self.a4 else
                     ("SUB" if fmt in q.SUB_BYTE else ("B" if wsb else ("A" if m > 16 else "GEMV"))))

    def step(self):
        import block_scaled_quantized_spec_gb300 as q
        for i in range(self.copies):
            if self.a8:
                q.qmm_a8(self.fmt, self.codes[i], self.scales[i], self.x[i], self.n, out=self.out[i], workspace=self.ws)
            elif self.a4:
                q.qmm_a4(self.fmt, self.codes[i], self.scales[i], self.g, self.x[i], self.n, out=self.out[i],
                         workspace=self.ws)
            elif self.ws is not None:
                q.qmm_ex(self.fmt, self.codes[i], self.scales[i], self.g, self.x[i], self.n, out=self.out[i],
                         workspace=self.ws)
            else:
                q.qmm(self.fmt, self.codes[i], self.scales[i], self.g, self.x[i], self.n, out=self.out[i])

    def graph(self):
        import torch
        s = torch.cuda.Stream()
        s.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(s):
            self.step()                                   # warm the library's per-device cache
        torch.cuda.current_stream().wait_stream(s)
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            self.step()
        return g


def time_graph(graph, steps, warmup, world, clocks_index=None):
    import torch
    for _ in range(warmup):
        graph.replay()
    torch.cuda.synchronize()
    barrier(world)
    st = torch.cuda.current_stream()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    clk = Clocks(clocks_index) if clocks_index is not None else None
    if clk:
        clk.__enter__()
        time.sleep(0.3)
    torch.cuda.synchronize()
    e0.record(st)
    for _ in range(steps):
        graph.replay()
    e1.record(st)
    torch.cuda.synchronize()
    if clk:
        clk.__exit__(None, None, None)
    barrier(world)
    ms = e0.elapsed_time(e1) / steps
    return max_over_ranks(ms, world), (clk.summary() if clk else None)


def step_spread(graph, steps):
    """Per-step device times of a second pass (events around each replay): p10 / p50 / p90 in ms."""
    import statistics
    import torch
    st = torch.cuda.current_stream()
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(steps + 1)]
    torch.cuda.synchronize()
    ev[0].record(st)
    for i in range(steps):
        graph.replay()
        ev[i + 1].record(st)
    torch.cuda.synchronize()
    t = sorted(ev[i].elapsed_time(ev[i + 1]) for i in range(steps))
    q = statistics.quantiles(t, n=10, method="inclusive") if len(t) > 1 else [t[0]] * 9
    return {"p10": round(q[0], 4), "p50": round(statistics.median(t), 4), "p90": round(q[8], 4), "steps": steps}


def copies_for(nbytes, m):
    if m >= 128:
        return 2
    return max(4, min(64, -(-3 * L2_BYTES // nbytes)))


def measure_e2e(prob, steps, warmup):
    """Same metric through the public call with host buffers: per step, one H2D copy
    of every layer's activations from pinned memory, the qmm launches, and one D2H
    copy of every layer's output (weights stay resident, as in a decode step)."""
    import torch
    import block_scaled_quantized_spec_gb300 as q
    L, m, n, k = prob.copies, prob.m, prob.n, prob.k
    xh = prob.x_host.repeat(L, 1).pin_memory()                       # [L*M, K] bf16, pinned
    oh = torch.empty((L * m, n), dtype=torch.bfloat16).pin_memory()
    xd = torch.empty((L * m, k), dtype=torch.bfloat16, device="cuda")
    od = torch.empty((L * m, n), dtype=torch.bfloat16, device="cuda")

    def one():
        xd.copy_(xh, non_blocking=True)
        for i in range(L):
            q.qmm(prob.fmt, prob.codes[i], prob.scales[i], prob.g, xd[i * m:(i + 1) * m], n,
                  out=od[i * m:(i + 1) * m])
        oh.copy_(od, non_blocking=True)
    one()                                                             # warm the library's caches
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()                                    # the step's copies and launches
    with torch.cuda.graph(graph):
        one()
    for _ in range(warmup):
        graph.replay()
    torch.cuda.synchronize()
    st = torch.cuda.current_stream()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(st)
    for _ in range(steps):
        graph.replay()
    e1.record(st)
    torch.cuda.synchronize()
    ms = e0.elapsed_time(e1) / steps
    return ms, xh.numel() * 2, oh.numel() * 2


class OracleSample:
    """The CPU oracle as it stands, on whole calls of the workload (inputs prepared once)."""

    def __init__(self, fmt, m, n, k):
        import numpy as np
        from block_scaled_quantized_spec_gb300 import synth
        from oracle import pack as opack
        rng = np.random.default_rng(0)
        w = synth.weights(n, k, rng=rng, outliers=(fmt == "nvfp4"))
        self.xb = synth.activations_bf16(m, k, rng=rng)
        self.c, self.s, self.g = opack.pack(fmt, w)
        self.fmt, self.m, self.n, self.k = fmt, m, n, k
        self.nbytes = opack.codes_nbytes(fmt, n, k) + opack.scales_nbytes(fmt, n, k) + 2 * m * k + 2 * m * n

    def run(self, budget_s, min_calls=1):
        from oracle import reference as oref
        times = []
        t_end = time.perf_counter() + budget_s
        while time.perf_counter() < t_end or len(times) < min_calls:
            t0 = time.perf_counter()
            oref.qmm_ref(self.fmt, self.c, self.s, self.g, self.xb, "bf16", self.m, self.n, self.k)
            times.append(time.perf_counter() - t0)
        return times

    def summary(self, times):
        t = statistics.median(times)
        return {"value": self.nbytes / t / 1e9, "unit": "GB/s", "cores": _blas_threads(), "kind": "oracle",
                "host_cpus": os.cpu_count(), "cpu_model": _cpu_model(),
                "sample": f"{len(times)} whole oracle calls {self.fmt} M={self.m} N={self.n} K={self.k} "
                          f"(median {t * 1e3:.1f} ms each; numpy decode single-threaded, float64 matmul on "
                          f"the BLAS threads)"}


def cpu_baseline(fmt, m, n, k, budget_s=12.0):
    o = OracleSample(fmt, m, n, k)
    return o.summary(o.run(budget_s, min_calls=2))


def _cpu_model():
    """The host CPU's model string (x86 'model name'; on Arm the implementer/part codes)."""
    import platform
    try:
        info = open("/proc/cpuinfo").read().splitlines()
        for key in ("model name", "Model"):
            for line in info:
                if line.split(":")[0].strip() == key:
                    return line.split(":", 1)[1].strip()
        imp = [ln.split(":", 1)[1].strip() for ln in info if ln.startswith("CPU implementer")]
        part = [ln.split(":", 1)[1].strip() for ln in info if ln.startswith("CPU part")]
        if imp and part:
            return f"{platform.machine()} implementer {imp[0]} part {part[0]}"
    except OSError:
        pass
    return platform.machine()


def _blas_threads():
    try:
        from threadpoolctl import threadpool_info
        n = [i.get("num_threads", 1) for i in threadpool_info() if i.get("user_api") == "blas"]
        return max(n) if n else 1
    except Exception:
        return int(os.environ.get("OMP_NUM_THREADS", os.cpu_count() or 1))


def run_reference(args):
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    fmt, m, n, k = HEADLINE
    o = OracleSample(fmt, m, n, k)
    o.run(0.0, min_calls=max(1, args.warmup))
    per_step, all_times = [], []
    t0 = time.perf_counter()
    for _ in range(args.steps):
        ts = o.run(0.0, min_calls=3)        # one step: 3 whole oracle calls
        all_times += ts
        per_step.append(o.nbytes * len(ts) / sum(ts) / 1e9)
    wall = time.perf_counter() - t0
    v = statistics.median(per_step)
    cb = o.summary(all_times)
    line = {"impl": "reference", "metric": METRIC, "value": v, "unit": "GB/s", "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": wall * 1e3 / args.steps,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic",
            "config": {"workload": "mxfp4 decode qGEMV M=1 N=4096 K=4096 (CPU oracle; a step = 3 whole calls)"},
            "cpu_baseline": {"kind": "oracle", "cores": cb["cores"], "sample": cb["sample"], "value": v,
                             "unit": "GB/s", "host_cpus": cb["host_cpus"], "cpu_model": cb["cpu_model"]},
            "e2e": {"value": v, "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


# DRAM bytes (read + write) of one headline launch from an ncu capture, valid
# only for the kernel source it was taken on (checked by hash; a changed
# kernel reports null until it is captured again).
TRAFFIC = {
    "kernel_source": "block_scaled_quantized_spec_gb300/csrc/qgemv_m2.cuh",
    "sha256_16": "1c718fb308e9a9d9",
    "bytes": 8937472,
    "profile": "profiles/qgemv_m2_mxfp4_M1_N4096_K4096.md",
}


def measured_traffic():
    import hashlib
    path = os.path.join(ROOT, TRAFFIC["kernel_source"])
    try:
        h = hashlib.sha256(open(path, "rb").read()).hexdigest()[:16]
    except OSError:
        return None
    return TRAFFIC["bytes"] if h == TRAFFIC["sha256_16"] else None


def roofline_gemv(prob, ms_step, hbm, kind):
    per_launch_ms = ms_step / prob.copies
    achieved = prob.bytes / (per_launch_ms * 1e-3) / 1e9
    return {"bound": "hbm", "achieved": round(achieved, 1), "peak": hbm, "unit": "GB/s",
            "frac": round(achieved / hbm, 4), "traffic": measured_traffic(),
            "traffic_source": TRAFFIC["profile"], "peak_kind": f"{kind} (STREAM copy, burst)",
            "kernel": f"qgemv_m2_kernel<{prob.fmt}, 1 row, 16 warps, staged weights>",
            "per_launch_us": round(per_launch_ms * 1e3, 3),
            "algorithmic_bytes_per_launch": prob.bytes}


BREAKDOWN = [
    ("nvfp4", 1, 14336, 4096), ("nvfp4", 8, 14336, 4096),
    ("mxfp8_e4m3", 2048, 4096, 4096),
    ("int4_affine", 1, 11008, 4096), ("int4_affine", 16, 11008, 4096),
    ("int4_affine", 128, 11008, 4096), ("int4_affine", 4096, 11008, 4096),
    ("mxfp8_e5m2", 1, 11008, 4096), ("mxfp8_e5m2", 16, 11008, 4096),
    ("mxfp8_e5m2", 128, 11008, 4096), ("mxfp8_e5m2", 4096, 11008, 4096),
    ("nvfp8", 1, 11008, 4096), ("nvfp8", 16, 11008, 4096),
    ("nvfp8", 128, 11008, 4096), ("nvfp8", 4096, 11008, 4096),
    ("mxint8", 1, 11008, 4096), ("mxint8", 4096, 11008, 4096),
    ("int8", 1, 11008, 4096), ("int8", 4096, 11008, 4096),
    ("int4", 1, 11008, 4096), ("int4", 4096, 11008, 4096),
    ("int8_f16", 1, 11008, 4096), ("int4_f16", 1, 11008, 4096),
    ("mxfp4x2", 1, 4096, 4096), ("mxfp4x2", 2048, 4096, 4096),
    ("mxint4", 1, 4096, 4096), ("mxint4", 2048, 4096, 4096),
    ("fp4", 1, 4096, 4096), ("fp8_e5m2", 1, 11008, 4096), ("fp8_e4m3", 2048, 4096, 4096),
    # the MX formats' GEMM rows again without a workspace (the bf16-decode GEMM), and mxfp4's prefill GEMM
    ("mxfp8_e4m3", 2048, 4096, 4096, "A"), ("mxfp8_e5m2", 128, 11008, 4096, "A"),
    ("mxfp8_e5m2", 4096, 11008, 4096, "A"),
    ("mxfp4", 2048, 4096, 4096), ("mxfp4", 2048, 4096, 4096, "A"),
    # both operands quantized (W . A8)
    ("mxfp8_e4m3", 2048, 4096, 4096, "A8"), ("mxfp4", 2048, 4096, 4096, "A8"),
    ("mxfp8_e5m2", 4096, 11008, 4096, "A8"),
    # the all-FP4 product (W . A4)
    ("mxfp4", 2048, 4096, 4096, "A4"), ("mxfp4", 4096, 11008, 4096, "A4"), ("nvfp4", 2048, 4096, 4096, "A4"),
    # the 2/3/5/6-bit bit streams
    ("int3", 1, 11008, 4096), ("mxint5", 16, 4096, 4096),
    # batch decode rows on [4096, 4096] (one decode per weight block for every activation row)
    ("mxfp4", 8, 4096, 4096), ("mxfp8_e4m3", 8, 4096, 4096), ("int8", 8, 4096, 4096),
]

# The standalone dequant kernel: [4096, 4096] weights to float32 and bf16.
DEQUANT = [("mxfp4", 4096, 4096, "f32"), ("mxfp4", 4096, 4096, "bf16"), ("nvfp4", 14336, 4096, "f32"),
           ("mxfp8_e4m3", 4096, 4096, "f32")]

# The five workloads of the method, each timed once through the CPU oracle
# (a bounded sample: whole calls within a small budget, at least one).
ORACLE_CONFIGS = [("mxfp4", 8, 16, 512, "f32"), ("mxfp4", 1, 4096, 4096, "bf16"),
                  ("nvfp4", 1, 14336, 4096, "bf16"), ("nvfp4", 8, 14336, 4096, "bf16"),
                  ("mxfp8_e4m3", 2048, 4096, 4096, "bf16")] + \
                 [(f, mm, 11008, 4096, "bf16") for f in ("int4_affine", "mxfp8_e5m2", "nvfp8") for mm in (1, 16, 128, 4096)]


# Expert-routed rows (MoE gather-qmm): one token's top-8 routing over 8 experts
# of [4096, 4096] mxfp4 weights, each row to a different expert; and prefill
# batches of 64 and 512 rows routed uniformly over the 8 experts, grouped by
# expert on the tensor cores (qmm_grouped).
GATHER = [("mxfp4", 8, 4096, 4096, 8)]
GROUPED = [("mxfp4", 64, 4096, 4096, 8), ("mxfp4", 512, 4096, 4096, 8)]


class GatherProblem:
    """L copies of one stacked [E * N, K] expert weight, the routed rows and their outputs."""

    def __init__(self, fmt, m, n, k, e, copies, seed=0):
        import numpy as np
        import torch
        import block_scaled_quantized_spec_gb300 as q
        from block_scaled_quantized_spec_gb300 import synth
        self.fmt, self.m, self.n, self.k, self.e = fmt, m, n, k, e
        rng = np.random.default_rng(seed)
        c, s, g = q.qfmt_pack(fmt, synth.weights(e * n, k, rng=rng))
        self.g = g
        dc, ds = torch.from_numpy(c).cuda(), torch.from_numpy(s).cuda()
        self.codes = [dc] + [dc.clone() for _ in range(copies - 1)]
        self.scales = [ds] + [ds.clone() for _ in range(copies - 1)]
        xb = synth.activations_bf16(m, k, rng=rng)
        self.x = torch.from_numpy(xb.view(np.int16)).view(torch.bfloat16).cuda()
        if m <= e:   # one token's routing: m distinct experts
            self.idx = [torch.from_numpy(rng.permutation(e)[:m].astype(np.int32)).cuda() for _ in range(copies)]
        else:        # a prefill batch routed uniformly
            self.idx = [torch.from_numpy(rng.integers(0, e, m).astype(np.int32)).cuda() for _ in range(copies)]
        self.out = [torch.empty((m, n), dtype=torch.bfloat16, device="cuda") for _ in range(copies)]
        self.copies = copies
        experts = len(set(int(v) for v in self.idx[0].cpu()))
        self.bytes = experts * (sizes(fmt, 0, n, k) - (4 if fmt == "nvfp4" else 0)) + 2 * m * k + 2 * m * n + \
            4 * m + (4 if fmt == "nvfp4" else 0)

    grouped = False

    def step(self):
        import block_scaled_quantized_spec_gb300 as q
        for i in range(self.copies):
            if self.grouped:
                q.qmm_grouped(self.fmt, self.codes[i], self.scales[i], self.x, self.idx[i], self.n, self.e,
                              out=self.out[i], workspace=self.ws)
            else:
                q.qmm_gather(self.fmt, self.codes[i], self.scales[i], self.g, self.x, self.idx[i], self.n, self.e,
                             out=self.out[i])

    graph = Problem.graph


# Fused decode forms: the Q/K/V projections of a grouped-query layer in one
# launch, and RMSNorm in front of one mxfp4 [4096, 4096] GEMV.
FUSED = [("batched", "mxfp4", 1, (4096, 1024, 1024), 4096), ("rmsnorm", "mxfp4", 1, (4096,), 4096),
         ("gated_rmsnorm", "mxfp4", 1, (4096,), 4096)]


class FusedProblem:
    """L copies of the weights of one fused call (1..4 matrices), their activations and outputs."""

    def __init__(self, kind, fmt, m, ns, k, copies, seed=0):
        import numpy as np
        import torch
        import block_scaled_quantized_spec_gb300 as q
        from block_scaled_quantized_spec_gb300 import synth
        self.kind, self.fmt, self.m, self.ns, self.k = kind, fmt, m, tuple(ns), k
        rng = np.random.default_rng(seed)
        packed = [q.qfmt_pack(fmt, synth.weights(n, k, rng=rng)) for n in ns]
        self.g = [p[2] for p in packed]
        base = [(torch.from_numpy(p[0]).cuda(), torch.from_numpy(p[1]).cuda()) for p in packed]
        self.w = [base] + [[(c.clone(), s.clone()) for (c, s) in base] for _ in range(copies - 1)]
        xb = synth.activations_bf16(m, k, rng=rng)
        self.x = torch.from_numpy(xb.view(np.int16)).view(torch.bfloat16).cuda()
        self.gamma = (1.0 + 0.1 * torch.randn(k, generator=torch.Generator().manual_seed(seed))).to(torch.bfloat16).cuda()
        zb = synth.activations_bf16(m, k, rng=rng)                        # the gate (gated_rmsnorm)
        self.gate = torch.from_numpy(zb.view(np.int16)).view(torch.bfloat16).cuda()
        self.outs = [[torch.empty((m, n), dtype=torch.bfloat16, device="cuda") for n in ns] for _ in range(copies)]
        self.copies = copies
        self.bytes = (sum(sizes(fmt, m, n, k) - 2 * m * k for n in ns) + 2 * m * k
                      + (2 * k if kind in ("rmsnorm", "gated_rmsnorm") else 0) + (2 * m * k if kind == "gated_rmsnorm" else 0))

    def step(self, separate=False):
        import block_scaled_quantized_spec_gb300 as q
        for i in range(self.copies):
            w, o = self.w[i], self.outs[i]
            if self.kind == "rmsnorm":
                q.qmm_rmsnorm(self.fmt, w[0][0], w[0][1], self.g[0], self.x, self.gamma, 1e-5, self.ns[0], out=o[0])
            elif self.kind == "gated_rmsnorm":
                q.qmm_gated_rmsnorm(self.fmt, w[0][0], w[0][1], self.g[0], self.x, self.gate, self.gamma, 1e-5,
                                    self.ns[0], out=o[0])
            elif separate:
                for j, n in enumerate(self.ns):
                    q.qmm(self.fmt, w[j][0], w[j][1], self.g[j], self.x, n, out=o[j])
            else:
                q.qmm_batched(self.fmt, [c for c, _ in w], [s for _, s in w], self.g, self.x, list(self.ns), outs=o)

    graph = Problem.graph


def fused_row(kind, fmt, m, ns, k, hbm, steps=10, warmup=3):
    import torch
    per_call = sum(sizes(fmt, m, n, k) for n in ns)
    prob = FusedProblem(kind, fmt, m, ns, k, max(4, min(64, -(-3 * L2_BYTES // per_call))))
    g = prob.graph()
    ms, _ = time_graph(g, steps, warmup, 1)
    per = ms / prob.copies
    gbs = prob.bytes / (per * 1e-3) / 1e9
    row = {"op": f"qmm_{kind}", "fmt": fmt, "M": m, "N": list(ns), "K": k, "us": round(per * 1e3, 2),
           "copies": prob.copies, "GB/s": round(gbs, 1), "hbm_frac": round(gbs / hbm, 4)}
    if kind == "batched":     # the same products as one qmm launch per matrix
        prob.step = lambda: FusedProblem.step(prob, separate=True)
        g2 = Problem.graph(prob)
        ms2, _ = time_graph(g2, steps, warmup, 1)
        row["us_separate_qmm"] = round(ms2 / prob.copies * 1e3, 2)
        del g2
    del prob, g
    torch.cuda.empty_cache()
    return row


def gather_row(fmt, m, n, k, e, hbm, steps=10, warmup=3, grouped=False):
    import torch
    import block_scaled_quantized_spec_gb300 as q
    per_call = sizes(fmt, 0, n, k) * min(m, e)
    prob = GatherProblem(fmt, m, n, k, e, max(2, -(-3 * L2_BYTES // per_call)))
    if grouped:
        prob.grouped = True
        prob.ws = torch.empty(q.qmm_grouped_workspace_bytes(fmt, m, k, e), dtype=torch.uint8, device="cuda")
    g = prob.graph()
    ms, _ = time_graph(g, steps, warmup, 1)
    per = ms / prob.copies
    gbs = prob.bytes / (per * 1e-3) / 1e9
    row = {"op": "qmm_grouped" if grouped else "qmm_gather", "fmt": fmt, "M": m, "N": n, "K": k, "E": e,
           "us": round(per * 1e3, 2),
           "copies": prob.copies, "GB/s": round(gbs, 1), "hbm_frac": round(gbs / hbm, 4),
           "bytes": prob.bytes}
    del prob, g
    torch.cuda.empty_cache()
    return row


class DequantProblem:
    """L copies of one packed weight and their dequantized outputs."""

    def __init__(self, fmt, n, k, out_dtype, copies, seed=0):
        import numpy as np
        import torch
        import block_scaled_quantized_spec_gb300 as q
        from block_scaled_quantized_spec_gb300 import synth
        self.fmt, self.n, self.k = fmt, n, k
        c, s, g = q.qfmt_pack(fmt, synth.weights(n, k, seed=seed, outliers=(fmt == "nvfp4")))
        self.g = g
        dc, ds = torch.from_numpy(c).cuda(), torch.from_numpy(s).cuda()
        self.codes = [dc] + [dc.clone() for _ in range(copies - 1)]
        self.scales = [ds] + [ds.clone() for _ in range(copies - 1)]
        dt = torch.float32 if out_dtype == "f32" else torch.bfloat16
        self.out = [torch.empty((n, k), dtype=dt, device="cuda") for _ in range(copies)]
        self.copies = copies
        self.bytes = q.qfmt_codes_bytes(fmt, n, k) + q.qfmt_scales_bytes(fmt, n, k) + n * k * (4 if dt == torch.float32 else 2)

    def step(self):
        import block_scaled_quantized_spec_gb300 as q
        for i in range(self.copies):
            q.qfmt_dequant(self.fmt, self.codes[i], self.scales[i], self.g, self.n, self.k, out=self.out[i])

    graph = Problem.graph


def dequant_row(fmt, n, k, out_dtype, hbm, steps=10, warmup=3):
    import torch
    import block_scaled_quantized_spec_gb300 as q
    per_call = q.qfmt_codes_bytes(fmt, n, k) + q.qfmt_scales_bytes(fmt, n, k) + n * k * (4 if out_dtype == "f32" else 2)
    copies = max(2, -(-3 * L2_BYTES // per_call))
    prob = DequantProblem(fmt, n, k, out_dtype, copies)
    g = prob.graph()
    ms, _ = time_graph(g, steps, warmup, 1)
    per = ms / copies
    gbs = prob.bytes / (per * 1e-3) / 1e9
    row = {"op": "qfmt_dequant", "fmt": fmt, "N": n, "K": k, "out": out_dtype, "us": round(per * 1e3, 2),
           "copies": copies, "GB/s": round(gbs, 1), "hbm_frac": round(gbs / hbm, 4), "bytes": prob.bytes}
    del prob, g
    torch.cuda.empty_cache()
    return row


def oracle_per_config(budget_s=1.0):
    """The CPU oracle timed on each workload of the method: median of whole calls within the budget."""
    rows = []
    for fmt, m, n, k, xd in ORACLE_CONFIGS:
        import numpy as np
        from block_scaled_quantized_spec_gb300 import synth
        from oracle import pack as opack
        from oracle import reference as oref
        rng = np.random.default_rng(0)
        c, s, g = opack.pack(fmt, synth.weights(n, k, rng=rng, outliers=(fmt == "nvfp4")))
        x = synth.activations_f32(m, k, rng=rng) if xd == "f32" else synth.activations_bf16(m, k, rng=rng)
        times = []
        t_end = time.perf_counter() + budget_s
        while not times or time.perf_counter() < t_end:
            t0 = time.perf_counter()
            oref.qmm_ref(fmt, c, s, g, x, xd, m, n, k)
            times.append(time.perf_counter() - t0)
        t = statistics.median(times)
        nbytes = opack.codes_nbytes(fmt, n, k) + opack.scales_nbytes(fmt, n, k) + (4 if xd == "f32" else 2) * (m * k + m * n)
        rows.append({"fmt": fmt, "M": m, "N": n, "K": k, "calls": len(times), "ms": round(t * 1e3, 2),
                     "GB/s": round(nbytes / t / 1e9, 4), "GFLOP/s": round(2.0 * m * n * k / t / 1e9, 2)})
    return {"kind": "oracle", "cores": _blas_threads(), "host_cpus": os.cpu_count(), "rows": rows,
            "note": "numpy decode (single-threaded) + float64 BLAS matmul; the result and its error bound per call"}


def breakdown_row(fmt, m, n, k, hbm, bf16, kind, steps=10, warmup=3, path="auto"):
    import torch
    nbytes = sizes(fmt, m, n, k)
    copies = copies_for(nbytes, m)
    prob = Problem(fmt, m, n, k, copies, path=path)
    g = prob.graph()
    ms, _ = time_graph(g, steps, warmup, 1)
    per = ms / copies
    prob_flops_per_byte = prob.flops / nbytes
    row = {"fmt": fmt, "M": m, "N": n, "K": k, "us": round(per * 1e3, 2), "copies": copies,
           "path": {"B": "block-scaled tcgen05 GEMM (X split + kind::mxf8f6f4)", "A": "bf16-decode tcgen05 GEMM",
                    "A8": "both operands quantized (X to MXFP8 E4M3, one kind::mxf8f6f4 MMA per block)",
                    "A4": "all-FP4 (X in W's FP4 family, kind::mxf4 / mxf4nvf4 per 64 K)",
                    "GEMV": "decode GEMV", "SUB": "CUDA-core sub-byte kernel"}[prob.path]}
    gbs = nbytes / (per * 1e-3) / 1e9
    tfl = prob.flops / (per * 1e-3) / 1e12
    row["GB/s"] = round(gbs, 1)
    row["TFLOP/s"] = round(tfl, 2)
    row["hbm_frac"] = round(gbs / hbm, 4)
    if m >= 128:
        # the format's own tensor rate (fp8 2x, fp4 6x bf16); int8 elements against bf16 (this part's int8 rate is lower)
        fp_peak = {"mxfp8_e4m3": 2 * bf16, "mxfp8_e5m2": 2 * bf16, "nvfp8": 2 * bf16, "nvfp8_f16": 2 * bf16,
                   "mxint8": bf16, "int8": bf16, "int8_f16": bf16, "int4": bf16, "int4_f16": bf16,
                   "mxfp4x2": bf16, "mxint4": bf16, "fp8_e4m3": 2 * bf16, "fp8_e5m2": 2 * bf16}.get(fmt, 6 * bf16)
        if prob.path == "A8":   # FP8 operands on both sides: the FP8 rate
            fp_peak = 2 * bf16
        if prob.path == "A4":   # FP4 operands on both sides: the FP4 rate
            fp_peak = 6 * bf16
        row["bf16_frac"] = round(tfl / bf16, 4)
        row["native_peak_frac"] = round(tfl / fp_peak, 4)
        # against the roofline at this arithmetic intensity: min(bf16 peak, FLOP/byte x HBM)
        ridge = min(bf16, prob_flops_per_byte * hbm / 1e3)
        row["roofline_frac"] = round(tfl / ridge, 4)
    del prob, g
    torch.cuda.empty_cache()
    return row


def main():
    args = parse()
    if args.impl == "reference":
        run_reference(args)
        return
    import torch
    from block_scaled_quantized_spec_gb300 import build
    build.build()
    import block_scaled_quantized_spec_gb300 as q
    q.load()
    rank, world, local = dist_init(args)
    hbm, bf16, bf16_sus, kind = peaks()

    fmt, m, n, k = HEADLINE
    nbytes = sizes(fmt, m, n, k)
    copies = copies_for(nbytes, m) if args.only is None else 4
    if args.only:
        parts = args.only.split(":")
        if parts[0] in ("gather", "grouped"):   # gather:fmt:M:N:K:E / grouped:fmt:M:N:K:E
            f, mm, nn, kk, ee = parts[1:]
            print(json.dumps(gather_row(f, int(mm), int(nn), int(kk), int(ee), hbm, args.steps, args.warmup,
                                        grouped=parts[0] == "grouped")))
            return
        if parts[0] in ("batched", "rmsnorm", "gated_rmsnorm"):   # batched:fmt:M:N1,N2,..:K  /  rmsnorm:fmt:M:N:K
            f, mm, nn, kk = parts[1:]
            ns = tuple(int(v) for v in nn.split(","))
            print(json.dumps(fused_row(parts[0], f, int(mm), ns, int(kk), hbm, args.steps, args.warmup)))
            return
        if parts[0] == "dequant":         # dequant:fmt:N:K:f32|bf16
            f, nn, kk, od = parts[1:]
            print(json.dumps(dequant_row(f, int(nn), int(kk), od, hbm, args.steps, args.warmup)))
            return
        f, mm, nn, kk = parts[:4]         # fmt:M:N:K[:A]
        print(json.dumps(breakdown_row(f, int(mm), int(nn), int(kk), hbm, bf16, kind, args.steps,
                                       args.warmup, path=parts[4] if len(parts) > 4 else "auto")))
        return
    prob = Problem(fmt, m, n, k, copies, seed=rank)
    graph = prob.graph()
    ms, clk = time_graph(graph, args.steps, args.warmup, world, clocks_index=local)
    spread = step_spread(graph, max(args.steps, 10))
    total_bytes = world * copies * nbytes
    value = total_bytes / (ms * 1e-3) / 1e9
    e2e_ms, h2d, d2h = measure_e2e(prob, max(3, args.steps // 2), 2)
    e2e_ms = max_over_ranks(e2e_ms, world)
    line = {
        "metric": METRIC, "value": round(value, 1), "unit": "GB/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(ms, 4), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": f"mxfp4 decode qGEMV M=1 N=4096 K=4096; a step = {copies} distinct weight "
                               f"copies, one qmm each ({copies * nbytes / 1e6:.0f} MB > 3x L2)",
                   "l2": "inputs larger than L2 (rotating weight copies), no flush",
                   "graph": "each step's launches replayed from one CUDA graph",
                   "accumulate": "f32"},
        "roofline": roofline_gemv(prob, ms, hbm, kind),
        "e2e": {"value": round(world * copies * nbytes / (e2e_ms * 1e-3) / 1e9, 1), "unit": "GB/s",
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                "note": "per step (one CUDA graph): one pinned H2D of all layers' X, L qmm calls, one D2H of all outputs; weights resident"},
        "step_ms_spread": spread,
        "gpu_launches": copies * args.steps,
        "clocks": clk,
    }
    del graph, prob
    torch.cuda.empty_cache()
    if rank == 0 and not args.no_breakdown and world == 1:
        rows = []
        for row in BREAKDOWN:
            f, mm, nn, kk = row[:4]
            rows.append(breakdown_row(f, mm, nn, kk, hbm, bf16, kind, path=row[4] if len(row) > 4 else "auto"))
        for (f, nn, kk, od) in DEQUANT:
            rows.append(dequant_row(f, nn, kk, od, hbm))
        for (f, mm, nn, kk, ee) in GATHER:
            rows.append(gather_row(f, mm, nn, kk, ee, hbm))
        for (f, mm, nn, kk, ee) in GROUPED:
            rows.append(gather_row(f, mm, nn, kk, ee, hbm, grouped=True))
        for (kind, f, mm, ns, kk) in FUSED:
            rows.append(fused_row(kind, f, mm, ns, kk, hbm))
        line["breakdown"] = rows
    if rank == 0 and world == 1:
        line["cpu_baseline"] = cpu_baseline(fmt, m, n, k)
        if not args.no_breakdown:
            line["cpu_baseline_per_config"] = oracle_per_config()
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
