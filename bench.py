#!/usr/bin/env python
"""Benchmark: SGEMM C = alpha*A*B + beta*C on one GB300, through the C ABI.

Default workload: the compute-bound 8192^3 case (alpha = 1, beta = 0, seed 4,
U[-1, 1) inputs).  One step = one sgemm_run over the whole problem.  Prints
one JSON line (rank 0).

  python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME]
                  [--impl ours|reference] [--no-cpu-baseline] [--no-workloads]

--impl reference times the FP64 CPU oracle (the only other implementation
here) on the same workload and metric, on the host cores, each step a bounded
sample of output rows.

Timing: CUDA events on the launching stream around exactly K back-to-back
steps, after W warm-up steps, with a barrier and a device synchronize on both
sides; the 8192^3 working set (768 MiB) is larger than L2 (129 MB).  For
N > 1 (torchrun) every rank runs its own replica and the slowest rank's time
is used.
"""
from __future__ import annotations

import argparse
import hashlib
import re
import json
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "SGEMM TFLOP/s (2MNK/t) at 4096³ and 8192³; % of GB300 FP32 peak"
UNIT = "TFLOP/s"

# DRAM bytes (read + write) of one headline call at 8192^3 -- every launch of
# the call: the transposed copy, the complete waves and the stream-K wave --
# keyed by (SHA-256 of the SIMT kernel source without comments, layout the
# kernel ran on, re-layout bits), from an ncu launch list of the headline
# command (gpu__time_duration and the DRAM byte counters of the library's
# launches in the timed steps); any other source gives traffic = null.
TRAFFIC_BY_SOURCE = {("134ea119637177b9", "TN", 1): 3.355e9}
TC_TRAFFIC_BY_SOURCE = {}
KERNEL_SOURCES = ["dense_fp32_matrix_09_gb300/csrc/sgemm_tma_kernel.cuh",
                  "dense_fp32_matrix_09_gb300/csrc/device_common.cuh",
                  "dense_fp32_matrix_09_gb300/csrc/internal.h"]
TC_KERNEL_SOURCES = ["dense_fp32_matrix_09_gb300/csrc/sgemm_tc.cu",
                     "dense_fp32_matrix_09_gb300/csrc/tcgen05.cuh",
                     "dense_fp32_matrix_09_gb300/csrc/device_common.cuh"]


RELAYOUT_NAMES = {0: "none", 1: "A", 2: "B", 3: "A+B"}


def layout_run(op: str, relayout: int) -> str:
    """Operand layout the GEMM kernel ran on after re-layout (bit 0: A was
    copied transposed, bit 1: B)."""
    ta = (op[0] == "T") ^ bool(relayout & 1)
    tb = (op[1] == "T") ^ bool(relayout & 2)
    return ("T" if ta else "N") + ("T" if tb else "N")


def kernel_code(text: str) -> str:
    """The code of a CUDA source without its comments and blank lines (a
    comment-only edit leaves the kernel, and counters taken on it, valid)."""
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    text = re.sub(r"//[^\n]*", "", text)
    return "\n".join(line.rstrip() for line in text.splitlines() if line.strip())


def kernel_source_hash(files=KERNEL_SOURCES) -> str:
    """sha256[:16] of the files' code (comments and blank lines removed)."""
    h = hashlib.sha256()
    for p in files:
        with open(os.path.join(ROOT, p), encoding="utf-8") as f:
            h.update(kernel_code(f.read()).encode())
    return h.hexdigest()[:16]


def measured_bf16_tflops(sustained: bool = False) -> dict:
    """Dense BF16 tensor throughput: the burst (or, for kernels timed in a
    long loop, the sustained) figure the driver measured on this machine
    (MEASURED_PEAKS.json), else the profiling recipe's fallback."""
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            key = "bf16_tflops_sustained" if sustained else "bf16_tflops"
            return {"value": float(json.load(f)[key]), "source": "measured"}
    except (OSError, KeyError, ValueError):
        return {"value": 1700.0 if sustained else 1900.0, "source": "fallback"}


def measured_hbm_gbs() -> dict:
    """HBM copy bandwidth measured on this machine (MEASURED_PEAKS.json), else
    the profiling recipe's fallback."""
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            return {"value": float(json.load(f)["hbm_gbs"]), "source": "measured"}
    except (OSError, KeyError, ValueError):
        return {"value": 6800.0, "source": "fallback"}


def compact(x):
    """x with every float rounded to 6 significant digits (JSON size)."""
    if isinstance(x, float):
        return float(f"{x:.6g}")
    if isinstance(x, dict):
        return {k: compact(v) for k, v in x.items()}
    if isinstance(x, (list, tuple)):
        return [compact(v) for v in x]
    return x


def parse():
    p = argparse.ArgumentParser()
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=100)
    p.add_argument("--warmup", type=int, default=5)
    p.add_argument("--workload", default=None,
                   help="workload name, or MxNxK for an ad-hoc alpha=1 beta=0 problem (default: 8192^3)")
    p.add_argument("--variant", default=os.environ.get("SGEMM_FORCE_VARIANT", "auto"),
                   help="pin a kernel variant by name (default: $SGEMM_FORCE_VARIANT, else auto)")
    p.add_argument("--impl", default="ours", choices=["ours", "reference"])
    p.add_argument("--no-cpu-baseline", action="store_true")
    p.add_argument("--no-workloads", action="store_true", help="skip the per-workload table")
    p.add_argument("--e2e-steps", type=int, default=10)
    p.add_argument("--no-tensor", action="store_true", help="skip the 3xTF32 tensor-core block")
    p.add_argument("--tensor-steps", type=int, default=50)
    p.add_argument("--op", default="NN", choices=["NN", "NT", "TN", "TT"],
                   help="operand layout of the timed step (sgemm_run_ex; square unpadded workloads only)")
    p.add_argument("--no-mixed", action="store_true",
                   help="skip the 16-bit-input (BF16 / FP16, FP32 accumulation) block (sgemm_run_mixed)")
    p.add_argument("--relayout", default="auto", choices=["auto", "off", "always"],
                   help="operand re-layout mode of the handle for the headline step (default: auto)")
    p.add_argument("--no-ex", action="store_true",
                   help="skip the transposed-layout and strided-batched block (sgemm_run_ex)")
    return p.parse_args()


# ------------------------------------------------------------------ clocks

class ClockSampler:
    """nvidia-smi samples every 200 ms while the timed region runs."""

    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_id: str | None):
        self.gpu_id = gpu_id
        self.lines: list[str] = []
        self.proc = None

    def start(self):
        cmd = ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits", "-lms", "200"]
        if self.gpu_id:
            cmd += ["-i", self.gpu_id]
        try:
            self.proc = subprocess.Popen(cmd, stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
            return
        self.t = threading.Thread(target=self._read, daemon=True)
        self.t.start()

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self) -> dict:
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"], "samples": 0}
        time.sleep(0.25)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.t.join(timeout=2)
        sm, smax, power, reasons = [], [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in self.lines:
            parts = [x.strip() for x in line.split(",")]
            if len(parts) < 8:
                continue
            try:
                sm.append(float(parts[0]))
                smax.append(float(parts[1]))
                power.append(float(parts[2]))
            except ValueError:
                continue
            for n, v in zip(names, parts[4:8]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"], "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(smax), "reasons": sorted(reasons),
                "samples": len(sm), "sm_mhz_min": min(sm), "power_w_max": max(power)}


def nvsmi_id(torch, dev: int) -> str | None:
    try:
        p = torch.cuda.get_device_properties(dev)
        return f"{p.pci_domain_id:08X}:{p.pci_bus_id:02X}:{p.pci_device_id:02X}.0"
    except Exception:
        return None


# ---------------------------------------------------------------- oracle arm

def cpu_oracle_rate(cfg, prob, seconds: float, rows_hint: int | None = None):
    """Time the oracle on a bounded sample of output rows; returns (TFLOP/s, rows, secs, cores)."""
    import oracle
    cores = oracle.num_threads()
    rows = rows_hint or max(1, min(cfg.M, cores))
    while True:
        sel = list(range(rows))
        t0 = time.perf_counter()
        oracle.sgemm_rows(sel, cfg.N, cfg.K, cfg.alpha, prob.A, cfg.lda, prob.B, cfg.ldb, cfg.beta,
                          prob.C0, cfg.ldc)
        dt = time.perf_counter() - t0
        if dt >= seconds * 0.5 or rows >= cfg.M:
            break
        rows = min(cfg.M, max(rows + 1, int(rows * seconds / max(dt, 1e-3))))
    flops = 2.0 * rows * cfg.N * cfg.K
    return flops / dt / 1e12, rows, dt, cores


def reference_arm(args, cfg, rank, world):
    if rank != 0:
        return
    from dense_fp32_matrix_09_gb300 import inputs
    import oracle
    prob = inputs.make_problem(cfg)
    cores = oracle.num_threads()
    # size one step: ~1 s of oracle work, so W + K steps stay within a few minutes
    _, rows, dt, _ = cpu_oracle_rate(cfg, prob, seconds=1.0)
    budget = 150.0
    per_step = min(1.0, budget / max(1, args.steps + args.warmup))
    rows = max(1, int(rows * per_step / max(dt, 1e-3)))
    rows = min(rows, cfg.M)
    sel = list(range(rows))

    def step():
        oracle.sgemm_rows(sel, cfg.N, cfg.K, cfg.alpha, prob.A, cfg.lda, prob.B, cfg.ldb, cfg.beta,
                          prob.C0, cfg.ldc)

    for _ in range(args.warmup):
        step()
    t0 = time.perf_counter()
    for _ in range(args.steps):
        step()
    dt = time.perf_counter() - t0
    value = 2.0 * rows * cfg.N * cfg.K * args.steps / dt / 1e12
    sample = f"{rows} of {cfg.M} output rows per step (x {cfg.N} columns, K = {cfg.K}), FP64 oracle"
    print(json.dumps({
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": dt / args.steps * 1e3,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic",
        "config": {"workload": cfg.name, "M": cfg.M, "N": cfg.N, "K": cfg.K, "alpha": cfg.alpha,
                   "beta": cfg.beta, "seed": cfg.seed},
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": cores, "kind": "oracle", "sample": sample},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }))


# ---------------------------------------------------------------- our arm

def flush_l2(torch, buf):
    buf.add_(1.0)


def time_workload(torch, sg, h, cfg, reps: int, cold: bool, flush_buf):
    """Median / mean per-call ms of one workload on device-resident inputs."""
    from dense_fp32_matrix_09_gb300 import inputs
    prob = inputs.make_problem(cfg)
    A = torch.from_numpy(prob.A).cuda()
    B = torch.from_numpy(prob.B).cuda()
    C0 = torch.from_numpy(prob.C0).cuda()
    C = C0.clone()
    stream = torch.cuda.current_stream()

    def call():
        sg.sgemm_run(h, cfg.M, cfg.N, cfg.K, cfg.alpha, A, cfg.lda, B, cfg.ldb, cfg.beta, C, cfg.ldc, stream)

    for _ in range(3):
        call()
    torch.cuda.synchronize()
    ms = []
    for _ in range(reps):
        if cfg.beta != 0:
            C.copy_(C0)
        if cold:
            flush_l2(torch, flush_buf)
        s, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        s.record(stream)
        call()
        e.record(stream)
        e.synchronize()
        ms.append(s.elapsed_time(e))
    # warm L2, per call: C restored from C0 outside each event pair (in-place
    # updates), no flush, so A, B and C are in L2 from the call before
    warm = None
    if cold and cfg.beta != 0:
        warm = []
        for _ in range(reps):
            C.copy_(C0)
            s, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            s.record(stream)
            call()
            e.record(stream)
            e.synchronize()
            warm.append(s.elapsed_time(e))
    # back-to-back (hot L2) mean, beta == 0 only (in-place updates would compound)
    hot = host_us = None
    if cfg.beta == 0:
        n = max(10, reps)
        s, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        s.record(stream)
        t0 = time.perf_counter()
        for _ in range(n):
            call()
        host_us = (time.perf_counter() - t0) / n * 1e6  # enqueue cost per call on the host (Python binding included)
        e.record(stream)
        e.synchronize()
        hot = s.elapsed_time(e) / n
    # launch-bound shapes: 20 calls captured in one CUDA graph, replayed (an
    # in-place workload updates C 20 times over: the same work per call)
    graph_ms = None
    if cfg.flops <= 2.5e9:
        gs = torch.cuda.Stream()
        gs.wait_stream(stream)
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph, stream=gs):
            for _ in range(20):
                sg.sgemm_run(h, cfg.M, cfg.N, cfg.K, cfg.alpha, A, cfg.lda, B, cfg.ldb, cfg.beta, C, cfg.ldc, gs)
        graph.replay()
        torch.cuda.synchronize()
        s, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        s.record(stream)
        for _ in range(5):
            graph.replay()
        e.record(stream)
        e.synchronize()
        graph_ms = s.elapsed_time(e) / 100
        del graph
    variant, splits = sg.sgemm_last_variant(h)
    med = statistics.median(ms)
    out = {"ms_median": med, "ms_mean": statistics.mean(ms), "ms_min": min(ms),
           "tflops": cfg.flops / (med * 1e-3) / 1e12,
           "gbs_compulsory": cfg.compulsory_bytes / (med * 1e-3) / 1e9, "reps": reps,
           "l2": "flushed before each rep" if cold else "warm", "variant": sg.variant_name(variant),
           "relayout": RELAYOUT_NAMES[sg.sgemm_last_relayout(h)]}
    if splits > 1:
        out["splits"] = splits
    if warm is not None:
        wmed = statistics.median(warm)
        out["ms_warm_median"] = wmed
        out["ms_warm_mean"] = statistics.mean(warm)
        out["tflops_warm"] = cfg.flops / (wmed * 1e-3) / 1e12
    if hot is not None:
        out["ms_back_to_back"] = hot
        out["tflops_back_to_back"] = cfg.flops / (hot * 1e-3) / 1e12
        out["us_host_enqueue_per_call"] = host_us
    if graph_ms is not None:
        out["ms_per_call_in_cuda_graph"] = graph_ms
        out["tflops_in_cuda_graph"] = cfg.flops / (graph_ms * 1e-3) / 1e12
    del A, B, C, C0
    return out


def time_calls(torch, stream, call, reps: int, warmup: int, flush_buf=None) -> list[float]:
    """Per-call device ms (CUDA events on the launching stream), L2 flushed
    before each call when flush_buf is given."""
    for _ in range(max(3, warmup)):
        call()
    torch.cuda.synchronize()
    ms = []
    for _ in range(reps):
        if flush_buf is not None:
            flush_l2(torch, flush_buf)
        s, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        s.record(stream)
        call()
        e.record(stream)
        e.synchronize()
        ms.append(s.elapsed_time(e))
    return ms


def bench_ex(torch, sg, h, cfg, A, B, C, stream, warmup: int) -> dict:
    n = cfg.M
    flops = 2.0 * n * n * n
    res = {}
    # each layout as the library runs it (operand re-layout on), then on the
    # operands as stored (re-layout off), for the layouts re-layout applies to
    for name, ta, tb in (("NN", 0, 0), ("NT", 0, 1), ("TN", 1, 0), ("TT", 1, 1)):
        def call(ta=ta, tb=tb):
            sg.sgemm_run_ex(h, ta, tb, n, n, n, 1.0, A, n, 0, B, n, 0, 0.0, C, n, 0, 1, stream)
        for mode, key in ((sg.RELAYOUT_AUTO, name), (sg.RELAYOUT_OFF, name + "_as_stored")):
            sg.sgemm_set_relayout(h, mode)
            ms = time_calls(torch, stream, call, 10, warmup)
            v, splits = sg.sgemm_last_variant(h)
            med = statistics.median(ms)
            res[key] = {"ms_median": med, "tflops": flops / (med * 1e-3) / 1e12, "variant": sg.variant_name(v),
                        "relayout": RELAYOUT_NAMES[sg.sgemm_last_relayout(h)],
                        "launches": sg.sgemm_last_launches(h)}
            if name == "TN":
                break  # TN is never re-laid out
    sg.sgemm_set_relayout(h, sg.RELAYOUT_AUTO)
    # the transposed copy of A: the NN call minus the TN call on the same
    # buffers (the same kernel on i.i.d. data of the same shape)
    if res["NN"]["relayout"] == "A":
        t_copy = res["NN"]["ms_median"] - res["TN"]["ms_median"]
        res["transpose_A_ms_est"] = t_copy
        res["transpose_A_gbs_est"] = 8.0 * n * n / (t_copy * 1e-3) / 1e9 if t_copy > 0 else None
    # strided batch: 1024 x (64 x 64) x (64 x 64), contiguous; 48 MiB < L2, so L2 is flushed before each call
    bs, m = 1024, 64
    g = torch.Generator(device="cpu").manual_seed(3)
    bA = (torch.rand(bs * m * m, generator=g) * 2 - 1).cuda()
    bB = (torch.rand(bs * m * m, generator=g) * 2 - 1).cuda()
    bC = torch.empty(bs * m * m, device="cuda")
    flush_buf = torch.empty(64 << 20, dtype=torch.float32, device="cuda")  # 256 MiB > L2

    def bcall():
        sg.sgemm_run_ex(h, 0, 0, m, m, m, 1.0, bA, m, m * m, bB, m, m * m, 0.0, bC, m, m * m, bs, stream)
    ms = time_calls(torch, stream, bcall, 50, warmup, flush_buf)
    v, _ = sg.sgemm_last_variant(h)
    med = statistics.median(ms)
    bflops = 2.0 * bs * m * m * m
    bbytes = 3 * bs * m * m * 4  # A and B read once, C written once (beta = 0)
    hbm = measured_hbm_gbs()
    res["batched_1024x64cube"] = {
        "ms_median": med, "ms_min": min(ms), "tflops": bflops / (med * 1e-3) / 1e12,
        "gbs_compulsory": bbytes / (med * 1e-3) / 1e9, "variant": sg.variant_name(v), "batch": bs,
        "l2": "flushed before each call", "compulsory_bytes": bbytes,
        "hbm_frac": (bbytes / (med * 1e-3) / 1e9) / hbm["value"] if hbm else None,
        "hbm_peak_gbs": hbm["value"] if hbm else None,
        "hbm_peak_source": hbm["source"] if hbm else None,
    }
    del bA, bB, bC, flush_buf
    # a strided batch of large products: 8 x (2048 x 2048)·(2048 x 2048), as
    # the library runs it (each A copied transposed) and on A as stored
    bs2, n2 = 8, 2048
    g2 = torch.Generator(device="cpu").manual_seed(5)
    lA = (torch.rand(bs2 * n2 * n2, generator=g2) * 2 - 1).cuda()
    lB = (torch.rand(bs2 * n2 * n2, generator=g2) * 2 - 1).cuda()
    lC = torch.empty(bs2 * n2 * n2, device="cuda")
    lflops = 2.0 * bs2 * n2 ** 3

    def lcall():
        sg.sgemm_run_ex(h, 0, 0, n2, n2, n2, 1.0, lA, n2, n2 * n2, lB, n2, n2 * n2, 0.0, lC, n2, n2 * n2, bs2,
                        stream)
    for mode, key in ((sg.RELAYOUT_AUTO, "batched_8x2048cube"), (sg.RELAYOUT_OFF, "batched_8x2048cube_as_stored")):
        sg.sgemm_set_relayout(h, mode)
        ms = time_calls(torch, stream, lcall, 20, warmup)
        v, _ = sg.sgemm_last_variant(h)
        med = statistics.median(ms)
        res[key] = {"ms_median": med, "tflops": lflops / (med * 1e-3) / 1e12, "variant": sg.variant_name(v),
                    "relayout": RELAYOUT_NAMES[sg.sgemm_last_relayout(h)], "batch": bs2,
                    "l2": "inputs larger than L2 (384 MiB)"}
    sg.sgemm_set_relayout(h, sg.RELAYOUT_AUTO)
    del lA, lB, lC
    return res


def bench_mixed(torch, sg, h, cfg, C, stream, warmup: int) -> dict:
    """16-bit A and B (i.i.d. U[-1,1) rounded to BF16 / FP16), FP32 C, n^3, all
    four layouts for BF16 and NN for FP16; roofline = the measured dense BF16
    tensor throughput (the same for FP16)."""
    n = cfg.M
    flops = 2.0 * n * n * n
    g = torch.Generator(device="cpu").manual_seed(5)
    res = {}
    peak = measured_bf16_tflops()
    for tname, in_type, dt in (("bf16", sg.IN_BF16, torch.bfloat16), ("f16", sg.IN_F16, torch.float16)):
        A16 = (torch.rand(n * n, generator=g) * 2 - 1).to(dt).cuda()
        B16 = (torch.rand(n * n, generator=g) * 2 - 1).to(dt).cuda()
        for name, ta, tb in (("NN", 0, 0), ("NT", 0, 1), ("TN", 1, 0), ("TT", 1, 1)):
            if tname == "f16" and name != "NN":
                continue
            def call(ta=ta, tb=tb):
                sg.sgemm_run_mixed(h, in_type, ta, tb, n, n, n, 1.0, A16, n, B16, n, 0.0, C, n, stream)
            ms = time_calls(torch, stream, call, 20, warmup)
            v, _ = sg.sgemm_last_variant(h)
            med = statistics.median(ms)
            tf = flops / (med * 1e-3) / 1e12
            res[f"{tname}_{name}"] = {"ms_median": med, "tflops": tf, "variant": sg.variant_name(v),
                                      "frac_of_bf16_peak": tf / peak["value"]}
        del A16, B16
    # sustained: BF16 NN back to back for about a second, clocks sampled meanwhile
    A16 = (torch.rand(n * n, generator=g) * 2 - 1).to(torch.bfloat16).cuda()
    B16 = (torch.rand(n * n, generator=g) * 2 - 1).to(torch.bfloat16).cuda()
    reps = max(1, int(1.0 / max(1e-6, res["bf16_NN"]["ms_median"] * 1e-3)))
    sampler = ClockSampler(nvsmi_id(torch, torch.cuda.current_device()))
    sampler.start()
    time.sleep(0.3)
    s0, s1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    s0.record(stream)
    for _ in range(reps):
        sg.sgemm_run_mixed(h, sg.IN_BF16, 0, 0, n, n, n, 1.0, A16, n, B16, n, 0.0, C, n, stream)
    s1.record(stream)
    s1.synchronize()
    clocks = sampler.stop()
    sus = flops * reps / (s0.elapsed_time(s1) * 1e-3) / 1e12
    del A16, B16
    peak_s = measured_bf16_tflops(sustained=True)
    res["bf16_NN_sustained"] = {"tflops": sus, "launches": reps, "clocks": clocks,
                                "frac_of_bf16_sustained_peak": sus / peak_s["value"]}
    res["roofline"] = {"bound": "tensor", "peak": peak["value"], "unit": "TFLOP/s", "peak_source": peak["source"],
                       "peak_basis": "dense BF16 (FP16 is the same rate), burst, MEASURED_PEAKS.json",
                       "sustained_peak": peak_s["value"]}
    return res


def main():
    args = parse()
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    from dense_fp32_matrix_09_gb300 import inputs
    if args.workload and args.workload in inputs.CONFIG_BY_NAME:
        cfg = inputs.CONFIG_BY_NAME[args.workload]
    elif args.workload:
        M, N, K = (int(x) for x in args.workload.lower().split("x"))
        cfg = inputs.GemmConfig(f"sgemm_{M}x{N}x{K}", M, N, K, K, N, N, 0, 1.0, 0.0)
    else:
        cfg = inputs.HEADLINE

    if args.impl == "reference":
        reference_arm(args, cfg, rank, world)
        return

    import numpy as np
    import torch
    import torch.distributed as dist
    from dense_fp32_matrix_09_gb300 import build, replicas, sgemm as sg

    if not torch.cuda.is_available():
        raise SystemExit("bench.py needs a CUDA GPU")
    torch.cuda.set_device(local)
    if world > 1:
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    build.build()

    def barrier():
        if world > 1:
            dist.barrier()

    h = sg.sgemm_create()
    sg.sgemm_set_relayout(h, {"auto": sg.RELAYOUT_AUTO, "off": sg.RELAYOUT_OFF,
                              "always": sg.RELAYOUT_ALWAYS}[args.relayout])
    if args.variant != "auto":
        names = {sg.variant_name(v): v for v in sg.GEMM_VARIANTS}
        sg.sgemm_set_variant(h, names[args.variant])
    prob = inputs.make_problem(cfg)
    A = torch.from_numpy(prob.A).cuda()
    B = torch.from_numpy(prob.B).cuda()
    C0 = torch.from_numpy(prob.C0).cuda()
    C = C0.clone()
    stream = torch.cuda.current_stream()
    in_place = cfg.beta != 0

    if args.op == "NN":
        def step():
            sg.sgemm_run(h, cfg.M, cfg.N, cfg.K, cfg.alpha, A, cfg.lda, B, cfg.ldb, cfg.beta, C, cfg.ldc, stream)
    else:
        # the same buffers read as the stored transposes (values are i.i.d., so
        # the transposed operands are as random as the originals)
        if not (cfg.M == cfg.N == cfg.K == cfg.lda == cfg.ldb == cfg.ldc):
            raise SystemExit("--op needs a square workload without padding")
        ta, tb = int(args.op[0] == "T"), int(args.op[1] == "T")

        def step():
            sg.sgemm_run_ex(h, ta, tb, cfg.M, cfg.N, cfg.K, cfg.alpha, A, cfg.lda, 0, B, cfg.ldb, 0, cfg.beta,
                            C, cfg.ldc, 0, 1, stream)

    for _ in range(args.warmup):
        if in_place:
            C.copy_(C0)
        step()
    torch.cuda.synchronize()

    # ---- timed region: K steps, events around each launch on the launching stream
    sampler = ClockSampler(nvsmi_id(torch, local))
    sampler.start()
    time.sleep(0.3)
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(2 * args.steps)]
    barrier()
    torch.cuda.synchronize()
    for i in range(args.steps):
        if in_place:
            C.copy_(C0)  # restore C outside the event pair
        ev[2 * i].record(stream)
        step()
        ev[2 * i + 1].record(stream)
    torch.cuda.synchronize()
    barrier()
    clocks = sampler.stop()
    launch_ms = [ev[2 * i].elapsed_time(ev[2 * i + 1]) for i in range(args.steps)]
    total_ms = replicas.slowest(sum(launch_ms), dist if world > 1 else None, "cuda")
    ms_step = total_ms / args.steps
    value = replicas.job_tflops(cfg.flops, ms_step, world)
    variant, splits = sg.sgemm_last_variant(h)
    launches_per_step = sg.sgemm_last_launches(h)
    relayout = sg.sgemm_last_relayout(h)
    kernel_layout = layout_run(args.op, relayout)
    status = sg.sgemm_get_device_status(h)
    if status != sg.OK:
        raise SystemExit(f"device status after the timed region: {sg.status_string(status)}")

    # ---- end to end: pinned host buffers -> device, sgemm_run, result -> host, every step
    hA = torch.from_numpy(prob.A).pin_memory()
    hB = torch.from_numpy(prob.B).pin_memory()
    hC0 = torch.from_numpy(prob.C0).pin_memory()
    hC = torch.empty_like(hC0).pin_memory()
    h2d = hA.numel() * 4 + hB.numel() * 4 + (hC0.numel() * 4 if in_place else 0)
    d2h = hC.numel() * 4

    # sgemm_run_host: host A, B (and C) -> device staging buffers in row panels,
    # each panel's GEMM as soon as its rows land, each finished panel of C back
    # to the host while the next one computes (in-place workloads: C takes the
    # previous step's result as its input, as repeated in-place updates do)
    hC.copy_(hC0)

    def e2e_step():
        sg.sgemm_run_host(h, cfg.M, cfg.N, cfg.K, cfg.alpha, hA, cfg.lda, hB, cfg.ldb, cfg.beta, hC, cfg.ldc,
                          A, B, C, stream)

    for _ in range(3):
        e2e_step()
    torch.cuda.synchronize()
    barrier()
    # events around every step: the host link is shared with other jobs on the
    # machine, and a step whose copies met their traffic is an outlier, so the
    # median step is the figure (mean, min and max reported beside it)
    e2e_ev = [torch.cuda.Event(enable_timing=True) for _ in range(args.e2e_steps + 1)]
    e2e_ev[0].record(stream)
    for i in range(args.e2e_steps):
        e2e_step()
        e2e_ev[i + 1].record(stream)
    e2e_ev[-1].synchronize()
    barrier()
    e2e_steps_ms = [e2e_ev[i].elapsed_time(e2e_ev[i + 1]) for i in range(args.e2e_steps)]
    e2e_ms = replicas.slowest(statistics.median(e2e_steps_ms), dist if world > 1 else None, "cuda")
    e2e_value = replicas.job_tflops(cfg.flops, e2e_ms, world)

    # ---- roofline of the dominant kernel (the only kernel of a step)
    props = torch.cuda.get_device_properties(local)
    sms = props.multi_processor_count
    max_mhz = clocks.get("sm_max_mhz") or 2070.0
    peak = 2 * 128 * sms * max_mhz * 1e6 / 1e12
    achieved = cfg.flops / (statistics.mean(launch_ms) * 1e-3) / 1e12
    src_hash = kernel_source_hash()
    roofline = {
        "bound": "alu", "achieved": achieved, "peak": peak, "unit": "TFLOP/s", "frac": achieved / peak,
        "traffic": (TRAFFIC_BY_SOURCE.get((src_hash, kernel_layout, relayout))
                    if cfg.name == inputs.HEADLINE.name else None),
        "kernel": f"sgemm_tma_kernel ({sg.variant_name(variant)}, {kernel_layout} layout)",
        "peak_basis": f"FP32 FFMA: 2 FLOP x 128 lanes x {sms} SMs x {max_mhz:.0f} MHz (max SM clock)",
        "achieved_basis": ("CUDA events around each sgemm_run call: "
                           + (f"the transposed copy of {RELAYOUT_NAMES[relayout]} (one HBM-bound launch) and "
                              if relayout else "") + f"the GEMM's {launches_per_step - bin(relayout).count('1')} "
                           "launch(es); traffic is the DRAM bytes of the same launches"),
    }
    if clocks.get("sm_mhz"):
        roofline["frac_at_measured_clock"] = achieved / (2 * 128 * sms * clocks["sm_mhz"] * 1e6 / 1e12)
    roofline["algorithmic_flops_per_launch"] = cfg.flops
    roofline["kernel_source_sha256_16"] = src_hash
    # the FP32 FMA rate with no memory traffic (the library's FMA probe), as a second reference
    sink = torch.empty(4 * sms * 256, device="cuda")
    fma_ms = []
    for i in range(8):
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        probe_flops = sg.sgemm_debug_fma_probe(h, sink, iters=16384, stream=stream)
        e1.record(stream)
        e1.synchronize()
        if i >= 3:
            fma_ms.append(e0.elapsed_time(e1))
    fma_tflops = probe_flops / (statistics.median(fma_ms) * 1e-3) / 1e12
    # the TF32 tensor-pipe rate with no memory traffic (the library's tensor
    # probe: the 3xTF32 pair kernel's MMA on resident tiles), for the tensor roofline
    tf32_ms = []
    for i in range(8):
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        tf32_flops = sg.sgemm_debug_tf32_probe(h, iters=4096, stream=stream)
        e1.record(stream)
        e1.synchronize()
        if i >= 3:
            tf32_ms.append(e0.elapsed_time(e1))
    tf32_tflops = tf32_flops / (statistics.median(tf32_ms) * 1e-3) / 1e12
    if sg.sgemm_get_device_status(h) != sg.OK:
        raise SystemExit("device status after the TF32 probe: timeout")
    roofline["tf32_microbench"] = {"tflops": tf32_tflops, "what": "sgemm_debug_tf32_probe: tcgen05.mma "
                                   "cta_group::2 kind::tf32 M = N = 256 on resident shared-memory tiles"}
    roofline["fma_microbench"] = {"tflops": fma_tflops, "frac": achieved / fma_tflops,
                                  "what": "sgemm_debug_fma_probe: 4 CTAs of 256 threads per SM, 16 independent "
                                          "packed FP32x2 FMA chains per thread, registers only"}
    del sink
    if variant in (sg.VARIANT_TC_3XTF32, sg.VARIANT_TC_3XTF32_PAIR):
        # a pinned tensor-core variant: its roofline is the tensor pipe's
        tc_peak = tf32_tflops / 3
        roofline = {"bound": "tensor", "achieved": achieved, "peak": tc_peak, "unit": "TFLOP/s",
                    "frac": achieved / tc_peak, "traffic": None,
                    "kernel": f"{sg.variant_name(variant)}",
                    "peak_basis": f"measured TF32 tensor-pipe rate {tf32_tflops:.1f} TFLOP/s "
                                  "(sgemm_debug_tf32_probe) / 3 TF32 MMAs per FP32 product",
                    "algorithmic_flops_per_launch": cfg.flops,
                    "kernel_source_sha256_16": kernel_source_hash(TC_KERNEL_SOURCES)}

    out = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms_step, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f32", "data": "synthetic",
        "config": {"workload": cfg.name, "M": cfg.M, "N": cfg.N, "K": cfg.K, "lda": cfg.lda,
                   "ldb": cfg.ldb, "ldc": cfg.ldc, "alpha": cfg.alpha, "beta": cfg.beta, "seed": cfg.seed,
                   "inputs": "i.i.d. U[-1,1) float32",
                   "l2": "inputs larger than L2 (working set %d MiB)" % ((prob.A.nbytes + prob.B.nbytes + prob.C0.nbytes) >> 20),
                   "variant": sg.variant_name(variant), "splits": splits, "op": args.op,
                   "relayout": RELAYOUT_NAMES[relayout], "kernel_layout": kernel_layout,
                   "launches_per_step": launches_per_step,
                   "parallelism": f"replicas x{world}" if world > 1 else "single GPU"},
        "e2e": {"value": e2e_value, "unit": UNIT, "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                "ms_per_step": e2e_ms, "steps": args.e2e_steps, "ms_per_step_basis": "median of per-step events",
                "ms_per_step_mean": statistics.mean(e2e_steps_ms), "ms_per_step_min": min(e2e_steps_ms),
                "ms_per_step_max": max(e2e_steps_ms),
                "api": "sgemm_run_host (page-locked host buffers, copies overlapped with row-panel GEMMs)"},
        "gpu_launches": args.steps * launches_per_step,
        "roofline": roofline,
        "clocks": clocks,
        "gpu": {"name": props.name, "sms": sms},
    }

    # ---- the optional tensor-core path (3xTF32) on the same workload, same timing method
    if not args.no_tensor:
        sg.sgemm_set_variant(h, sg.VARIANT_TC_3XTF32_PAIR)
        for _ in range(args.warmup):
            if in_place:
                C.copy_(C0)
            step()
        torch.cuda.synchronize()
        tc_ev = [torch.cuda.Event(enable_timing=True) for _ in range(2 * args.tensor_steps)]
        tc_sampler = ClockSampler(nvsmi_id(torch, torch.cuda.current_device()))
        tc_sampler.start()
        for i in range(args.tensor_steps):
            if in_place:
                C.copy_(C0)
            tc_ev[2 * i].record(stream)
            step()
            tc_ev[2 * i + 1].record(stream)
        torch.cuda.synchronize()
        tc_clocks = tc_sampler.stop()
        tc_ms = statistics.mean(tc_ev[2 * i].elapsed_time(tc_ev[2 * i + 1]) for i in range(args.tensor_steps))
        # the other operand layouts on the same kernel (transposed operands
        # reach it through copies into the NN layout), square workloads only
        tc_layouts = {}
        if cfg.M == cfg.N == cfg.K == cfg.lda == cfg.ldb == cfg.ldc and cfg.beta == 0:
            for name, ta, tb in (("NT", 0, 1), ("TN", 1, 0), ("TT", 1, 1)):
                def tcall(ta=ta, tb=tb):
                    sg.sgemm_run_ex(h, ta, tb, cfg.M, cfg.N, cfg.K, cfg.alpha, A, cfg.lda, 0, B, cfg.ldb, 0,
                                    cfg.beta, C, cfg.ldc, 0, 1, stream)
                lms = time_calls(torch, stream, tcall, 10, args.warmup)
                med = statistics.median(lms)
                tc_layouts[name] = {"ms_median": med, "tflops": cfg.flops / (med * 1e-3) / 1e12,
                                    "variant": sg.variant_name(sg.sgemm_last_variant(h)[0]),
                                    "copies": RELAYOUT_NAMES[sg.sgemm_last_relayout(h)]}
        sg.sgemm_set_variant(h, sg.VARIANT_AUTO)
        bf16 = measured_bf16_tflops()
        tf32_nominal_ratio = bf16["value"] * 1.1 / 2.25
        tf32_peak = tf32_tflops
        tc_tflops = cfg.flops / (tc_ms * 1e-3) / 1e12
        out["tensor_3xtf32"] = {
            "variant": "tc_3xtf32_pair", "ms_per_step": tc_ms, "value": tc_tflops, "unit": UNIT,
            "steps": args.tensor_steps, "gpu_launches": args.tensor_steps,
            "roofline": {"bound": "tensor", "achieved": tc_tflops, "peak": tf32_peak / 3, "unit": "TFLOP/s",
                         "frac": tc_tflops / (tf32_peak / 3),
                         "traffic": (TC_TRAFFIC_BY_SOURCE.get(kernel_source_hash(TC_KERNEL_SOURCES))
                                     if cfg.name == inputs.HEADLINE.name else None),
                         "kernel_source_sha256_16": kernel_source_hash(TC_KERNEL_SOURCES),
                         "peak_source": "measured",
                         "peak_basis": f"measured TF32 tensor-pipe rate {tf32_peak:.1f} TFLOP/s "
                                       "(sgemm_debug_tf32_probe: the pair kernel's MMA, M = N = 256, on resident "
                                       "tiles, one cluster per SM pair) / 3 TF32 MMAs per FP32 product",
                         "tf32_from_bf16_nominal_ratio": tf32_nominal_ratio,
                         "tensor_mma_tflops": 3 * tc_tflops, "tensor_mma_frac": 3 * tc_tflops / tf32_peak},
            "layouts": tc_layouts,
            # clocks while the steps ran: the pair kernel draws far more power
            # than the SIMT kernel, and the TF32 probe's rate is a burst figure
            "clocks": tc_clocks,
        }

    # ---- sgemm_run_ex: the four operand layouts on the headline shape, and a
    # strided batch of 1024 products of 64 x 64 matrices (device-resident)
    if not args.no_ex and rank == 0 and cfg.M == cfg.N == cfg.K == cfg.lda == cfg.ldb == cfg.ldc:
        out["layouts_and_batched"] = bench_ex(torch, sg, h, cfg, A, B, C, stream, args.warmup)

    # ---- sgemm_run_mixed: BF16 / FP16 inputs, FP32 accumulation, at the headline size
    if not args.no_mixed and rank == 0 and cfg.M == cfg.N == cfg.K == cfg.lda == cfg.ldb == cfg.ldc:
        out["mixed_16bit"] = bench_mixed(torch, sg, h, cfg, C, stream, args.warmup)

    # ---- per-workload table (device-resident; not part of the headline value)
    if not args.no_workloads and rank == 0:
        flush_buf = torch.empty(64 << 20, dtype=torch.float32, device="cuda")  # 256 MiB > L2
        table = {}
        for w, reps in zip(inputs.WORKLOADS, (200, 200, 50, 50, 20)):
            cold = (w.compulsory_bytes < 2 * 129e6)
            row = time_workload(torch, sg, h, w, reps, cold, flush_buf)
            row["frac_of_fp32_peak"] = row["tflops"] / peak  # same unit-count peak as the roofline
            if "tflops_back_to_back" in row:
                row["frac_of_fp32_peak_back_to_back"] = row["tflops_back_to_back"] / peak
            table[w.name] = row
        out["workloads"] = table
        del flush_buf

    # ---- CPU baseline: the oracle on the host cores, bounded sample (rank 0, N = 1)
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        rate, rows, dt, cores = cpu_oracle_rate(cfg, prob, seconds=12.0)
        out["cpu_baseline"] = {"value": rate, "unit": UNIT, "cores": cores, "kind": "oracle",
                               "sample": f"{rows} of {cfg.M} output rows (x {cfg.N} columns, K = {cfg.K}) "
                                         f"in {dt:.1f} s, FP64 accumulation"}
        # the oracle on every workload (all host cores, about a second each), and on one
        # core for the two smallest
        import oracle
        per = {}
        for w in inputs.WORKLOADS:
            wp = prob if w.name == cfg.name else inputs.make_problem(w)
            r, n_rows, t, c = cpu_oracle_rate(w, wp, seconds=1.0)
            per[w.name] = {"gflops": r * 1e3, "cores": c, "rows": n_rows, "seconds": t}
            if w.M * w.N * w.K <= 1024 ** 3:
                oracle.set_num_threads(1)
                try:
                    r1, n1, t1, _ = cpu_oracle_rate(w, wp, seconds=1.0)
                finally:
                    oracle.set_num_threads(c)
                per[w.name]["gflops_1_thread"] = r1 * 1e3
        out["cpu_baseline"]["workloads"] = per
    sg.sgemm_destroy(h)
    if rank == 0:
        # the per-workload table last, so that a reader keeping only the end
        # of the line still has it; floats to 6 significant digits
        if "workloads" in out:
            out["workloads"] = out.pop("workloads")
        print(json.dumps(compact(out)))
    if world > 1:
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
