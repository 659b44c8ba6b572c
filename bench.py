"""Throughput of the quantized-weight OUT_PROD on GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME] [--impl ours|reference]

A step is one pass of every call of the workload (default: the backward of
the seven projections of a 7B-shaped decoder layer at T = 8192 tokens: q/k/v/o
and gate/up in Q4_K, down in Q8_0), each call one rg_out_prod through the C
ABI with inputs resident in HBM.  Prints one JSON line (rank 0).

  value       whole-job TFLOP/s = sum 2*T*N*K over the step / step time
  e2e         the same with host inputs: pinned host -> device copies of W
              and dY and the device -> host copy of dX inside the timed loop
  roofline    the tensor-core kernel's achieved TFLOP/s over the measured
              dense bf16/fp16 peak (MEASURED_PEAKS.json: the burst figure,
              or the sustained one for a seconds-long region under the power
              cap), and the whole step's fraction of the same peak
  per_config  the method's other workloads, one call each, with their
              roofline fractions (default workload only; --no-configs)
  cpu_baseline  the CPU oracle on a bounded sample of the same workload

--impl reference times the CPU oracle itself (the only baseline this method
has; its pages publish no GPU throughput) on the same sample per step.
Multi-GPU (torchrun): every rank runs its own replica of the workload
(replicas only: the calls are independent); the step time is the max over
ranks.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from quantized_weight_out_gb300 import inputs  # noqa: E402

L2_BYTES = 129 * 1024 * 1024
METRIC = "out_prod TFLOP/s (2*T*N*K / time)"


def _traffic_record():
    """DRAM bytes per tensor-core launch from the committed ncu summary, or
    None when the kernel source has changed since those counters were taken."""
    import hashlib
    rec = os.path.join(ROOT, "profiles", "tc_traffic.json")
    csrc = os.path.join(ROOT, "quantized_weight_out_gb300", "csrc")
    srcs = [os.path.join(csrc, f) for f in ("rg_tc_kernel.cuh", "rg_tc.cu")]
    if not (os.path.exists(rec) and all(os.path.exists(x) for x in srcs)):
        return None, None
    with open(rec) as f:
        d = json.load(f)
    h = hashlib.sha256()
    for x in srcs:
        with open(x, "rb") as f:
            h.update(f.read())
    sha = h.hexdigest()
    if d.get("source_sha256") != sha:
        return None, d.get("workload")
    return d.get("dram_bytes_per_launch"), d.get("workload")


def _peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return d, "measured"
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}, "fallback"


# ---------------------------------------------------------------------------
# clocks during the timed region

class ClockSampler:
    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap,"
              "pci.bus_id,utilization.gpu")

    def __init__(self, bus_id: str | None):
        self.bus_id = bus_id
        self.proc = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "200"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
            out, _ = self.proc.communicate()
        rows = []
        for line in out.splitlines():
            c = [x.strip() for x in line.split(",")]
            if len(c) < 10:
                continue
            if self.bus_id and self.bus_id.lower() not in c[8].lower():
                continue
            rows.append(c)
        if not rows:
            return None
        load = [r for r in rows if r[9].isdigit() and int(r[9]) > 50] or rows
        sm = [float(r[0]) for r in load if r[0].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in load for i in range(4) if r[4 + i] == "Active"})
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": float(load[0][1]) if load[0][1].replace(".", "").isdigit() else None,
                "reasons": reasons, "samples": len(load),
                "power_w_max": max(float(r[2]) for r in load if r[2].replace(".", "").isdigit())}


def _bus_id(torch, dev):
    try:
        p = torch.cuda.get_device_properties(dev)
        return f"{p.pci_bus_id:02X}:{p.pci_device_id:02X}.0"
    except Exception:
        return None


# ---------------------------------------------------------------------------
# CPU oracle on a bounded sample

def oracle_sample(problems, t_rows: int, n_rows: int | None = None, min_seconds: float = 0.0):
    """Time the oracle as it stands on a slice of every call of the workload:
    the first `t_rows` rows of dY and the first `n_rows` rows of W (all of
    them when None), i.e. decode that slice of W (oracle.dequant) and contract
    it (oracle.out_prod), repeated until `min_seconds` have passed.  Returns
    (flops done, seconds, description)."""
    import oracle
    data = []
    for p in problems:
        n = p.N if n_rows is None else min(n_rows, p.N)
        tr = min(t_rows, p.T)  # a call with fewer rows of dY: all of them
        W = p.weight(n)
        dY = np.ascontiguousarray(p.dy(tr)[:, :n])
        data.append((p, n, tr, W, dY, p.dx0(tr)))
    t0 = time.perf_counter()
    flops = 0
    reps = 0
    while True:  # a tiny workload is repeated until the timing spans min_seconds
        for p, n, tr, W, dY, dX0 in data:
            Wd = oracle.dequant(p.wtype, W, n, p.K)
            oracle.out_prod(p.wtype, W, n, p.K, dY, tr, dX0, p.beta, Wd=Wd)
            flops += 2 * tr * n * p.K
        reps += 1
        dt = time.perf_counter() - t0
        if dt >= min_seconds or reps >= 10000:
            break
    what = "all" if n_rows is None else f"the first {n_rows}"
    return flops, dt, (f"every call of the workload: the first min({t_rows}, T) rows of dY, {what} "
                       f"rows of W (decode + F64 contraction), {reps} pass(es)")


# ---------------------------------------------------------------------------
# the route the method replaces: a dense F32 copy of W, then a full-F32 GEMM

def second_reference(torch, rg, problems, devbuf, stream, dev, flush, reps: int = 5):
    """Time rg_dequant into a dense F32 [N, K] buffer followed by cuBLAS SGEMM
    (TF32 off) for every call of the workload, on the resident inputs.  dX
    buffers are overwritten (the timed leg has already run)."""
    tf32 = torch.backends.cuda.matmul.allow_tf32
    torch.backends.cuda.matmul.allow_tf32 = False
    try:
        wf = torch.empty(max(p.N * p.K for p in problems), dtype=torch.float32, device=dev)

        def one():
            for i, p in enumerate(problems):
                W, dY, dX = devbuf[i]
                w = wf[:p.N * p.K].view(p.N, p.K)
                rg.check(rg.rg_dequant_async(p.wtype, W, p.N, p.K, w, stream), "rg_dequant_async")
                if p.beta != 0.0:
                    dX.addmm_(dY, w, beta=p.beta)
                else:
                    torch.mm(dY, w, out=dX)

        def dequant_only():
            for i, p in enumerate(problems):
                w = wf[:p.N * p.K].view(p.N, p.K)
                rg.check(rg.rg_dequant_async(p.wtype, devbuf[i][0], p.N, p.K, w, stream),
                         "rg_dequant_async")

        times, dq = [], []
        for r in range(2 + reps):
            for fn, out in ((one, times), (dequant_only, dq)):
                if flush is not None:
                    flush()
                a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                a.record(stream)
                fn()
                b.record(stream)
                torch.cuda.synchronize()
                if r >= 2:
                    out.append(a.elapsed_time(b))
    finally:
        torch.backends.cuda.matmul.allow_tf32 = tf32
    dq_ms = statistics.median(dq)
    dq_bytes = sum(inputs.row_bytes(p.wtype, p.K) * p.N + 4 * p.N * p.K for p in problems)
    return {"ms_per_step": statistics.median(times), "unit": "TFLOP/s", "reps": reps,
            "what": "rg_dequant to a dense F32 copy of W, then cuBLAS SGEMM with TF32 off "
                    "(median of the reps)",
            "extra_bytes_per_step": sum(8 * p.N * p.K for p in problems),
            "dequant": {"ms_per_step": dq_ms, "bytes_per_step": dq_bytes,
                        "gbs": dq_bytes / (dq_ms * 1e-3) / 1e9,
                        "what": "rg_dequant alone (bytes(W) read + 4*N*K written)"}}


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=500)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--workload", default="layer7b_t8192")
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--op", default="out_prod", choices=["out_prod", "mul_mat", "lora"],
                    help="out_prod (the backward, default), mul_mat (the forward rg_mul_mat) or "
                         "lora (the backward through W plus a low-rank adapter)")
    ap.add_argument("--rank", type=int, default=16, help="adapter rank of --op lora")
    ap.add_argument("--cpu-rows", type=int, default=1024,
                    help="dY rows per call of the CPU oracle's sample (the CPU baseline and the "
                         "reference arm's step; fewer when steps + warm-ups exceed 60)")
    ap.add_argument("--no-configs", action="store_true",
                    help="skip the per-config block (the other workloads, one call each)")
    ap.add_argument("--no-cpu", action="store_true", help="skip the CPU baseline")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-second-ref", action="store_true",
                    help="skip timing rg_dequant + cuBLAS SGEMM (the dense-F32 route)")
    ap.add_argument("--custom", default=None,
                    help="a custom call instead of --workload, e.g. q8_0:4096x14336:t8192:beta0")
    ap.add_argument("--variant", default="auto", choices=["auto", "tc", "tc1", "tc2", "smallt", "simt32"],
                    help="force a kernel variant (rg_out_prod_variant)")
    args = ap.parse_args()
    if args.custom:
        wt, nk, t, b = args.custom.split(":")
        n, k = nk.split("x")
        prob = inputs.Problem(args.custom, inputs.NAME_TO_TYPE[wt], int(n), int(k), int(t[1:]),
                              1e-3, float(b[4:]))
        inputs.WORKLOADS[args.custom] = [prob]
        args.workload = args.custom
    return args


def _dist():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def max_over_ranks(x: float, device=None) -> float:
    """The largest value of x over all ranks (the step time of a job is its
    slowest rank's); x itself without a process group."""
    import torch
    import torch.distributed as dist
    if not dist.is_available() or not dist.is_initialized() or dist.get_world_size() == 1:
        return x
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_tflops(flops_per_replica_step: int, ms_per_step: float, world: int) -> float:
    """Whole-job throughput of `world` replicas, each doing the step's flops,
    timed by the slowest rank."""
    return world * flops_per_replica_step / (ms_per_step * 1e-3) / 1e12


def _dtype_name(problems):
    return "bf16" if all(p.wtype == inputs.BF16 for p in problems) else \
        "f16" if all(p.wtype != inputs.BF16 for p in problems) else "f16+bf16"


# The BASELINE-table configs the default JSON line also reports, one call
# each (C1-C4 of the method's workloads, and one row of dY over the two
# largest layer weights: the weight-streaming small-T path).
PER_CONFIG = ["q8_0_256x256_t32", "q4_0_4096x4096_t512", "q4_k_14336x4096_t2048",
              "f16_5120x17408_t4096_beta1", "bf16_5120x17408_t4096_beta1",
              "smallt_q4_k_14336x4096_t1", "smallt_q8_0_4096x14336_t1"]


def choose_peak(peaks: dict, clocks, timed_s: float):
    """The dense tensor peak that matches how the timed region ran: the burst
    figure (a short GEMM at full clock) unless the region lasted seconds with
    the power cap active, which is how the sustained figure was measured.
    Returns (TFLOP/s, which figure)."""
    burst = float(peaks.get("bf16_tflops", peaks.get("bf16_tflops_sustained", 0.0)))
    sustained = float(peaks.get("bf16_tflops_sustained", burst))
    capped = bool(clocks) and "sw_power_cap" in (clocks.get("reasons") or [])
    if timed_s >= 1.0 and capped:
        return sustained, "bf16_tflops_sustained"
    return burst, "bf16_tflops"


def sample_rows(steps: int, warmup: int, full: int = 1024, budget_steps: int = 60) -> int:
    """dY rows per call of the CPU oracle's sample: `full`, or fewer (a
    multiple of 64, at least 64) when the reference arm's steps + warm-ups
    would otherwise run past a few minutes (about 2 s a step at 1024 rows on
    16 cores).  The reference arm and the CPU baseline take the same rows."""
    n = steps + warmup
    if n <= budget_steps:
        return full
    return max(64, (full * budget_steps // n) // 64 * 64)


def _l2_policy(step_bytes: int) -> str:
    if step_bytes >= 2 * L2_BYTES:
        return f"inputs larger than L2 ({step_bytes / 1e9:.2f} GB per step > 129 MB); no flush"
    return (f"inputs fit in L2 ({step_bytes / 1e6:.1f} MB per step): between steps a "
            f"{2 * L2_BYTES >> 20} MB write then a read of it leaves L2 holding clean lines; "
            "step time = sum of the calls' event times")


def workload_config(workload: str, problems, world: int) -> dict:
    """The JSON line's `config`, the same for both arms."""
    step_bytes = sum(p.algorithmic_bytes() for p in problems)
    return {"workload": workload, "calls": len(problems),
            "flops_per_step": sum(p.flops for p in problems),
            "algorithmic_bytes_per_step": step_bytes, "l2": _l2_policy(step_bytes),
            "parallelism": f"replicas x{world}"}


def run_reference(args):
    world, rank, _ = _dist()
    if rank != 0:
        return
    problems = inputs.WORKLOADS[args.workload]
    rows = sample_rows(args.steps, args.warmup, args.cpu_rows)
    for _ in range(args.warmup):
        oracle_sample(problems, rows)
    times, flops = [], 0
    for _ in range(args.steps):
        f, dt, desc = oracle_sample(problems, rows)
        times.append(dt)
        flops = f
    ms = 1e3 * sum(times) / len(times)
    value = flops / (ms * 1e-3) / 1e12
    cores = os.cpu_count()
    line = {"impl": "reference", "metric": METRIC, "value": value,
            "unit": "TFLOP/s", "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": ms, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": "f64", "data": "synthetic",
            "config": workload_config(args.workload, problems, world),
            "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": cores, "kind": "oracle",
                             "sample": desc},
            "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


class L2Flush:
    """Evicts L2 between timed steps: a write of twice its size, then a read
    of the same buffer, so that the lines left behind are clean and a timed
    call does not stream its inputs behind the write-back of dirty lines."""

    def __init__(self, torch, dev):
        self.torch = torch
        self.buf = torch.empty(2 * L2_BYTES // 4, dtype=torch.float32, device=dev)
        self.sink = torch.empty(1, dtype=torch.float32, device=dev)

    def __call__(self, v: float = 0.0):
        self.buf.fill_(v)
        self.torch.sum(self.buf, (0,), keepdim=True, out=self.sink)


def time_calls(torch, rg, problems, devbuf, steps: int, warmup: int, forced: int, stream, dev,
               world: int) -> dict:
    """Warm-up, then `steps` timed steps of every call of `problems` on its
    resident buffers (W, dY, dX) with nothing recorded inside a call: their
    time is the step time, the library's launch count over them the launch
    count.  Then the same steps once more with events around every call and
    around its tensor-core GEMM kernel (rg_profile_next_gemm): the per-call
    and per-kernel times.  (An event between the dY conversion and the GEMM
    stops the GEMM's programmatic early launch: about 3 % of a layer step, so
    the step is timed without those events.)  nvidia-smi clocks are sampled
    over both.  Inputs that fit in L2 are flushed between steps (outside the
    calls, whose event times then make up the step time: the first pass
    records events around each call, none inside)."""
    variants = [forced if forced else rg.rg_select_variant(p.wtype, p.N, p.K, p.T) for p in problems]
    is_tc = [v in (rg.RG_VARIANT_TC, rg.RG_VARIANT_TC_SINGLE, rg.RG_VARIANT_TC_PAIR) for v in variants]
    plans = []
    for p in problems:
        info = rg.rg_plan_info()
        rg.check(rg.rg_plan(forced, p.wtype, p.N, p.K, p.T, info), "rg_plan")
        plans.append(info.as_dict())
    step_bytes = sum(p.algorithmic_bytes() for p in problems)
    flush = L2Flush(torch, dev) if step_bytes < 2 * L2_BYTES else None

    def call(p, W, dY, dX):
        if forced:
            return rg.rg_out_prod_variant(forced, p.wtype, W, p.N, p.K, dY, p.T, dX, p.beta, stream)
        return rg.rg_out_prod(p.wtype, W, p.N, p.K, dY, p.T, dX, p.beta, stream)

    def step(events=None, kernels=False):
        for i, p in enumerate(problems):
            W, dY, dX = devbuf[i]
            if events is not None:
                events[i][0].record(stream)
                if kernels and is_tc[i]:  # the library records these around its GEMM kernel
                    rg.rg_profile_next_gemm(events[i][2], events[i][3])
            st = call(p, W, dY, dX)
            if events is not None:
                events[i][1].record(stream)
            if st != 0:
                raise RuntimeError(f"{p.name}: {rg.strerror(st)}")

    for _ in range(warmup):
        step()
        if flush is not None:
            flush()
    rg.check(rg.rg_check(stream), "warmup")
    def new_events():
        evs = [[[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in problems]
               for _ in range(steps)]
        # torch creates an event's handle at its first record; record every event
        # once so the library gets real handles (its later records are the ones timed)
        for row in evs:
            for quad in row:
                for e in quad:
                    e.record(stream)
        return evs

    evs1, evs = new_events(), new_events()
    sampler = ClockSampler(_bus_id(torch, dev))
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    sampler.start()
    time.sleep(0.3)
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    launches0 = rg.rg_launch_count()
    ev0.record(stream)
    for s in range(steps):
        step(evs1[s] if flush is not None else None)
        if flush is not None:
            flush(float(s))
    ev1.record(stream)
    launches = rg.rg_launch_count() - launches0
    torch.cuda.synchronize()
    rg.check(rg.rg_check(stream), "timed region")
    # the same steps with events around every call and its tensor-core kernel
    for s in range(steps):
        step(evs[s], kernels=True)
        if flush is not None:
            flush(float(s))
    torch.cuda.synchronize()
    clocks = sampler.stop()
    rg.check(rg.rg_check(stream), "timed kernels")
    per_call = [[evs[s][i][0].elapsed_time(evs[s][i][1]) for s in range(steps)]
                for i in range(len(problems))]
    per_gemm = [[evs[s][i][2].elapsed_time(evs[s][i][3]) for s in range(steps)] if is_tc[i] else []
                for i in range(len(problems))]
    ms_total = ev0.elapsed_time(ev1)
    if flush is not None:
        ms_total = sum(evs1[s][i][0].elapsed_time(evs1[s][i][1]) for s in range(steps)
                       for i in range(len(problems)))
    planned = steps * sum(pl["launches"] for pl in plans)
    if launches != planned:
        raise RuntimeError(f"{launches} kernel launches in the timed region, the plans say {planned}")
    return {"ms_total": ms_total, "per_call": per_call, "per_gemm": per_gemm, "launches": launches,
            "clocks": clocks, "variants": variants, "is_tc": is_tc, "plans": plans,
            "flush": flush, "step_bytes": step_bytes, "timed_s": ev0.elapsed_time(ev1) * 1e-3}


def tc_launch_bytes(p) -> int:
    """Algorithmic bytes of one tensor-core GEMM launch: the packed W, dY's
    16-bit copy (2TN), dX written (4TK; read as well when beta != 0)."""
    return p.w_bytes + 2 * p.T * p.N + 4 * p.T * p.K * (2 if p.beta != 0.0 else 1)


def config_entry(torch, rg, workload: str, steps: int, warmup: int, stream, dev, peaks: dict) -> dict:
    """One BASELINE config measured on its own (resident inputs, flushed L2
    when they fit in it): time, TFLOP/s, effective GB/s and the fractions of
    its roofline, max(2TNK / tensor peak, algorithmic bytes / HBM bandwidth).
    The call's time is the mean over the steps of the pass with nothing
    recorded inside the call; the GEMM's own time comes from the second pass."""
    problems = inputs.WORKLOADS[workload]
    devbuf = []
    for p in problems:
        dX0 = p.dx0()
        devbuf.append((torch.from_numpy(p.weight()).to(dev), torch.from_numpy(p.dy()).to(dev),
                       torch.from_numpy(dX0).to(dev) if dX0 is not None
                       else torch.zeros((p.T, p.K), device=dev)))
    r = time_calls(torch, rg, problems, devbuf, steps, warmup, 0, stream, dev, 1)
    peak, kind = choose_peak(peaks, r["clocks"], r["timed_s"])
    hbm = float(peaks["hbm_gbs"])
    p = problems[0]
    t_ms = r["ms_total"] / steps
    t = t_ms * 1e-3
    e = {"workload": workload, "wtype": inputs.TYPE_NAMES[p.wtype], "N": p.N, "K": p.K, "T": p.T,
         "beta": p.beta, "variant": int(r["variants"][0]), "plan": r["plans"][0], "steps": steps,
         "ms": t_ms, "tflops": p.flops / t / 1e12, "effective_gbs": p.algorithmic_bytes() / t / 1e9,
         "roofline_frac": max(p.flops / (peak * 1e12), p.algorithmic_bytes() / (hbm * 1e9)) / t,
         "bound": "tensor" if p.flops / (peak * 1e12) >= p.algorithmic_bytes() / (hbm * 1e9) else "hbm",
         "peak_tflops": peak, "peak_kind": kind, "hbm_gbs": hbm,
         "l2": _l2_policy(r["step_bytes"]),
         "sm_mhz": (r["clocks"] or {}).get("sm_mhz"), "clock_reasons": (r["clocks"] or {}).get("reasons")}
    if r["is_tc"][0]:
        g_ms = statistics.median(r["per_gemm"][0])
        e["gemm_ms"] = g_ms
        e["kernel_frac"] = p.flops / (g_ms * 1e-3) / 1e12 / peak
        e["step_frac"] = p.flops / t / 1e12 / peak
    del devbuf
    torch.cuda.empty_cache()
    return e


def run_ours(args):
    import torch
    world, rank, local = _dist()
    from quantized_weight_out_gb300 import binding as rg
    from quantized_weight_out_gb300 import build as rgbuild
    rgbuild.build()
    rg.load()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=dev)
    problems = inputs.WORKLOADS[args.workload]

    # inputs: generated on the host, pinned copies for the end-to-end leg,
    # device copies resident for the kernel leg
    host, devbuf = [], []
    for p in problems:
        W = torch.from_numpy(p.weight()).pin_memory()
        dY = torch.from_numpy(p.dy()).pin_memory()
        dX0 = p.dx0()
        dXh = torch.empty((p.T, p.K), dtype=torch.float32).pin_memory()
        host.append((W, dY, dXh))
        devbuf.append((W.to(dev), dY.to(dev),
                       torch.from_numpy(dX0).to(dev) if dX0 is not None
                       else torch.zeros((p.T, p.K), device=dev)))
    torch.cuda.synchronize()
    stream = torch.cuda.current_stream()
    forced = rg.VARIANTS[args.variant]

    r = time_calls(torch, rg, problems, devbuf, args.steps, args.warmup, forced, stream, dev, world)
    per_call, per_gemm, is_tc, plans = r["per_call"], r["per_gemm"], r["is_tc"], r["plans"]
    variants, clocks, launches, step_bytes = r["variants"], r["clocks"], r["launches"], r["step_bytes"]
    ms_total = max_over_ranks(r["ms_total"], dev)
    ms_step = ms_total / args.steps
    flops_step = sum(p.flops for p in problems)
    value = job_tflops(flops_step, ms_step, world)

    def call(p, W, dY, dX):
        if forced:
            return rg.rg_out_prod_variant(forced, p.wtype, W, p.N, p.K, dY, p.T, dX, p.beta, stream)
        return rg.rg_out_prod(p.wtype, W, p.N, p.K, dY, p.T, dX, p.beta, stream)

    # end to end: host buffers, copies inside the timed loop
    e2e = None
    if not args.no_e2e:
        h2d = sum(h[0].numel() * h[0].element_size() + h[1].numel() * 4 for h in host)
        d2h = sum(p.T * p.K * 4 for p in problems)

        # copies on two side streams, overlapped with compute on `stream`:
        # H2D(i) -> rg_out_prod(i) -> D2H(i).  Two sets of device buffers
        # alternate between steps, so a step's host -> device copies do not
        # wait for the previous step's calls and read-backs; the hazards on a
        # set (its previous use) are ordered by events.
        s_in, s_out = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
        sets = [devbuf, [(W.clone(), dY.clone(), dX.clone()) for W, dY, dX in devbuf]]
        ev_in = [[torch.cuda.Event() for _ in problems] for _ in sets]
        ev_done = [[torch.cuda.Event() for _ in problems] for _ in sets]
        ev_out = [[torch.cuda.Event() for _ in problems] for _ in sets]

        def e2e_step(k):
            for i, p in enumerate(problems):
                W, dY, dX = sets[k][i]
                s_in.wait_event(ev_done[k][i])
                with torch.cuda.stream(s_in):
                    W.copy_(host[i][0], non_blocking=True)
                    dY.copy_(host[i][1], non_blocking=True)
                ev_in[k][i].record(s_in)
                stream.wait_event(ev_in[k][i])
                stream.wait_event(ev_out[k][i])
                st = call(p, W, dY, dX)
                if st != 0:
                    raise RuntimeError(rg.strerror(st))
                ev_done[k][i].record(stream)
                s_out.wait_event(ev_done[k][i])
                with torch.cuda.stream(s_out):
                    host[i][2].copy_(dX, non_blocking=True)
                ev_out[k][i].record(s_out)

        e2e_step(0)
        e2e_step(1)
        torch.cuda.synchronize()
        if world > 1:
            torch.distributed.barrier()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        s_in.wait_event(e0)
        for k in range(args.steps):
            e2e_step(k % 2)
        for evs_k in ev_out:
            for ev in evs_k:
                stream.wait_event(ev)
        e1.record(stream)
        torch.cuda.synchronize()
        ems = max_over_ranks(e0.elapsed_time(e1) / args.steps, dev)
        e2e = {"value": job_tflops(flops_step, ems, world), "unit": "TFLOP/s",
               "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "ms_per_step": ems}

    # roofline of the tensor-core launches (the dominant kernel)
    peaks, src = _peaks()
    peak, peak_kind = choose_peak(peaks, clocks, r["timed_s"])
    traffic, traffic_wl = _traffic_record()
    if traffic_wl is not None and traffic_wl != args.workload:
        traffic = None
    tc = [i for i in range(len(problems)) if is_tc[i]]
    tc_flops = sum(problems[i].flops for i in tc)
    gemm_ms = sum(statistics.mean(per_gemm[i]) for i in tc) if tc else 0.0
    call_ms = sum(statistics.mean(per_call[i]) for i in tc) if tc else 0.0
    achieved = tc_flops / (gemm_ms * 1e-3) / 1e12 if gemm_ms > 0 else None
    alg_launch = sum(tc_launch_bytes(problems[i]) for i in tc) / max(1, len(tc))
    roof = {"bound": "tensor", "achieved": achieved, "peak": peak, "unit": "TFLOP/s",
            "frac": achieved / peak if achieved else None,
            "step_frac": value / world / peak if all(is_tc) else None,
            "traffic": traffic,
            "algorithmic_bytes_per_launch": alg_launch,
            "traffic_ratio": traffic / alg_launch if traffic and alg_launch else None,
            "traffic_unit": "bytes per launch (ncu dram read+write, profiles/tc_traffic.json)",
            "peak_source": f"{src} {peak_kind} (dense fp16 = bf16 nominal); the burst figure unless "
                           "the timed region lasted seconds under sw_power_cap",
            "kernel": "out_prod_tc_kernel (fused decode + tcgen05 GEMM), events around each launch "
                      "in a second pass of the same steps (the value's pass records none inside a call)",
            "launches_per_step": len(tc), "flops_per_launch": tc_flops / max(1, len(tc)),
            "ms_per_launch": gemm_ms / max(1, len(tc)),
            "dy_conversion_share_of_calls": (call_ms - gemm_ms) / call_ms if call_ms > 0 else None}
    if not tc:
        # no tensor-core call (small-T or SIMT workloads): the weight stream
        # bounds them; algorithmic bytes per call over the call's event time
        hbm = float(peaks["hbm_gbs"])
        call_ms = sum(statistics.mean(per_call[i]) for i in range(len(problems)))
        bytes_call = sum(p.algorithmic_bytes() for p in problems) / len(problems)
        achieved = step_bytes / (call_ms * 1e-3) / 1e9 if call_ms > 0 else None
        roof = {"bound": "hbm", "achieved": achieved, "peak": hbm, "unit": "GB/s",
                "frac": achieved / hbm if achieved else None, "traffic": None,
                "peak_source": f"{src} hbm_gbs",
                "kernel": "the calls' kernels (small-T: main kernel and, with a row split, "
                          "the partial-sum reduction), events around each call",
                "launches_per_step": sum(pl["launches"] for pl in plans),
                "bytes_per_call": bytes_call, "ms_per_call": call_ms / len(problems)}

    calls = []
    for i, p in enumerate(problems):
        t = statistics.median(per_call[i]) * 1e-3
        calls.append({"name": p.name, "wtype": inputs.TYPE_NAMES[p.wtype], "N": p.N, "K": p.K,
                      "T": p.T, "variant": int(variants[i]), "ms": t * 1e3,
                      "gemm_ms": statistics.median(per_gemm[i]) if per_gemm[i] else None,
                      "tflops": p.flops / t / 1e12,
                      "effective_gbs": p.algorithmic_bytes() / t / 1e9,
                      "plan": plans[i],
                      "roofline_frac": max(p.flops / (peak * 1e12),
                                           p.algorithmic_bytes() / (peaks["hbm_gbs"] * 1e9)) / t})

    second = None if args.no_second_ref else second_reference(torch, rg, problems, devbuf, stream,
                                                                   dev, r["flush"])
    if second is not None:
        second["ms_per_step"] = max_over_ranks(second["ms_per_step"], dev)
        second["value"] = job_tflops(flops_step, second["ms_per_step"], world)

    per_config = None
    if world == 1 and not args.no_configs and args.workload == "layer7b_t8192" and not forced:
        del host, devbuf
        torch.cuda.empty_cache()
        per_config = [config_entry(torch, rg, wl, 50, max(args.warmup, 3), stream, dev, peaks)
                      for wl in PER_CONFIG]

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu:
        f, dt, desc = oracle_sample(problems, sample_rows(args.steps, args.warmup, args.cpu_rows),
                                    min_seconds=10.0)
        cpu = {"value": f / dt / 1e12, "unit": "TFLOP/s", "cores": os.cpu_count(),
               "kind": "oracle", "sample": desc, "seconds": dt}

    line = {
        "metric": METRIC, "value": value, "unit": "TFLOP/s",
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_step,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": _dtype_name(problems), "data": "synthetic",
        "config": workload_config(args.workload, problems, world),
        "effective_gbs": world * step_bytes / (ms_step * 1e-3) / 1e9,
        "roofline": roof, "cpu_baseline": cpu, "e2e": e2e, "gpu_launches": launches,
        "clocks": clocks, "second_reference": second, "per_call": calls, "per_config": per_config,
    }
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        torch.distributed.destroy_process_group()


def _timed_calls(torch, rg, problems, call, args, stream, dev, world):
    """Warm-up, then `args.steps` timed steps of call(i, p) over the problems
    with nothing recorded inside a call (the step time and the launch count),
    then the same steps again with a pair of events around each call and a
    pair around its main tensor-core kernel (rg_profile_next_gemm); clocks
    sampled over both.  Returns (ms per step over ranks, launches, clocks,
    per-call ms, GEMM ms per step)."""
    def step(evs=None):
        for i, p in enumerate(problems):
            if evs is not None:
                evs[i][0].record(stream)
                rg.rg_profile_next_gemm(evs[i][2], evs[i][3])
            st = call(i, p)
            if evs is not None:
                evs[i][1].record(stream)
            if st != 0:
                raise RuntimeError(f"{p.name}: {rg.strerror(st)}")

    for _ in range(args.warmup):
        step()
    rg.check(rg.rg_check(stream), "warmup")
    evs = [[[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in problems]
           for _ in range(args.steps)]
    for row in evs:
        for quad in row:
            for e in quad:
                e.record(stream)
    sampler = ClockSampler(_bus_id(torch, dev))
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    sampler.start()
    time.sleep(0.3)
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    launches0 = rg.rg_launch_count()
    ev0.record(stream)
    for k in range(args.steps):
        step()
    ev1.record(stream)
    launches = rg.rg_launch_count() - launches0
    torch.cuda.synchronize()
    rg.check(rg.rg_check(stream), "timed region")
    for k in range(args.steps):
        step(evs[k])
    torch.cuda.synchronize()
    clocks = sampler.stop()
    rg.check(rg.rg_check(stream), "timed kernels")
    ms_step = max_over_ranks(ev0.elapsed_time(ev1) / args.steps, dev)
    per_call = [statistics.median(evs[k][i][0].elapsed_time(evs[k][i][1]) for k in range(args.steps))
                for i in range(len(problems))]
    gemm_ms = sum(statistics.mean(evs[k][i][2].elapsed_time(evs[k][i][3]) for k in range(args.steps))
                  for i in range(len(problems)))
    return ms_step, launches, clocks, per_call, gemm_ms


def _setup_gpu(torch):
    world, rank, local = _dist()
    from quantized_weight_out_gb300 import binding as rg
    from quantized_weight_out_gb300 import build as rgbuild
    rgbuild.build()
    rg.load()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=dev)
    return rg, world, rank, dev


def run_mul_mat(args):
    """The forward Y = X . deq(W)^T (rg_mul_mat) on the workload's shapes:
    same timing rules as the backward (warm-up, events, clocks, the GEMM
    alone against the measured peak); inputs resident, no e2e leg."""
    import torch
    rg, world, rank, dev = _setup_gpu(torch)
    problems = inputs.WORKLOADS[args.workload]
    bufs = []
    for p in problems:
        X = inputs.normal_f32(p.seed, 2 + p.stream_base, p.T * p.K, 1e-2).reshape(p.T, p.K)
        bufs.append((torch.from_numpy(p.weight()).to(dev), torch.from_numpy(X).to(dev),
                     torch.zeros((p.T, p.N), device=dev)))
    stream = torch.cuda.current_stream()

    def call(i, p):
        W, X, Y = bufs[i]
        return rg.rg_mul_mat(p.wtype, W, p.N, p.K, X, p.T, Y, 0.0, stream)

    ms_step, launches, clocks, per_call, gemm_ms = _timed_calls(torch, rg, problems, call, args,
                                                                stream, dev, world)
    flops_step = sum(p.flops for p in problems)
    peaks, src = _peaks()
    peak, peak_kind = choose_peak(peaks, clocks, ms_step * args.steps * 1e-3)
    achieved = flops_step / (gemm_ms * 1e-3) / 1e12
    roof = {"bound": "tensor", "achieved": achieved, "peak": peak, "unit": "TFLOP/s",
            "frac": achieved / peak, "traffic": None, "peak_source": f"{src} {peak_kind}",
            "kernel": "out_prod_tc_kernel with FWD (W decoded in the kernel as the K-major operand), "
                      "events around each launch in a second pass"}
    if all(rg.rg_mul_mat_workspace_bytes(p.wtype, p.N, p.K, p.T) == 0 for p in problems):
        # one or two rows of X: the W-streaming kernel, bound by the weight's bytes
        gbs = sum(p.w_bytes for p in problems) / (gemm_ms * 1e-3) / 1e9
        roof = {"bound": "hbm", "achieved": gbs, "peak": peaks["hbm_gbs"], "unit": "GB/s",
                "frac": gbs / peaks["hbm_gbs"], "traffic": None, "peak_source": f"{src} hbm_gbs",
                "kernel": "smallt_fwd_kernel (W streamed once, exact F32 decode), events around "
                          "each launch in a second pass; W stays in L2 between steps (no flush)"}
    calls = [{"name": p.name, "wtype": inputs.TYPE_NAMES[p.wtype], "N": p.N, "K": p.K, "T": p.T,
              "ms": t, "tflops": p.flops / (t * 1e-3) / 1e12} for p, t in zip(problems, per_call)]
    line = {"metric": "mul_mat TFLOP/s (2*T*N*K / time)", "op": "mul_mat",
            "value": job_tflops(flops_step, ms_step, world), "unit": "TFLOP/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_step,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": _dtype_name(problems), "data": "synthetic",
            "config": {"workload": args.workload, "calls": len(problems),
                       "flops_per_step": flops_step, "parallelism": f"replicas x{world}"},
            "roofline": roof,
            "gpu_launches": launches, "clocks": clocks, "per_call": calls}
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        torch.distributed.destroy_process_group()


def run_lora(args):
    """The input gradient through the resident weight plus a rank-r adapter
    (rg_out_prod_lora) on the workload's shapes, beside the base product
    alone (rg_out_prod) timed the same way, so the adapter's cost shows."""
    import torch
    rg, world, rank, dev = _setup_gpu(torch)
    problems = inputs.WORKLOADS[args.workload]
    R, scale = args.rank, 0.5
    bufs = []
    for p in problems:
        A = inputs.normal_f32(p.seed, 7 + p.stream_base, R * p.K, 0.05).reshape(R, p.K)
        B = inputs.normal_f32(p.seed, 8 + p.stream_base, p.N * R, 0.05).reshape(p.N, R)
        bufs.append((torch.from_numpy(p.weight()).to(dev), torch.from_numpy(p.dy()).to(dev),
                     torch.zeros((p.T, p.K), device=dev), torch.from_numpy(A).to(dev),
                     torch.from_numpy(B).to(dev)))
    stream = torch.cuda.current_stream()

    def call_lora(i, p):
        W, dY, dX, A, B = bufs[i]
        return rg.rg_out_prod_lora(0, p.wtype, W, p.N, p.K, dY, p.T, dX, p.beta, A, B, R, scale,
                                   stream)

    def call_base(i, p):
        W, dY, dX, _, _ = bufs[i]
        return rg.rg_out_prod_variant(0, p.wtype, W, p.N, p.K, dY, p.T, dX, p.beta, stream)

    base_ms, _, _, _, _ = _timed_calls(torch, rg, problems, call_base, args, stream, dev, world)
    ms_step, launches, clocks, per_call, gemm_ms = _timed_calls(torch, rg, problems, call_lora,
                                                                args, stream, dev, world)
    flops = [p.flops + 2 * p.T * R * (p.N + p.K) for p in problems]
    flops_step = sum(flops)
    peaks, src = _peaks()
    peak, peak_kind = choose_peak(peaks, clocks, ms_step * args.steps * 1e-3)
    # the main kernel's tensor work: the base product plus the adapter's
    # chunks (64 * ceil(r / 64) extra contraction rows)
    gemm_flops = sum(2 * p.T * p.K * (p.N + 64 * ((R + 63) // 64)) for p in problems)
    achieved = gemm_flops / (gemm_ms * 1e-3) / 1e12
    calls = [{"name": p.name, "wtype": inputs.TYPE_NAMES[p.wtype], "N": p.N, "K": p.K, "T": p.T,
              "rank": R, "ms": t, "tflops": f / (t * 1e-3) / 1e12}
             for p, t, f in zip(problems, per_call, flops)]
    line = {"metric": "out_prod+LoRA TFLOP/s (2*T*(N*K + r*(N + K)) / time)", "op": "lora",
            "value": job_tflops(flops_step, ms_step, world), "unit": "TFLOP/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_step,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": _dtype_name(problems), "data": "synthetic",
            "config": {"workload": args.workload, "calls": len(problems), "rank": R,
                       "scale": scale, "flops_per_step": flops_step,
                       "parallelism": f"replicas x{world}"},
            "base_only": {"ms_per_step": base_ms,
                          "adapter_overhead": ms_step / base_ms - 1.0},
            "roofline": {"bound": "tensor", "achieved": achieved, "peak": peak, "unit": "TFLOP/s",
                         "frac": achieved / peak, "traffic": None,
                         "peak_source": f"{src} {peak_kind}",
                         "kernel": "out_prod_tc_kernel with the adapter's chunks"},
            "gpu_launches": launches, "clocks": clocks, "per_call": calls}
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        torch.distributed.destroy_process_group()


def main():
    args = parse()
    if args.impl == "reference":
        run_reference(args)
    elif args.op == "mul_mat":
        run_mul_mat(args)
    elif args.op == "lora":
        run_lora(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
