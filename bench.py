"""Benchmark: executed TFLOP/s of the Tile-Low-Rank GEMM on the large variable-rank workload.

Workload (one step = one whole product C <- alpha A B + beta C through the C ABI):
dense C <- TLR x TLR, N = 32768, b = 1024 (32 x 32 tile grid), off-diagonal ranks
r_ij = clamp(round(256 exp(-|i-j|/4)), 8, 256) for A and B, bf16 factors ~N(0,1)/sqrt(b),
dense bf16 diagonal tiles ~N(0,1), fp32 accumulation and fp32 C, alpha = 1,
beta = 0, workspace budget 2 GiB (which forces the planner to split C).
Inputs are seeded synthetic data (``tlr_inputs``).

Default arm: ``value`` is executed TFLOP/s with inputs resident in device memory;
``e2e`` repeats the measurement with the inputs copied host-to-device from pinned
memory and C copied back every step, steps pipelined over two device copies of
the problem (one step's upload and product overlap the previous step's copy
back). ``--impl reference`` times the CPU fp64
oracle on a bounded sample of the same workload (there is no other reference
implementation to run).

Multi-GPU (torchrun): every rank runs an independent replica of the workload
(the product is not sharded), timing is the max over ranks and ``value`` sums
the ranks' executed FLOPs.
"""
from __future__ import annotations

import argparse
import json
import math
import os
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "TLR GEMM executed TFLOP/s and % of GB300 tensor peak (N=32768, var. rank)"
WORKLOAD = "large_var_rank_bf16_N32768_b1024"

# DRAM bytes (dram__bytes_read.sum + dram__bytes_write.sum) of one launch of the
# dominant kernel on this workload (the final-product launch), from one ncu
# capture. The figure belongs to the kernel sources it was taken with:
# `sources_sha256` is their hash, and the bench reports null traffic once the
# sources differ.
TRAFFIC = {"sources_sha256": "a730b281de2415948edef83104c26a92030ad638c3ff0ca52e828bb42d37bd57",
           # final-product launch (CTA pairs) of the default per-triple plan, one launch per
           # product, from a capture at N = 16384 (0.807 GB read, 1.020 GB written) scaled
           # to N = 32768: reads by the algorithmic reads (2.006 / 0.634 GB), writes by C (x4)
           "bytes_per_launch": 2.554e9 + 4.081e9,
           # its operands once and C once: terminal blocks T^R, T^L 1.662 GB, U 0.105,
           # Z 0.105 and the diagonal tiles 0.134 GB read, C 4.295 GB written
           "algorithmic_bytes_per_launch": 6.301e9}


def recorded_traffic(main_workload: bool, scale_down: int, per_triple: bool):
    """The recorded DRAM bytes per final-product launch, or None unless they were
    captured on this workload and plan with the kernel sources as they are now."""
    if not (main_workload and per_triple) or scale_down != 1 or sources_sha256() != TRAFFIC["sources_sha256"]:
        return None
    return TRAFFIC["bytes_per_launch"]


def sources_sha256() -> str:
    """Hash of the sources that decide the product's launches: the task kernel,
    its tables and the planner (the recompression unit is not part of it)."""
    import hashlib
    root = os.path.join(ROOT, "gemm_tlr_gb300", "csrc")
    h = hashlib.sha256()
    for f in ("tlr_kernels.cu", "tlr_plan.cu", "tlr_tables.h"):
        h.update(f.encode())
        with open(os.path.join(root, f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()


def _peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            m = json.load(f)
        return m, "measured"
    except OSError:
        return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}, "fallback"


class ClockSampler:
    """nvidia-smi samples (every 200 ms), kept when they fall inside the timed region.

    The sampler is started, and its first sample awaited, before the region
    opens; `mark()` brackets the region in host time, which ends after the
    closing synchronize.
    """

    def __init__(self, index: int):
        self.index = index
        self.samples = []
        self.times = []
        self.proc = None
        self.t0 = self.t1 = None

    def mark(self, which: str):
        if which == "start":
            self.t0 = time.time()
        else:
            self.t1 = time.time()

    def __enter__(self):
        q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")
        try:
            self.proc = subprocess.Popen(["nvidia-smi", f"--id={self.index}", f"--query-gpu={q}",
                                          "--format=csv,noheader,nounits", "-lms", "200"],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
            t_wait = time.time()
            while not self.samples and self.proc.poll() is None and time.time() - t_wait < 5.0:
                time.sleep(0.02)
        except OSError:
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.times.append(time.time())
            self.samples.append([x.strip() for x in line.split(",")])

    def __exit__(self, *exc):
        if self.proc:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
        return False

    def summary(self):
        if self.t0 is not None and self.t1 is not None:
            inside = [s for s, t in zip(self.samples, self.times) if self.t0 <= t <= self.t1]
            if inside:
                self.samples = inside
        if not self.samples:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
        sm = sorted(float(s[1]) for s in self.samples if len(s) > 2 and s[1].replace(".", "").isdigit())
        mx = max((float(s[2]) for s in self.samples if len(s) > 2 and s[2].replace(".", "").isdigit()), default=None)
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = set()
        for s in self.samples:
            for k, name in enumerate(names):
                if len(s) > 5 + k and s[5 + k].lower().startswith("active"):
                    reasons.add(name)
        return {"sm_mhz": sm[len(sm) // 2] if sm else None, "sm_max_mhz": mx, "reasons": sorted(reasons),
                "samples": len(self.samples)}


def reduce_max(x: float, dist=None, device: str = "cuda") -> float:
    """The largest of every rank's x (the slowest replica sets the step time)."""
    if dist is None:
        return x
    import torch
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def whole_job_tflops(world: int, flops_per_replica_step: float, ms_per_step: float) -> float:
    """Replicas only: every rank runs the whole product, so the job does world x the FLOPs."""
    return world * flops_per_replica_step / (ms_per_step * 1e-3) / 1e12


def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def sample_rc(n, b, per_tile, seed):
    import numpy as np
    rng = np.random.default_rng(seed)
    idx = set()
    for t0 in range(0, n, b):
        t1 = min(n, t0 + b)
        idx.update(int(x) for x in rng.integers(t0, t1, size=per_tile))
    return np.array(sorted(idx))


def cpu_baseline(p, flops_total, target_s=10.0, per_tile=None):
    """Time the fp64 oracle on a bounded sample of C's entries, scaled to the metric.

    Without `per_tile` the sample grows (rows and columns per tile doubling)
    until one evaluation takes a quarter of `target_s`; with it, one evaluation
    of that sample is timed. Returns the baseline record, the seconds of the
    timed evaluation and the sample size used."""
    import numpy as np
    import oracle
    oracle.build()
    grow = per_tile is None
    per_tile = per_tile or 4
    while True:
        rows = sample_rc(p.m, p.A.b, per_tile, 1)
        cols = sample_rc(p.n, p.A.b, per_tile, 2)
        t0 = time.perf_counter()
        oracle.gemm_problem(p, rows, cols)
        dt = time.perf_counter() - t0
        if not grow or dt >= target_s / 4 or per_tile >= 64:
            break
        per_tile *= 2
    frac = (len(rows) * len(cols)) / float(p.m * p.n)
    tflops = flops_total * frac / dt / 1e12
    # the oracle's own arithmetic: a dense dot product of length K per sampled entry
    K = p.A.cols if p.opA == "N" else p.A.rows
    own = 2.0 * len(rows) * len(cols) * K / dt / 1e12
    return {"value": tflops, "unit": "TFLOP/s", "cores": oracle.num_threads(), "kind": "oracle",
            "value_own_flops": own,
            "sample": f"{len(rows)} rows x {len(cols)} columns of C ({frac:.2e} of the entries), "
                      f"{dt:.2f} s; value: the method's executed FLOPs scaled by that fraction; "
                      f"value_own_flops: the oracle's own 2 K FLOPs per sampled entry (K = {K})"}, dt, per_tile


def default_plan_flops(p) -> float:
    """Executed FLOPs of the default plan, counted from the ranks alone with the
    default's rule (per-triple order when its final stage needs at most 90 % of
    the cheaper single order's), so that both arms divide by the same count."""
    from gemm_tlr_gb300 import flops as fl
    if p.A.kind == "tlr" and p.B.kind == "tlr" and p.dtype != "f32":
        tri = fl.executed_flops_triple(p)
        single = min(fl.executed_flops(p, "R")["stage3"], fl.executed_flops(p, "L")["stage3"])
        if tri["stage3"] <= 0.9 * single:
            return tri["total"]
    return fl.executed_flops(p, "R")["total"]


def time_other_plan(g, h, dp, order: str, steps: int, stream) -> dict:
    """The same product under another plan (same buffers and workspace), timed
    like the main measurement over `steps` products."""
    import torch
    plan = g.tlr_plan_create(h, dp.opA, dp.opB, dp.A.desc, dp.B.desc, dp.ws.data_ptr(), dp.ws_bytes, ORDERS[order])
    try:
        info = g.tlr_plan_info(plan)
        for _ in range(3):
            g.tlr_plan_execute(plan, dp.p.alpha, dp.p.beta, dp.C.data_ptr(), dp.ldc)
        torch.cuda.synchronize()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        for _ in range(steps):
            g.tlr_plan_execute(plan, dp.p.alpha, dp.p.beta, dp.C.data_ptr(), dp.ldc)
        b.record(stream)
        torch.cuda.synchronize()
        ms = a.elapsed_time(b) / steps
        return {"order": order, "ms_per_step": ms, "flops_per_step": info["flops_executed"],
                "executed_tflops": info["flops_executed"] / (ms * 1e-3) / 1e12, "runs": info["runs"],
                "runs_left": info["runs_left"], "runs_triple": info["runs_triple"], "steps": steps}
    finally:
        g.tlr_plan_destroy(plan)


def run_reference(args):
    world, rank, _ = dist_env()
    if rank != 0:
        return 0
    import tlr_inputs
    p = tlr_inputs.problem(5)
    total = default_plan_flops(p)
    # one sample size for every step, chosen so the whole run stays near two minutes
    per_step_s = min(4.0, max(0.1, 120.0 / max(1, args.steps + args.warmup)))
    _, _, per_tile = cpu_baseline(p, total, target_s=4 * per_step_s)
    for _ in range(args.warmup):
        cpu_baseline(p, total, per_tile=per_tile)
    vals, times = [], []
    for _ in range(args.steps):
        cb, dt, _ = cpu_baseline(p, total, per_tile=per_tile)
        vals.append(cb["value"])
        times.append(dt)
    value = sum(vals) / len(vals)
    line = {"metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": 1e3 * sum(times) / len(times), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic", "impl": "reference",
            "config": {"workload": WORKLOAD, "N": 32768, "b": 1024, "note": "CPU fp64 oracle on sampled entries"},
            "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": cb["cores"], "kind": "oracle",
                             "sample": cb["sample"]},
            "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)
    return 0


ORDERS = {"auto": 0, "right": 1, "left": 2, "triple": 3, "per_rect": 4}   # tlr_order_t

# Nominal dense tensor-core peaks of one GB300 (TFLOP/s): bf16/fp16 2250, tf32 1100.
NOMINAL_TFLOPS = {"bf16": 2250.0, "f16": 2250.0, "f32": 1100.0}
LINK_PROBES = 5   # timed copies of a step's inputs and result for the link-rate estimate


def dtype_peaks(dtype: str, peaks: dict):
    """(burst, sustained) TFLOP/s for the tensor-core type a product runs on: the
    measured bf16 figures, times the nominal tf32/bf16 ratio for fp32 inputs."""
    scale = NOMINAL_TFLOPS[dtype] / NOMINAL_TFLOPS["bf16"]
    burst = float(peaks.get("bf16_tflops")) * scale
    sus = float(peaks.get("bf16_tflops_sustained", peaks.get("bf16_tflops"))) * scale
    return burst, sus


def peak_choice(region_ms: float) -> str:
    """The measured peak a timed region is compared with: the burst figure for a
    region shorter than three seconds (the power cap has not settled), else the
    sustained one."""
    return "burst" if region_ms < 3000.0 else "sustained"


def gpu_local_cpus(index: int):
    """CPUs the kernel lists as local to GPU `index` (its PCI device's
    local_cpulist), restricted to this process's affinity; None if unknown."""
    try:
        out = subprocess.run(["nvidia-smi", f"--id={index}", "--query-gpu=pci.bus_id", "--format=csv,noheader"],
                             capture_output=True, text=True, timeout=20).stdout.strip()
        dom, rest = out.split(":", 1)
        sysid = "%04x:%s" % (int(dom, 16), rest.lower())
        text = open(f"/sys/bus/pci/devices/{sysid}/local_cpulist").read().strip()
    except (OSError, ValueError, subprocess.SubprocessError):
        return None
    cpus = set()
    for part in text.split(","):
        if "-" in part:
            a, b = part.split("-")
            cpus.update(range(int(a), int(b) + 1))
        elif part:
            cpus.add(int(part))
    mine = os.sched_getaffinity(0)
    local = sorted(cpus & mine)
    return local if local and len(local) < len(mine) else None


class near_gpu:
    """Runs the block with this thread bound to the GPU's local CPUs, so that host
    memory it allocates and first touches (the pinned staging buffers) lands on
    the GPU's NUMA node; the previous affinity comes back afterwards."""

    def __init__(self, index: int):
        self.index = index
        self.cpus = None

    def __enter__(self):
        self.saved = os.sched_getaffinity(0)
        self.cpus = gpu_local_cpus(self.index)
        if self.cpus:
            os.sched_setaffinity(0, self.cpus)
        return self

    def __exit__(self, *exc):
        os.sched_setaffinity(0, self.saved)
        return False


def input_bytes(p) -> int:
    es = 4 if p.dtype == "f32" else 2
    n = 0
    for X in (p.A, p.B):
        if X.kind == "dense":
            n += X.data.size * es
        else:
            n += X.nbytes_device()
    return n


def algorithmic_bytes(p) -> int:
    """Every input once, C written once (and read once when beta != 0)."""
    return input_bytes(p) + p.m * p.n * 4 * (2 if p.beta != 0.0 else 1)


def per_config_timings(h, stream, local: int, peaks: dict, cfgs=(1, 2, 3, 4)) -> dict:
    """The other four workloads at full size: per config the mean product time
    (CUDA events around each product on the library's stream, L2 flushed by a
    256 MiB write before every timed product, 10 untimed products first; at
    least 100 timed products for configs 1-2 and 20 for 3-4, and at least 0.5 s
    of them), executed TFLOP/s, tensor-core and HBM fractions, and the SM clock."""
    import torch
    import gemm_tlr_gb300 as g
    import tlr_inputs
    from gemm_tlr_gb300 import flops as fl
    from gemm_tlr_gb300.device import DeviceProblem
    flush = torch.empty(256 << 20, dtype=torch.uint8, device="cuda")
    out = {}
    for cfg in cfgs:
        p = tlr_inputs.problem(cfg)
        dp = DeviceProblem(p)
        try:
            dp.make_plan(h)
            info = dp.info()
            rects = g.tlr_plan_rects(dp.plan)
            flops = info["flops_executed"]
            counted = fl.executed_flops_rects(p, rects)["total"]
            assert abs(counted - flops) <= 1e-9 * flops, (cfg, counted, flops)
            for _ in range(10):
                dp.run()
            torch.cuda.synchronize()
            min_iters = 100 if cfg in (1, 2) else 20
            evs = []
            with ClockSampler(local) as clk:
                clk.mark("start")
                t_start = time.time()
                while len(evs) < min_iters or time.time() - t_start < 0.5:
                    flush.fill_(len(evs) & 255)
                    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                    a.record(stream)
                    dp.run()
                    b.record(stream)
                    evs.append((a, b))
                    if len(evs) % 64 == 0:
                        torch.cuda.synchronize()
                    if len(evs) >= 20000:
                        break
                torch.cuda.synchronize()
                clk.mark("end")
            assert g.tlr_get_device_status(h) == 0
            ms = sum(a.elapsed_time(b) for a, b in evs) / len(evs)
            burst, sus = dtype_peaks(p.dtype, peaks)
            tflops = flops / (ms * 1e-3) / 1e12
            ab = algorithmic_bytes(p)
            out[str(cfg)] = {
                "workload": p.name, "dtype": p.dtype, "ms": ms, "runs_timed": len(evs),
                "flops_executed": flops, "executed_tflops": tflops,
                "tensor_frac_of_burst": tflops / burst, "tensor_peak_burst_tflops": burst,
                "algorithmic_bytes": ab, "hbm_gbs": ab / (ms * 1e-3) / 1e9,
                "hbm_frac": ab / (ms * 1e-3) / 1e9 / float(peaks["hbm_gbs"]),
                "rects": len(rects), "orders": "".join(r[4] for r in rects),
                "clocks": clk.summary(),
            }
        finally:
            dp.close()
    del flush
    return out


# fp32 lanes per SM, SMs and the maximum SM clock of a GB300: the ALU peak the
# recompression's SIMT kernels are measured against (2 FLOP per fused multiply-add)
FP32_LANES_PER_SM, SMS, SM_MAX_GHZ = 128, 152, 2.07


def tlr_output_timings(h, stream, local: int, peaks: dict, n: int, eps: float, r_max: int, s: int,
                       steps: int, warmup: int) -> dict:
    """TLR output of the large product's family at order n (b = 1024, bf16): the
    dense-output product into a scratch C, then tlr_compress of C's tiles
    (sketch of s columns, rank at most r_max, tolerance eps). Each stage timed
    with CUDA events on the library's stream over `steps` products."""
    import numpy as np
    import torch
    import gemm_tlr_gb300 as g
    import tlr_inputs
    from gemm_tlr_gb300.device import DeviceCompression, DeviceProblem
    p = tlr_inputs.var_rank_grid(n)
    dp = DeviceProblem(p)
    b = p.A.b
    dc = DeviceCompression(p.m, p.n, b, True, eps, r_max, tlr_inputs.sketch(b, s))
    try:
        dp.make_plan(h)
        for _ in range(warmup):
            dp.run()
            dc.run(h, dp.C, dp.ldc)
        torch.cuda.synchronize()
        ev = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(steps)]
        with ClockSampler(local) as clk:
            clk.mark("start")
            for e in ev:
                e[0].record(stream)
                dp.run()
                e[1].record(stream)
                dc.run(h, dp.C, dp.ldc)
                e[2].record(stream)
            torch.cuda.synchronize()
            clk.mark("end")
        assert g.tlr_get_device_status(h) == 0
        prod_ms = sum(e[0].elapsed_time(e[1]) for e in ev) / steps
        comp_ms = sum(e[1].elapsed_time(e[2]) for e in ev) / steps
        ranks = dc.ranks.cpu().numpy().reshape(dc.nI, dc.nJ)
        errors = dc.errors.cpu().numpy().reshape(dc.nI, dc.nJ)
        nt = dc.nI
        low = ~np.eye(nt, dtype=bool)
        tiles = int(low.sum())
        # SIMT work per low-rank tile (b x b): sketch and projection 2 b^2 s each,
        # core 2 s^2 b, factors 2 (2 b) s r_max, Gram-Schmidt 2 (2 b s^2 / 2)
        flop = tiles * (4.0 * b * b * s + 2.0 * s * s * b + 4.0 * b * s * r_max + 2.0 * b * s * s)
        c_bytes = 4.0 * p.m * p.n
        out_bytes = 4.0 * float(ranks[low].sum()) * 2 * b + 4.0 * nt * b * b
        alu_peak = FP32_LANES_PER_SM * SMS * 2 * SM_MAX_GHZ / 1e3   # TFLOP/s
        return {
            "workload": f"{p.name} with TLR output", "n": n, "b": b, "eps": eps, "r_max": r_max, "sketch": s,
            "steps": steps, "product_ms": prod_ms, "compress_ms": comp_ms,
            "ranks": {"mean": float(ranks[low].mean()), "min": int(ranks[low].min()), "max": int(ranks[low].max()),
                      "at_cap": float((ranks[low] == r_max).mean())},
            "errors": {"mean": float(errors[low].mean()), "max": float(errors[low].max())},
            "compress_simt_tflops": flop / (comp_ms * 1e-3) / 1e12,
            "compress_alu": {"bound": "alu", "achieved": flop / (comp_ms * 1e-3) / 1e12, "peak": alu_peak,
                             "unit": "TFLOP/s", "frac": flop / (comp_ms * 1e-3) / 1e12 / alu_peak,
                             "peak_source": "152 SMs x 128 fp32 lanes x 2 FLOP x 2.07 GHz"},
            "compress_hbm": {"algorithmic_bytes": c_bytes + out_bytes,
                             "gbs": (c_bytes + out_bytes) / (comp_ms * 1e-3) / 1e9,
                             "frac": (c_bytes + out_bytes) / (comp_ms * 1e-3) / 1e9 / float(peaks["hbm_gbs"]),
                             "note": "C read once and the factors written once; the kernels read C three times"},
            "clocks": clk.summary(),
        }
    finally:
        dp.close()


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=500)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--e2e-steps", type=int, default=0,
                    help="end-to-end steps (0: about two seconds at the link's usual rate, 40 to 400)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-per-config", action="store_true", help="skip the timings of the other four workloads")
    ap.add_argument("--scale-down", type=int, default=1,
                    help="profile a smaller member of the workload family (N/s, b/s, budget/s^2); "
                         "bench lines are taken at 1")
    ap.add_argument("--workload", default="large_var_rank",
                    choices=["large_var_rank", "skewed8x8", "var_rank", "tlr_output"],
                    help="skewed8x8: the pages' variable-rank 8 x 8 grid (b = N/8, ranks on [b/32, b/16]), "
                         "a second measurement beside the metric's workload; var_rank: the large product's "
                         "tiles and rank rule at order --n (smaller cases for profiling); tlr_output: that "
                         "product with TLR output (recompression timed beside the product)")
    ap.add_argument("--n", type=int, default=65536, help="order of the skewed8x8 or var_rank workload")
    ap.add_argument("--dtype", default="f16", choices=["f16", "bf16", "f32"], help="element type of skewed8x8")
    ap.add_argument("--budget-gib", type=float, default=None,
                    help="workspace budget in GiB for the skewed8x8 / var_rank workloads (profiling)")
    ap.add_argument("--order", default="auto", choices=["auto", "right", "left", "triple", "per_rect"],
                    help="association order of the plan: per rectangle (auto), forced, or per tile triple")
    args = ap.parse_args()
    args.warmup = max(args.warmup, 3)
    if args.impl == "reference":
        return run_reference(args)

    import numpy as np
    import torch
    import __graft_entry__
    import gemm_tlr_gb300 as g
    import tlr_inputs
    from gemm_tlr_gb300 import flops as fl
    from gemm_tlr_gb300.device import DeviceProblem

    world, rank, local = dist_env()
    torch.cuda.set_device(local)
    if args.workload == "tlr_output":
        __graft_entry__.build()
        h = g.tlr_create(torch.cuda.current_stream().cuda_stream)
        peaks, _ = _peaks()
        n = args.n if args.n != 65536 else 16384
        res = tlr_output_timings(h, torch.cuda.current_stream(), local, peaks, n, 1e-2, 96, 128,
                                 min(args.steps, 20), args.warmup)
        g.tlr_destroy(h)
        if rank == 0:
            print(json.dumps({"metric": "TLR-output GEMM: recompression time beside the dense-output product",
                              "value": res["compress_ms"], "unit": "ms", "higher_is_better": False,
                              "n_gpus": 1, "dtype": "f32", "data": "synthetic", "config": {"workload": res["workload"]},
                              "tlr_output": res}), flush=True)
        return 0
    dist = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    __graft_entry__.build()
    stream = torch.cuda.current_stream()
    h = g.tlr_create(stream.cuda_stream)

    main_workload = args.workload == "large_var_rank"
    if main_workload:
        p = tlr_inputs.problem(5, scale_down=args.scale_down)
    elif args.workload == "var_rank":
        p = tlr_inputs.var_rank_grid(args.n)
        args.no_cpu_baseline = True
    else:
        p = tlr_inputs.skewed_grid(args.n, args.dtype)
        args.no_cpu_baseline = True
    if args.budget_gib is not None and not main_workload:
        p.budget = int(args.budget_gib * (1 << 30))
    # pinned host copies of the inputs (end-to-end timing) on the GPU's NUMA node
    with near_gpu(local) as numa:
        dp = DeviceProblem(p, pinned=True)
        C_host = torch.empty(p.m * p.n, dtype=torch.float32).pin_memory()
        C_host.zero_()
    dp.make_plan(h, order=ORDERS[args.order])
    info = dp.info()
    order = ("per-triple" if info["runs_triple"] == info["runs"] else
             "L" if info["runs_left"] == info["runs"] else ("R" if info["runs_left"] == 0 else "mixed"))
    flops_step = info["flops_executed"]
    # the planner's count, recounted from the ranks rectangle by rectangle with each one's order
    rects = g.tlr_plan_rects(dp.plan)
    counted = fl.executed_flops_rects(p, rects)["total"]
    assert abs(counted - flops_step) <= 1e-9 * flops_step, (counted, flops_step)

    def barrier():
        if dist is not None:
            dist.barrier()
        torch.cuda.synchronize()

    def max_over_ranks(x):
        return reduce_max(x, dist, "cuda")

    # ---- device-resident timing (value)
    for _ in range(args.warmup):
        dp.run()
    g.tlr_reset_timing(h)
    g.tlr_set_timing(h, True)
    barrier()
    with ClockSampler(local) as clk:
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        clk.mark("start")
        e0.record(stream)
        for _ in range(args.steps):
            dp.run()
        e1.record(stream)
        barrier()
        clk.mark("end")
    g.tlr_set_timing(h, False)
    ms_total = max_over_ranks(e0.elapsed_time(e1))
    ms_step = ms_total / args.steps
    status = g.tlr_get_device_status(h)
    kern = {k: g.tlr_get_timing(h, k) for k in range(6)}
    value = whole_job_tflops(world, flops_step, ms_step)

    # ---- end-to-end through the same entry point, host buffers in and out
    h2d = sum(t.numel() * t.element_size() for t in dp.A.host.values()) + \
        sum(t.numel() * t.element_size() for t in dp.B.host.values())
    d2h = C_host.numel() * 4

    def e2e_step():
        dp.A.upload()
        dp.B.upload()
        dp.run()
        C_host.copy_(dp.C, non_blocking=True)

    # link rates of the same buffers, copies alone (for the expected end-to-end
    # time): the median of LINK_PROBES probes, so that one probe caught in a slow
    # phase of the host link does not set the estimate
    e2e_step()
    barrier()
    probes = []
    for _ in range(LINK_PROBES):
        l0, l1, l2 = (torch.cuda.Event(enable_timing=True) for _ in range(3))
        l0.record(stream)
        dp.A.upload()
        dp.B.upload()
        l1.record(stream)
        C_host.copy_(dp.C, non_blocking=True)
        l2.record(stream)
        barrier()
        probes.append((l0.elapsed_time(l1), l1.elapsed_time(l2)))
    h2d_ms = sorted(q[0] for q in probes)[len(probes) // 2]
    d2h_ms = sorted(q[1] for q in probes)[len(probes) // 2]
    # steps for about two seconds at the link's usual rate, and at least 40: the
    # host link of this machine has slow phases (copies at a fifth of their usual
    # rate for a second or more), which a long region averages and the per-step
    # spread below shows; a probe copy caught in one must not shorten the region
    usual_ms = (h2d + d2h) / 150e9 * 1e3 + ms_step
    e2e_steps = args.e2e_steps or min(400, max(40, math.ceil(2000.0 / max(1e-3, usual_ms))))
    e2e_steps = int(max_over_ranks(float(e2e_steps)))   # every rank runs the same number
    # Steps are pipelined over two device copies of the problem (inputs, C,
    # workspace and plan): step q uploads its inputs on a copy-in stream, runs
    # the product on the library's stream and copies its C back on a copy-out
    # stream, so that step q + 1's upload and product overlap step q's copy back
    # on the full-duplex link. Every step still moves its own inputs in and its
    # whole C out inside the timed region; a copy's buffers are reused only
    # after the step two back has finished with them.
    dp2 = DeviceProblem(p)
    dp2.make_plan(h, order=ORDERS[args.order])
    sets = (dp, dp2)
    s_in, s_out = torch.cuda.Stream(), torch.cuda.Stream()

    def upload(dst, src):
        for name, hbuf in src.host.items():
            dst.dev[name].copy_(hbuf, non_blocking=True)

    dp2.run()   # the second plan's first execution outside the timed region
    barrier()
    start = torch.cuda.Event(enable_timing=True)
    ev_comp, ev_out = [], []
    start.record(stream)
    s_in.wait_event(start)
    s_out.wait_event(start)
    for q in range(e2e_steps):
        d = sets[q % 2]
        with torch.cuda.stream(s_in):
            if q >= 2:
                s_in.wait_event(ev_comp[q - 2])   # the product two back has read these inputs
            upload(d.A, dp.A)
            upload(d.B, dp.B)
            e_in = torch.cuda.Event()
            e_in.record(s_in)
        stream.wait_event(e_in)
        if q >= 2:
            stream.wait_event(ev_out[q - 2])      # the copy two back has read this C
        d.run()
        ev_comp.append(torch.cuda.Event())
        ev_comp[-1].record(stream)
        with torch.cuda.stream(s_out):
            s_out.wait_event(ev_comp[-1])
            C_host.copy_(d.C, non_blocking=True)
            ev_out.append(torch.cuda.Event(enable_timing=True))
            ev_out[-1].record(s_out)
    barrier()
    per_step = sorted([start.elapsed_time(ev_out[0])] +
                      [ev_out[q - 1].elapsed_time(ev_out[q]) for q in range(1, e2e_steps)])
    e2e_ms = max_over_ranks(start.elapsed_time(ev_out[-1])) / e2e_steps
    e2e_value = whole_job_tflops(world, flops_step, e2e_ms)
    # the host copy of the last step's C is that step's device result
    last = sets[(e2e_steps - 1) % 2].C
    pick = torch.randint(0, C_host.numel(), (65536,))
    e2e_check = bool(torch.equal(C_host[pick], last[pick.to(last.device)].cpu()))

    peaks, peak_src = _peaks()
    peak_burst, peak_sus = dtype_peaks(p.dtype, peaks)
    peak_nominal = NOMINAL_TFLOPS[p.dtype]
    which = peak_choice(ms_total)
    peak_used = peak_burst if which == "burst" else peak_sus
    # dominant kernel: the launch class with the most time. Classes: 5 = a whole
    # product in one launch; 1 = Stages 1-2 of a rectangle and 2 = its final
    # products (two launches per rectangle); 0 = Stage 1 alone (diagnostic split).
    fl = info["flops_launch"]
    class_flops = {5: flops_step, 2: fl[2], 1: fl[0] + fl[1], 0: fl[0]}
    if os.environ.get("TLR_SPLIT_LAUNCHES") == "1":
        class_flops[1] = fl[1]
    et = {"bf16": "bf16", "f16": "fp16", "f32": "tf32"}[p.dtype]
    names = {5: f"tlr_task_gemm<{et}>: Stages 1-3 and the dense-tile terms of a product in one persistent launch",
             2: f"tlr_task_gemm<{et}, CTA pairs>: final products (Stage 3 and the dense-tile segment) of a rectangle",
             1: f"tlr_task_gemm<{et}, single CTAs>: Stages 1-2 and the dense precomputes of a rectangle",
             0: f"tlr_task_gemm<{et}>: Stage 1 and the dense precomputes in a launch of their own"}
    dom = max((k for k in (5, 2, 1, 0) if kern[k][1]), key=lambda k: kern[k][0], default=None)
    roof = None
    if dom is not None:
        k_ms, k_n = kern[dom]
        launches_per_step = k_n / args.steps
        per_launch_flops = class_flops[dom] / launches_per_step
        avg_ms = k_ms / k_n
        achieved = per_launch_flops / (avg_ms * 1e-3) / 1e12
        roof = {"bound": "tensor", "achieved": achieved, "peak": peak_used, "unit": "TFLOP/s",
                "frac": achieved / peak_used, "traffic": recorded_traffic(main_workload, args.scale_down, order == "per-triple"),
                "traffic_unit": "bytes per launch (DRAM read + write)",
                "algorithmic_bytes": (TRAFFIC["algorithmic_bytes_per_launch"]
                                      if main_workload and args.scale_down == 1 and order == "per-triple" else None),
                "kernel": names[dom] + " (executed FLOPs per launch / mean launch time)",
                "launches_per_step": launches_per_step,
                "peak_source": f"{peak_src} bf16 {which} (timed region {ms_total / 1e3:.2f} s: burst below 3 s, "
                               f"sustained from 3 s)" + ("; tf32 = bf16 x 1.1/2.25" if p.dtype == "f32" else ""),
                "frac_of_burst": achieved / peak_burst, "frac_of_sustained": achieved / peak_sus,
                "frac_of_nominal": achieved / peak_nominal, "nominal_peak": peak_nominal}
    line = {
        "metric": METRIC if main_workload else (
            "TLR GEMM executed TFLOP/s (variable-rank grid, b = 1024)" if args.workload == "var_rank"
            else "TLR GEMM executed TFLOP/s (pages' skewed-rank 8x8 grid)"),
        "value": value, "unit": "TFLOP/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms_step, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": p.dtype, "data": "synthetic",
        "config": {"workload": WORKLOAD if main_workload and args.scale_down == 1 else p.name, "N": p.m, "b": p.A.b,
                   "tile_grid": [p.m // p.A.b, p.n // p.A.b],
                   "ranks": "clamp(round(256 exp(-|i-j|/4)), 8, 256)" if args.workload != "skewed8x8" else
                            "b/32 + floor((b/32 + 1) u^2), u ~ U[0,1), on [b/32, b/16]",
                   "alpha": p.alpha, "beta": p.beta,
                   "workspace_budget_bytes": p.budget, "runs": info["runs"], "order": order,
                   "l2": f"inputs larger than L2 (C alone is {p.m * p.n * 4 / 1e9:.1f} GB)",
                   "parallelism": f"replicas x{world}" if world > 1 else "single GPU"},
        "pct_of_peak": {"burst": value / world / peak_burst, "sustained": value / world / peak_sus,
                        "nominal": value / world / peak_nominal, "used": which,
                        "source": f"{peak_src} bf16 (torch.matmul 8192^3 burst and 4 s loop); nominal "
                                  f"{peak_nominal:.0f} TFLOP/s dense",
                        "target": "whole product >= 0.70 of the tensor-core peak"},
        "flops_per_step": flops_step,
        "kernel_ms_per_step": {name: kern[k][0] / args.steps for k, name in
                               enumerate(["stage1", "stages1_2" if os.environ.get("TLR_SPLIT_LAUNCHES") != "1"
                                          else "stage2", "final", "round", "scale", "tasks"]) if kern[k][1]},
        "roofline": roof,
        "e2e": {"value": e2e_value, "unit": "TFLOP/s", "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                "ms_per_step": e2e_ms, "steps": e2e_steps,
                "step_ms": {"min": per_step[0], "median": per_step[len(per_step) // 2], "max": per_step[-1]},
                "link_gbs": {"h2d": h2d / (h2d_ms * 1e-3) / 1e9, "d2h": d2h / (d2h_ms * 1e-3) / 1e9,
                             "probes": LINK_PROBES, "of": "median per direction"},
                "pipelined": "two device copies; step q+1's upload and product overlap step q's copy back",
                "expected_ms": max(h2d_ms, ms_step, d2h_ms),
                "expected_serial_ms": h2d_ms + ms_step + d2h_ms,
                "result_check": "65536 sampled elements of the host C equal the last step's device C: "
                                + ("yes" if e2e_check else "NO"),
                "host_buffers": (f"pinned, allocated on CPUs {numa.cpus[0]}-{numa.cpus[-1]} local to the GPU"
                                 if numa.cpus else "pinned, default placement (GPU-local CPUs unknown)")},
        "clocks": clk.summary(),
        "gpu_launches": int(sum(v[1] for v in kern.values())),
        "device_status": g.tlr_status_string(status),
    }
    if main_workload and args.scale_down == 1 and args.order == "auto":
        # the per-rectangle plan of the same product, which the default gives up here
        other = time_other_plan(g, h, dp, "per_rect", max(20, args.steps // 5), stream)
        other["executed_tflops_frac_of_burst"] = other["executed_tflops"] / peak_burst
        other["note"] = "same buffers and workspace budget; more executed FLOPs, more time"
        line["other_plans"] = {"per_rect": other}
    if main_workload and args.scale_down == 1 and world == 1 and not args.no_per_config:
        line["per_config"] = per_config_timings(h, stream, local, peaks)
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"], _, _ = cpu_baseline(p, flops_step)
    dp.close()
    g.tlr_destroy(h)
    if rank == 0:
        print(json.dumps(line), flush=True)
    if dist is not None:
        dist.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())
