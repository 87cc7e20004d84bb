#!/usr/bin/env python3
"""MaxSim scoring benchmark on GB300.

Default workload (one JSON line on rank 0): ColBERTv2-shaped inference
scoring, Q[32,128] against D[100000,128,128] bf16 (L2-normalised Gaussian
tokens, full-length documents), one maxsim_score call per step. The inputs
(3.28 GB of documents) are larger than the 129 MB L2, so no flush is needed
between steps.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                    [--workload NAME] [--dtype bf16|fp16|fp32] [--B B] [--d D] [--nd ND]

Under torchrun (N > 1) every rank scores its own B documents (weak scaling;
documents are independent, so there is no data-path collective); timing is
bracketed by a barrier and a device synchronise and the max over ranks is
reported. ``--impl reference`` times the fp64 CPU oracle on the host cores on
a bounded sample of the same workload (rank 0 only).
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402
import torch  # noqa: E402

METRIC = "docs/s and HBM GB/s (% of GB300 peak) at Nq=32, Nd=128, d=128, B=100K bf16"
FALLBACK_HBM_GBS = 6800.0
FALLBACK_BF16_TFLOPS = 1900.0
_ELEM = {"bf16": 2, "fp16": 2, "fp32": 4}


# ------------------------------------------------------------------ peaks

def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            p = json.load(f)
        return {"hbm_gbs": float(p["hbm_gbs"]), "bf16_tflops": float(p["bf16_tflops"]),
                "bf16_tflops_sustained": float(p.get("bf16_tflops_sustained", p["bf16_tflops"])),
                "source": "measured"}
    except Exception:
        return {"hbm_gbs": FALLBACK_HBM_GBS, "bf16_tflops": FALLBACK_BF16_TFLOPS,
                "bf16_tflops_sustained": 1700.0, "source": "fallback"}


def kernel_source_hash(files):
    h = hashlib.sha256()
    for f in files:
        with open(os.path.join(ROOT, "maxsim_scoring_02_gb300", "csrc", f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def recorded_traffic(kernel, src_hash, workload):
    """DRAM bytes per launch from a committed ncu summary, if it was taken on
    the current kernel source; else None."""
    try:
        with open(os.path.join(ROOT, "profiles", "traffic.json")) as f:
            rec = json.load(f)
        e = rec.get(kernel, {}).get(workload)
        if e and e.get("source_hash") == src_hash:
            return float(e["dram_bytes_per_launch"])
    except Exception:
        pass
    return None


# ----------------------------------------------------------------- clocks

class ClockSampler:
    """nvidia-smi clocks / throttle reasons sampled every 100 ms while active."""
    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        self.index = index
        self.samples = []
        self.proc = None
        self.active = False
        self._thr = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None
            return
        self._thr = threading.Thread(target=self._read, daemon=True)
        self._thr.start()

    def _read(self):
        for line in self.proc.stdout:
            if self.active:
                self.samples.append([x.strip() for x in line.split(",")])

    def stop(self):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()

    def summary(self):
        if not self.samples:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples in timed region"], "samples": 0}
        sm = [float(s[0]) for s in self.samples if s[0].replace(".", "").isdigit()]
        mx = [float(s[1]) for s in self.samples if s[1].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = set()
        for s in self.samples:
            for n, v in zip(names, s[4:8]):
                if v.lower() == "active":
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": sorted(reasons), "samples": len(self.samples)}


# -------------------------------------------------------------- workloads

class Headline:
    """Padded documents, optional length mask: configs 'colbert_*' and the d/Nd sweep."""
    kernel = "fwd_tc"
    kernel_files = ("fwd_tc.cu", "ptx.cuh")

    def __init__(self, args, device, rank):
        import maxsim_scoring_02_gb300 as m
        import workloads as w
        self.m = m
        self.dtype = args.dtype
        self.B, self.nd, self.d, self.nq = args.B, args.nd, args.d, 32
        self.lenmask = args.workload == "colbert_lenmask"
        seed = 1000 * rank
        self.Q = w.normalized_tokens((self.nq, self.d), seed=seed, dtype=self.dtype, device=device)
        self.D = w.normalized_tokens((self.B, self.nd, self.d), seed=seed + 1, dtype=self.dtype, device=device)
        self.L = None
        if self.lenmask:
            self.L = w.uniform_lengths(self.B, 32, self.nd, seed=seed + 2, device=device)
            w.zero_padding(self.D, self.L)
        self.out = torch.empty((1, self.B), dtype=torch.float32, device=device)
        if self.dtype == "fp32":
            self.kernel, self.kernel_files = "fwd_f32", ("fwd_f32.cu",)
        esz = _ELEM[self.dtype]
        tok = float(self.L.sum().item()) if self.L is not None else float(self.B * self.nd)
        # algorithmic bytes per launch: every real document token once, the query, one fp32 score per doc
        self.bytes_per_launch = tok * self.d * esz + self.nq * self.d * esz + self.B * 4
        self.flops_per_launch = 2.0 * self.nq * tok * self.d
        self.units = self.B
        self.launches_per_step = 1
        self.bound = "hbm"
        self.workload = (f"colbert_{'lenmask' if self.lenmask else 'full'}_q{self.nq}_nd{self.nd}_d{self.d}"
                         f"_B{self.B}_{self.dtype}")
        self.config = {"workload": self.workload, "Nq": self.nq, "Nd": self.nd, "d": self.d, "B": self.B,
                       "doc_lengths": "U{32..%d} zero-padded, masked" % self.nd if self.lenmask else "full",
                       "inputs": "L2-normalised N(0,1) tokens, seeded",
                       "l2": "inputs (%.2f GB) larger than L2 (129 MB); no flush" % (self.D.numel() * esz / 1e9)}

    def step(self):
        self.m.maxsim_score(self.Q, self.D, self.L, out=self.out)

    # end-to-end: host (pinned) -> device copy of the step's inputs, the call, result back
    def e2e_setup(self):
        self.hQ = self.Q.cpu().pin_memory()
        self.hD = self.D.cpu().pin_memory()
        self.hL = self.L.cpu().pin_memory() if self.L is not None else None
        self.hout = torch.empty((1, self.B), dtype=torch.float32).pin_memory()
        self.h2d = self.hQ.numel() * self.hQ.element_size() + self.hD.numel() * self.hD.element_size() + (
            self.hL.numel() * 4 if self.hL is not None else 0)
        self.d2h = self.B * 4

    def e2e_step(self):
        self.Q.copy_(self.hQ, non_blocking=True)
        self.D.copy_(self.hD, non_blocking=True)
        if self.hL is not None:
            self.L.copy_(self.hL, non_blocking=True)
        self.m.maxsim_score(self.Q, self.D, self.L, out=self.out)
        self.hout.copy_(self.out, non_blocking=True)

    def cpu_sample(self, n):
        n = min(n, self.B)
        Qn = self.Q.cpu().double().numpy()
        Dn = self.D[:n].cpu().double().numpy()
        Ln = self.L[:n].cpu().numpy() if self.L is not None else None
        return (lambda: __import__("oracle").maxsim(Qn, Dn, Ln)), n


WORKLOADS = {"colbert_full": Headline, "colbert_lenmask": Headline}


# ------------------------------------------------------------------- main

def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=300)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default="colbert_full", choices=sorted(WORKLOADS))
    ap.add_argument("--dtype", default="bf16", choices=["bf16", "fp16", "fp32"])
    ap.add_argument("--B", type=int, default=100_000)
    ap.add_argument("--nd", type=int, default=128)
    ap.add_argument("--d", type=int, default=128)
    ap.add_argument("--e2e-steps", type=int, default=5)
    ap.add_argument("--cpu-seconds", type=float, default=10.0)
    ap.add_argument("--no-cpu", action="store_true")
    return ap.parse_args()


def dist_setup(args):
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        torch.cuda.set_device(local) if args.impl == "ours" else None
        import torch.distributed as dist
        dist.init_process_group("nccl" if args.impl == "ours" else "gloo")
    return world, rank, local


def cpu_baseline(wl, seconds):
    import oracle
    fn, n = wl.cpu_sample(2000 if wl.nd * wl.d <= 128 * 128 else 500)
    cores = oracle.num_threads()
    fn()                                  # warm (page-in, thread pool)
    t0 = time.perf_counter()
    reps = 0
    while True:
        fn()
        reps += 1
        el = time.perf_counter() - t0
        if el >= seconds:
            break
    return {"value": reps * n / el, "unit": "docs/s", "cores": cores, "kind": "oracle",
            "sample": f"{n} documents of the same workload (fp64 oracle, OpenMP over documents), "
                      f"{reps} passes in {el:.1f} s", "cpu": _cpu_model()}


def _cpu_model():
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True).stdout
        for line in out.splitlines():
            if line.startswith("Model name"):
                return line.split(":", 1)[1].strip()
    except Exception:
        pass
    return "unknown"


def run_reference(args, world, rank):
    """The oracle on the host cores, on the same config, steps of a bounded sample."""
    if rank != 0:
        return
    import copy

    import oracle
    n = 1000 if args.nd * args.d <= 128 * 128 else 250
    sargs = copy.copy(args)
    sargs.B = min(args.B, n)          # the sample is drawn on the host; no GPU work in this arm
    wl = WORKLOADS[args.workload](sargs, "cpu", 0)
    wl.config = dict(wl.config, B=args.B, workload=wl.workload.replace(f"_B{sargs.B}_", f"_B{args.B}_"))
    fn, n = wl.cpu_sample(n)
    for _ in range(max(args.warmup, 1)):
        fn()
    t0 = time.perf_counter()
    for _ in range(args.steps):
        fn()
    el = time.perf_counter() - t0
    v = args.steps * n / el
    line = {"metric": METRIC, "value": v, "unit": "docs/s", "n_gpus": args.gpus, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": 1e3 * el / args.steps, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic", "impl": "reference",
            "config": wl.config,
            "cpu_baseline": {"value": v, "unit": "docs/s", "cores": oracle.num_threads(), "kind": "oracle",
                             "sample": f"{n} documents per step (fp64 oracle)", "cpu": _cpu_model()},
            "e2e": {"value": v, "unit": "docs/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def main():
    args = parse()
    world, rank, local = dist_setup(args)
    if args.impl == "reference":
        # spawn-safe: the oracle runs in this process on the host cores only
        run_reference(args, world, rank)
        return
    import maxsim_scoring_02_gb300 as m
    m.load_library()
    device = torch.device("cuda", local)
    torch.cuda.set_device(device)
    peaks = load_peaks()
    wl = WORKLOADS[args.workload](args, device, rank)
    stream = torch.cuda.current_stream()

    def barrier():
        if world > 1:
            import torch.distributed as dist
            dist.barrier()
        torch.cuda.synchronize()

    for _ in range(args.warmup):
        wl.step()
    barrier()
    st, flags = m.maxsim_device_status()
    if st != 0:
        raise SystemExit(f"device status after warm-up: {st} flags {flags}")

    clocks = ClockSampler(local)
    clocks.start()
    time.sleep(0.3)
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
    barrier()
    clocks.active = True
    t_start = torch.cuda.Event(enable_timing=True)
    t_end = torch.cuda.Event(enable_timing=True)
    t_start.record(stream)
    for i in range(args.steps):
        ev[i][0].record(stream)
        wl.step()
        ev[i][1].record(stream)
    t_end.record(stream)
    barrier()
    time.sleep(0.25)
    clocks.active = False
    clocks.stop()
    elapsed_ms = t_start.elapsed_time(t_end)
    per_launch_ms = [a.elapsed_time(b) for a, b in ev]
    kernel_ms = sum(per_launch_ms) / len(per_launch_ms) / wl.launches_per_step
    if world > 1:
        import torch.distributed as dist
        t = torch.tensor([elapsed_ms], device=device)
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
        elapsed_ms = float(t.item())
    st, flags = m.maxsim_device_status()
    if st != 0:
        raise SystemExit(f"device status after timed region: {st} flags {flags}")

    units_total = wl.units * args.steps * world
    value = units_total / (elapsed_ms / 1e3)

    # roofline of the dominant kernel
    if wl.bound == "hbm":
        achieved = wl.bytes_per_launch / (kernel_ms / 1e3) / 1e9
        peak, unit = peaks["hbm_gbs"], "GB/s"
    else:
        achieved = wl.flops_per_launch / (kernel_ms / 1e3) / 1e12
        peak, unit = peaks["bf16_tflops"], "TFLOP/s"
    src_hash = kernel_source_hash(wl.kernel_files)
    traffic = recorded_traffic(wl.kernel, src_hash, wl.workload)

    # end to end through the public API with host buffers
    e2e = None
    if args.e2e_steps > 0:
        wl.e2e_setup()
        wl.e2e_step()
        barrier()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        for _ in range(args.e2e_steps):
            wl.e2e_step()
        b.record(stream)
        barrier()
        e_ms = a.elapsed_time(b)
        if world > 1:
            import torch.distributed as dist
            t = torch.tensor([e_ms], device=device)
            dist.all_reduce(t, op=dist.ReduceOp.MAX)
            e_ms = float(t.item())
        e2e = {"value": wl.units * args.e2e_steps * world / (e_ms / 1e3), "unit": "docs/s",
               "h2d_bytes_per_step": int(wl.h2d), "d2h_bytes_per_step": int(wl.d2h),
               "ms_per_step": e_ms / args.e2e_steps}

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu:
        cpu = cpu_baseline(wl, args.cpu_seconds)

    if rank == 0:
        hbm_gbs = wl.bytes_per_launch / (kernel_ms / 1e3) / 1e9
        line = {
            "metric": METRIC, "value": value, "unit": "docs/s", "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": elapsed_ms / args.steps, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": wl.dtype, "data": "synthetic",
            "config": wl.config,
            "hbm_gbs": hbm_gbs, "hbm_frac_of_measured_peak": hbm_gbs / peaks["hbm_gbs"],
            "roofline": {"bound": wl.bound, "achieved": achieved, "peak": peak, "unit": unit,
                         "frac": achieved / peak, "traffic": traffic, "kernel": wl.kernel,
                         "peak_source": peaks["source"],
                         "algorithmic_bytes_per_launch": wl.bytes_per_launch,
                         "kernel_ms": kernel_ms},
            "cpu_baseline": cpu, "e2e": e2e, "clocks": clocks.summary(),
            "gpu_launches": wl.launches_per_step * args.steps,
        }
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
