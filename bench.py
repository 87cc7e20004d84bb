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
import re
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
L2_BYTES = 129 * 1024 * 1024
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


def smem_peak_gbs(device):
    """Shared-memory load peak: one 128-byte wavefront per SM per clock."""
    sms = torch.cuda.get_device_properties(device).multi_processor_count
    mhz = 2070.0
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            mhz = float(json.load(f).get("sm_max_mhz", mhz))
    except Exception:
        pass
    return sms * 128 * mhz * 1e6 / 1e9


def ffma_peak_tflops(device):
    """FP32 FMA peak from unit counts and clock: 128 FP32 lanes per SM x 2 FLOP
    x SMs x maximum SM clock (80.5 TFLOP/s on a 152-SM part at 2070 MHz)."""
    sms = torch.cuda.get_device_properties(device).multi_processor_count
    mhz = 2070.0
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            mhz = float(json.load(f).get("sm_max_mhz", mhz))
    except Exception:
        pass
    return sms * 128 * 2 * mhz * 1e6 / 1e12


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
    kernel_files = ("fwd_tc.cu", "fwd_common.cuh", "ptx.cuh")

    def __init__(self, args, device, rank):
        import maxsim_scoring_02_gb300 as m
        import workloads as w
        self.m = m
        self.dtype = args.dtype
        self.B, self.nd, self.d, self.nq = args.B, args.nd, args.d, 32
        self.lenmask = args.workload == "colbert_lenmask"
        seed = rank_seed(rank)
        self.Q = w.normalized_tokens((self.nq, self.d), seed=seed, dtype=self.dtype, device=device)
        self.D = w.normalized_tokens((self.B, self.nd, self.d), seed=seed + 1, dtype=self.dtype, device=device)
        self.L = None
        if self.lenmask:
            self.L = w.uniform_lengths(self.B, 32, self.nd, seed=seed + 2, device=device)
            w.zero_padding(self.D, self.L)
        self.out = torch.empty((1, self.B), dtype=torch.float32, device=device)
        self.order = None
        if getattr(args, "order", "index") == "length" and torch.device(device).type == "cuda":
            # length-bucketed walk: depends only on the lengths, computed once per corpus (not timed per step)
            L = self.L if self.L is not None else torch.full((self.B,), self.nd, dtype=torch.int32, device=device)
            t0 = time.perf_counter()
            self.order = m.maxsim_length_order(doc_len=L, nd=self.nd)
            torch.cuda.synchronize()
            self.order_ms = 1e3 * (time.perf_counter() - t0)
        self.bound = "hbm"
        if self.dtype == "fp32":
            if self.d % 64 == 0 and self.nq <= 64 and (self.d // 64) * 3 * (32 if self.nq <= 32 else 64) * 128 <= 48 * 1024:
                # tensor cores on three bf16 parts of each fp32 value: each fp32 byte read once, HBM-bound
                self.kernel, self.kernel_files = "fwd_x3", ("fwd_x3.cu", "fwd_common.cuh", "ptx.cuh")
            else:
                # FFMA: 16 FLOP per document byte against a ~12 FLOP/B FP32 ridge, the FMA pipe bounds it
                self.kernel, self.kernel_files = "fwd_f32", ("fwd_f32.cu", "ptx.cuh")
                self.bound, self.alu_unit = "alu", "ffma"
        esz = _ELEM[self.dtype]
        tok = float(self.L.sum().item()) if self.L is not None else float(self.B * self.nd)
        # algorithmic bytes per launch: every real document token once, the query, one fp32 score per doc
        self.bytes_per_launch = tok * self.d * esz + self.nq * self.d * esz + self.B * 4
        self.flops_per_launch = 2.0 * self.nq * tok * self.d
        self.units = self.B
        self.launches_per_step = 1
        self.workload = (f"colbert_{'lenmask' if self.lenmask else 'full'}_q{self.nq}_nd{self.nd}_d{self.d}"
                         f"_B{self.B}_{self.dtype}")
        self.config = {"workload": self.workload, "Nq": self.nq, "Nd": self.nd, "d": self.d, "B": self.B,
                       "doc_lengths": "U{32..%d} zero-padded, masked" % self.nd if self.lenmask else "full",
                       "inputs": "L2-normalised N(0,1) tokens, seeded",
                       "l2": "inputs (%.2f GB) larger than L2 (129 MB); no flush" % (self.D.numel() * esz / 1e9)}
        if self.order is not None:
            self.workload += "_length_ordered"
            self.config.update(workload=self.workload,
                               doc_order="length-bucketed (maxsim_length_order once per corpus: %.2f ms host-timed, "
                                         "outside the timed steps)" % self.order_ms)

    def step(self, ev=None):
        if ev is not None:
            ev[0].record()
        if self.order is not None:
            self.m.maxsim_score_ordered(self.Q, self.D, self.order, self.L, out=self.out)
        else:
            self.m.maxsim_score(self.Q, self.D, self.L, out=self.out)
        if ev is not None:
            ev[1].record()

    # end-to-end: the documents stay in pinned host memory and are scored
    # through maxsim_score_streamed (chunked host -> device copies overlapped
    # with scoring); the query is copied in and the scores back every step
    E2E_CHUNK = 16384

    def e2e_setup(self):
        self.hQ = self.Q.cpu().pin_memory()
        self.hD = self.D.cpu().pin_memory()
        self.hL = self.L.cpu().pin_memory() if self.L is not None else None
        self.hout = torch.empty((1, self.B), dtype=torch.float32).pin_memory()
        nb = self.m.maxsim_score_streamed_workspace_size(1, self.nq, self.nd, self.d, self.Q.dtype, self.E2E_CHUNK)
        self.ws = torch.empty(nb, dtype=torch.uint8, device=self.Q.device)
        self.h2d = self.hQ.numel() * self.hQ.element_size() + self.hD.numel() * self.hD.element_size() + (
            self.hL.numel() * 4 if self.hL is not None else 0)
        self.d2h = self.B * 4

    def e2e_step(self):
        self.Q.copy_(self.hQ, non_blocking=True)
        self.m.maxsim_score_streamed(self.Q, self.hD, self.hL, chunk_docs=self.E2E_CHUNK, out=self.out,
                                     workspace=self.ws)
        self.hout.copy_(self.out, non_blocking=True)

    def cpu_sample(self, n):
        n = min(n, self.B)
        Qn = self.Q.cpu().double().numpy()
        Dn = self.D[:n].cpu().double().numpy()
        Ln = self.L[:n].cpu().numpy() if self.L is not None else None
        return (lambda: __import__("oracle").maxsim(Qn, Dn, Ln)), n


def _lognormal_csr(w, B, seed, device):
    """Lengths round(exp(N(ln 70, 0.5^2))) clipped to [8, 256] and CSR offsets."""
    L = w.lognormal_lengths(B, math.log(70), 0.5, 8, 256, seed=seed, device=device)
    return L, w.csr_offsets(L)


class Varlen:
    """Padding-free CSR documents, bf16 (B=500000 by default)."""
    kernel = "fwd_tc"
    kernel_files = ("fwd_tc.cu", "fwd_common.cuh", "ptx.cuh")
    bound = "hbm"

    default_B = 500_000    # documents when --B is left at its default

    def __init__(self, args, device, rank):
        import maxsim_scoring_02_gb300 as m
        import workloads as w
        self.m, self.dtype, self.d, self.nq = m, args.dtype, args.d, 32
        self.B = args.B if args.B != 100_000 else self.default_B
        seed = rank_seed(rank) + 50
        self.L, self.off = _lognormal_csr(w, self.B, seed, device)
        self.T = int(self.off[-1].item())
        self.Q = w.normalized_tokens((self.nq, self.d), seed=seed + 1, dtype=self.dtype, device=device)
        self.D = w.normalized_tokens((self.T, self.d), seed=seed + 2, dtype=self.dtype, device=device)
        self.out = torch.empty((1, self.B), dtype=torch.float32, device=device)
        esz = _ELEM[self.dtype]
        self.bytes_per_launch = self.T * self.d * esz + 8 * (self.B + 1) + self.nq * self.d * esz + 4 * self.B
        self.flops_per_launch = 2.0 * self.nq * self.T * self.d
        self.units, self.launches_per_step = self.B, 1
        self.workload = f"varlen_csr_q{self.nq}_d{self.d}_B{self.B}_{self.dtype}"
        self.config = {"workload": self.workload, "Nq": self.nq, "d": self.d, "B": self.B, "tokens": self.T,
                       "doc_lengths": "round(lognormal(ln 70, 0.5)) clipped to [8, 256], CSR-packed",
                       "inputs": "L2-normalised N(0,1) tokens, seeded",
                       "l2": "inputs (%.2f GB) larger than L2; no flush" % (self.T * self.d * esz / 1e9)}

    def step(self, ev=None):
        if ev is not None:
            ev[0].record()
        self.m.maxsim_score_varlen(self.Q, self.D, self.off, out=self.out)
        if ev is not None:
            ev[1].record()

    def e2e_setup(self):
        self.h = [t.cpu().pin_memory() for t in (self.Q, self.D, self.off)]
        self.hout = torch.empty_like(self.out, device="cpu").pin_memory()
        self.h2d = sum(t.numel() * t.element_size() for t in self.h)
        self.d2h = self.B * 4

    def e2e_step(self):
        for dst, src in zip((self.Q, self.D, self.off), self.h):
            dst.copy_(src, non_blocking=True)
        self.m.maxsim_score_varlen(self.Q, self.D, self.off, out=self.out)
        self.hout.copy_(self.out, non_blocking=True)

    def cpu_sample(self, n):
        n = min(n, self.B)
        off = self.off[:n + 1].cpu().numpy()
        Qn = self.Q.cpu().double().numpy()
        Dn = self.D[:int(off[-1])].cpu().double().numpy()
        return (lambda: __import__("oracle").maxsim_varlen(Qn, Dn, off)), n


class PQ:
    """Fused PQ scoring: M=16 subspaces x 8 dims, K=256 centroids, uint8 codes."""
    kernel = "pq_score"
    kernel_files = ("pq.cu", "ptx.cuh")
    bound = "alu"

    default_B = 500_000    # documents when --B is left at its default

    def __init__(self, args, device, rank):
        import maxsim_scoring_02_gb300 as m
        import workloads as w
        self.m, self.dtype, self.d, self.nq, self.M, self.K = m, "fp32", 128, 32, 16, 256
        self.B = args.B if args.B != 100_000 else self.default_B
        seed = rank_seed(rank) + 60
        self.L, self.off = _lognormal_csr(w, self.B, seed, device)
        self.T = int(self.off[-1].item())
        self.C, self.codes = w.pq_inputs(self.T, self.M, self.K, self.d, seed=seed + 1, device=device)
        self.Q = w.normalized_tokens((self.nq, self.d), seed=seed + 2, dtype="fp32", device=device)
        self.out = torch.empty(self.B, dtype=torch.float32, device=device)
        self.ws = torch.empty(m.maxsim_score_pq_workspace_size(self.nq, self.M, self.K) if device != "cpu" else 1,
                              dtype=torch.uint8, device=device)
        # on-chip roofline: every token reads nq * M table entries of 4 B from shared memory
        self.bytes_per_launch = 4.0 * self.nq * self.M * self.T
        self.hbm_bytes = self.T * self.M + 8 * (self.B + 1) + 4 * self.B
        self.flops_per_launch = float(self.nq * self.M * self.T)
        self.units, self.launches_per_step = self.B, 2
        self.workload = f"pq_m{self.M}_k{self.K}_q{self.nq}_d{self.d}_B{self.B}"
        self.config = {"workload": self.workload, "Nq": self.nq, "d": self.d, "M": self.M, "K": self.K,
                       "B": self.B, "tokens": self.T,
                       "doc_lengths": "round(lognormal(ln 70, 0.5)) clipped to [8, 256], CSR-packed",
                       "inputs": "C ~ N(0,1) fp32, codes uniform uint8, Q L2-normalised fp32",
                       "l2": "codes (%.2f GB) larger than L2; no flush" % (self.T * self.M / 1e9)}

    def step(self, ev=None):
        if ev is not None:
            ev[0].record()
        self.m.maxsim_score_pq(self.Q, self.C, self.codes, self.off, out=self.out, workspace=self.ws)
        if ev is not None:
            ev[1].record()

    def e2e_setup(self):
        self.h = [t.cpu().pin_memory() for t in (self.Q, self.C, self.codes, self.off)]
        self.hout = torch.empty_like(self.out, device="cpu").pin_memory()
        self.h2d = sum(t.numel() * t.element_size() for t in self.h)
        self.d2h = self.B * 4

    def e2e_step(self):
        for dst, src in zip((self.Q, self.C, self.codes, self.off), self.h):
            dst.copy_(src, non_blocking=True)
        self.m.maxsim_score_pq(self.Q, self.C, self.codes, self.off, out=self.out, workspace=self.ws)
        self.hout.copy_(self.out, non_blocking=True)

    def cpu_sample(self, n):
        import oracle
        n = min(n, self.B)
        off = self.off[:n + 1].cpu().numpy()
        Qn, Cn = self.Q.cpu().double().numpy(), self.C.cpu().double().numpy()
        cn = self.codes[:int(off[-1])].cpu().numpy()
        return (lambda: oracle.maxsim_pq(oracle.pq_table(Qn, Cn), cn, off)), n


class I8:
    """INT8 x INT8 scoring with per-token symmetric scales, d=128 (tcgen05, int8 -> fp16 on chip,
    documents on the MMA's M dimension)."""
    kernel = "fwd_i8x"
    kernel_files = ("fwd_i8x.cu", "fwd_common.cuh", "i8_common.cuh", "ptx.cuh")
    bound = "hbm"

    default_B = 500_000    # documents when --B is left at its default

    def __init__(self, args, device, rank):
        import maxsim_scoring_02_gb300 as m
        import workloads as w
        self.m, self.dtype, self.d, self.nq = m, "int8", 128, 32
        self.B = args.B if args.B != 100_000 else self.default_B
        seed = rank_seed(rank) + 70
        self.L, self.off = _lognormal_csr(w, self.B, seed, device)
        self.T = int(self.off[-1].item())
        Qf = w.normalized_tokens((self.nq, self.d), seed=seed + 1, dtype="fp32", device=device)
        self.Qi, self.sq = w.quantize_int8(Qf)
        self.Di = torch.empty((self.T, self.d), dtype=torch.int8, device=device)
        self.sd = torch.empty(self.T, dtype=torch.float32, device=device)
        step = 1 << 22
        for r0 in range(0, self.T, step):          # quantise in slices (bounded fp32 temporaries)
            r1 = min(self.T, r0 + step)
            x = w.normalized_tokens((r1 - r0, self.d), seed=seed + 2 + r0, dtype="fp32", device=device)
            self.Di[r0:r1], self.sd[r0:r1] = w.quantize_int8(x)
        self.out = torch.empty(self.B, dtype=torch.float32, device=device)
        self.bytes_per_launch = self.T * (self.d + 4) + 8 * (self.B + 1) + 4 * self.B + self.nq * (self.d + 4)
        self.flops_per_launch = 2.0 * self.nq * self.T * self.d
        self.units, self.launches_per_step = self.B, 1
        self.workload = f"i8_q{self.nq}_d{self.d}_B{self.B}"
        self.config = {"workload": self.workload, "Nq": self.nq, "d": self.d, "B": self.B, "tokens": self.T,
                       "doc_lengths": "round(lognormal(ln 70, 0.5)) clipped to [8, 256], CSR-packed",
                       "inputs": "per-token symmetric int8 of L2-normalised N(0,1) tokens + fp32 scales",
                       "l2": "inputs (%.2f GB) larger than L2; no flush" % (self.T * (self.d + 4) / 1e9)}

    def step(self, ev=None):
        if ev is not None:
            ev[0].record()
        self.m.maxsim_score_i8(self.Qi, self.sq, self.Di, self.sd, self.off, out=self.out)
        if ev is not None:
            ev[1].record()

    def e2e_setup(self):
        self.h = [t.cpu().pin_memory() for t in (self.Qi, self.sq, self.Di, self.sd, self.off)]
        self.hout = torch.empty_like(self.out, device="cpu").pin_memory()
        self.h2d = sum(t.numel() * t.element_size() for t in self.h)
        self.d2h = self.B * 4

    def e2e_step(self):
        for dst, src in zip((self.Qi, self.sq, self.Di, self.sd, self.off), self.h):
            dst.copy_(src, non_blocking=True)
        self.m.maxsim_score_i8(self.Qi, self.sq, self.Di, self.sd, self.off, out=self.out)
        self.hout.copy_(self.out, non_blocking=True)

    def cpu_sample(self, n):
        import oracle
        n = min(n, self.B)
        off = self.off[:n + 1].cpu().numpy()
        Q, sq = self.Qi.cpu().numpy(), self.sq.cpu().numpy()
        D, sd = self.Di[:int(off[-1])].cpu().numpy(), self.sd[:int(off[-1])].cpu().numpy()
        return (lambda: oracle.maxsim_i8(Q, sq, D, sd, off)), n


class ColPaliTrain:
    """Training step: forward with saved argmax, then the argmax-routed backward
    (inverse-CSR dD, destination-owned dQ). Q[16,1024,128], D[10000,1024,128] bf16."""
    kernel = "fwd_qm"
    kernel_files = ("fwd_qm.cu", "ptx.cuh")
    bound = "tensor"
    default_B = 10_000    # documents when --B is left at its default

    def __init__(self, args, device, rank):
        import maxsim_scoring_02_gb300 as m
        import workloads as w
        self.m, self.dtype, self.d = m, "bf16", 128
        self.nQ, self.nq, self.nd = 16, 1024, 1024
        self.B = args.B if args.B != 100_000 else self.default_B
        seed = rank_seed(rank) + 80
        self.Q = w.normalized_tokens((self.nQ, self.nq, self.d), seed=seed, dtype="bf16", device=device)
        self.D = w.normalized_tokens((self.B, self.nd, self.d), seed=seed + 1, dtype="bf16", device=device)
        self.dS = w.normal((self.nQ, self.B), seed=seed + 2, device=device)
        self.out = torch.empty((self.nQ, self.B), dtype=torch.float32, device=device)
        self.am = torch.empty((self.nQ, self.B, self.nq), dtype=torch.int32, device=device)
        self.dQ = torch.empty((self.nQ, self.nq, self.d), dtype=torch.float32, device=device)
        self.dD = torch.empty((self.B, self.nd, self.d), dtype=torch.float32, device=device)
        self.ws = None
        if torch.device(device).type == "cuda":
            nb = m.maxsim_backward_workspace_size(self.nQ, self.nq, self.d, self.B, self.nd)
            self.ws = torch.empty(max(nb, 16), dtype=torch.uint8, device=device)
        self.flops_per_launch = 2.0 * self.nQ * self.nq * self.B * self.nd * self.d
        self.bytes_per_launch = self.B * self.nd * self.d * 2 + 4.0 * self.nQ * self.B * self.nq
        # forward, dD, dQ and (B >= 2048) the ordered sum of the dQ document ranges
        self.units, self.launches_per_step = self.B, 4 if self.B >= 2048 else 3
        self.workload = f"colpali_train_q{self.nQ}x{self.nq}_nd{self.nd}_d{self.d}_B{self.B}_bf16"
        self.config = {"workload": self.workload, "queries": self.nQ, "Lq": self.nq, "Ld": self.nd, "d": self.d,
                       "B": self.B, "step": "forward (scores + argmax) + backward (dQ, dD)",
                       "inputs": "L2-normalised N(0,1) bf16 tokens; dS ~ N(0,1)",
                       "l2": "inputs (%.2f GB) larger than L2; no flush" % (self.B * self.nd * self.d * 2 / 1e9)}
        if torch.device(device).type == "cuda":
            torch.cuda.synchronize(device)
            torch.cuda.reset_peak_memory_stats(device)   # the footprint below counts the step, not input generation

    def step(self, ev=None):
        if ev is not None:
            ev[0].record()
        self.m.maxsim_score(self.Q, self.D, out=self.out, argmax_out=self.am)
        if ev is not None:
            ev[1].record()
            e = [torch.cuda.Event(enable_timing=True) for _ in range(3)]
            e[0].record()
        # the two halves of maxsim_backward, called separately so that each
        # kernel has its own events: dD (inverse CSR) then dQ (+ ordered range sum)
        self.m.maxsim_backward_dd(self.Q, self.am, self.dS, self.nd, dD=self.dD)
        if ev is not None:
            e[1].record()
        self.m.maxsim_backward_dq(self.D, self.am, self.dS, dQ=self.dQ, workspace=self.ws)
        self.m.allreduce_dq(self.dQ)   # sharded documents: sum the dQ partials over ranks (no-op on one rank)
        if ev is not None:
            e[2].record()
            self.bwd_events.append(e)

    bwd_events = []

    def backward_bytes(self):
        """Algorithmic HBM bytes per launch of the two backward kernels, and
        the bytes each gathers row by row from L2 (one bf16 row per argmax
        entry: Q rows for dD, D rows for dQ)."""
        am = 4.0 * self.nQ * self.B * self.nq
        ds = 4.0 * self.nQ * self.B
        dd = am + ds + 4.0 * self.B * self.nd * self.d + 2.0 * self.nQ * self.nq * self.d
        dq = am + ds + 2.0 * self.B * self.nd * self.d + 4.0 * self.nQ * self.nq * self.d
        gather = 2.0 * self.nQ * self.B * self.nq * self.d
        return {"dd_kernel": (dd, gather), "dq_kernel": (dq, gather)}

    def extra(self):
        """Backward (dD + dQ kernels) times and bytes, and the step's memory
        footprint against what a materialising implementation would add."""
        n = max(1, len(self.bwd_events))
        dd_ms = sum(e[0].elapsed_time(e[1]) for e in self.bwd_events) / n
        dq_ms = sum(e[1].elapsed_time(e[2]) for e in self.bwd_events) / n
        bb = self.backward_bytes()
        # memory footprint: this step's peak device bytes (every buffer is a torch tensor handed to the
        # library) against the similarity tensor S [nQ,B,Nq,Nd] fp32 and its gradient that a
        # materialising implementation would hold on top of the same inputs and outputs
        sim_bytes = 4.0 * self.nQ * self.B * self.nq * self.nd
        return {"backward_ms": dd_ms + dq_ms, "dd_ms": dd_ms, "dq_ms": dq_ms,
                "backward_hbm_bytes": bb["dd_kernel"][0] + bb["dq_kernel"][0],
                "backward_gbs": (bb["dd_kernel"][0] + bb["dq_kernel"][0]) / ((dd_ms + dq_ms) / 1e3) / 1e9,
                "peak_device_bytes": int(torch.cuda.max_memory_allocated()),
                "materialising_extra_bytes": {"forward": int(sim_bytes), "training": int(2 * sim_bytes)}}

    def kernel_rooflines(self, peaks):
        """HBM roofline of each backward kernel: algorithmic bytes / its own
        event time, against the measured copy bandwidth; the L2 row gathers
        are reported beside it."""
        n = max(1, len(self.bwd_events))
        times = {"dd_kernel": sum(e[0].elapsed_time(e[1]) for e in self.bwd_events) / n,
                 "dq_kernel": sum(e[1].elapsed_time(e[2]) for e in self.bwd_events) / n}
        src = kernel_source_hash(("bwd.cu", "ptx.cuh"))
        res = {}
        for k, (nbytes, gather) in self.backward_bytes().items():
            ms = times[k]
            gbs = nbytes / (ms / 1e3) / 1e9
            res[k] = {"bound": "hbm", "achieved": gbs, "peak": peaks["hbm_gbs"], "unit": "GB/s",
                      "frac": gbs / peaks["hbm_gbs"], "traffic": recorded_traffic(k, src, self.workload),
                      "peak_source": peaks["source"], "algorithmic_bytes_per_launch": nbytes, "kernel_ms": ms,
                      "l2_gather_bytes_per_launch": gather, "l2_gather_gbs": gather / (ms / 1e3) / 1e9}
        return res

    def e2e_setup(self):
        self.h = [t.cpu().pin_memory() for t in (self.Q, self.D, self.dS)]
        self.hres = [torch.empty_like(t, device="cpu").pin_memory() for t in (self.out, self.dQ)]
        self.h2d = sum(t.numel() * t.element_size() for t in self.h)
        self.d2h = sum(t.numel() * t.element_size() for t in self.hres)

    def e2e_step(self):
        for dst, src in zip((self.Q, self.D, self.dS), self.h):
            dst.copy_(src, non_blocking=True)
        self.step()
        for dst, src in zip(self.hres, (self.out, self.dQ)):
            dst.copy_(src, non_blocking=True)

    def cpu_sample(self, n):
        import oracle
        n = min(n, self.B, 1)
        Qn = self.Q.cpu().double().numpy()
        Dn = self.D[:n].cpu().double().numpy()
        dS = self.dS[:, :n].cpu().double().numpy()

        def run():
            _, a, _ = oracle.maxsim(Qn, Dn)
            oracle.backward(Qn, Dn, a, dS)
        return run, n


class Footprint:
    """Memory footprint of the fused path against a materialising one
    (FLASH-MAXSIM Abstract: memory savings; review page Fig. 2: the batch
    sizes at which materialising implementations run out of memory).

    For a sweep of ColPali-shaped batches (16 queries x 1024 tokens against B
    documents of 1024 tokens, d = 128, bf16) it measures the peak device
    bytes of the fused inference call (scores) and of the fused training step
    (scores + argmax, then dD and dQ), from torch's allocator: every buffer
    the library touches is a caller-owned torch tensor. Beside each it puts
    the bytes a materialising implementation would need on top of the same
    inputs and outputs -- the similarity tensor S[nQ,B,Lq,Ld] in fp32, and
    for training also its gradient -- and, from the device's capacity, the
    batch size at which that alone no longer fits. No materialising
    implementation is run: its extra bytes follow from the shapes."""
    kernel = "fwd_qm"
    kernel_files = ("fwd_qm.cu", "ptx.cuh")
    bound = "tensor"
    SWEEP = (1000, 2000, 5000, 10000, 20000, 40000)

    def __init__(self, args, device, rank):
        import maxsim_scoring_02_gb300 as m
        self.m, self.device = m, device
        self.nQ, self.nq, self.nd, self.d = 16, 1024, 1024, 128
        self.workload = f"footprint_colpali_q{self.nQ}x{self.nq}_nd{self.nd}_d{self.d}_bf16"

    def measure(self):
        import workloads as w
        dev = self.device
        cap = torch.cuda.get_device_properties(dev).total_memory
        rows = []
        for B in self.SWEEP:
            torch.cuda.synchronize(dev)
            torch.cuda.empty_cache()
            Q = w.normalized_tokens((self.nQ, self.nq, self.d), seed=B, dtype="bf16", device=dev)
            D = w.normalized_tokens((B, self.nd, self.d), seed=B + 1, dtype="bf16", device=dev)
            torch.cuda.synchronize(dev)
            torch.cuda.reset_peak_memory_stats(dev)
            base = torch.cuda.memory_allocated(dev)
            out = self.m.maxsim_score(Q, D)
            torch.cuda.synchronize(dev)
            inf_peak = torch.cuda.max_memory_allocated(dev)
            del out
            torch.cuda.reset_peak_memory_stats(dev)
            dS = w.normal((self.nQ, B), seed=B + 2, device=dev)
            out, am = self.m.maxsim_score(Q, D, want_argmax=True)
            dQ, dD = self.m.maxsim_backward(Q, D, am, dS)
            torch.cuda.synchronize(dev)
            st, flags = self.m.maxsim_device_status()
            if st != 0:
                raise SystemExit(f"device status in footprint sweep: {st} flags {flags}")
            train_peak = torch.cuda.max_memory_allocated(dev)
            del Q, D, dS, out, am, dQ, dD
            sim = 4 * self.nQ * B * self.nq * self.nd
            rows.append({"B": B, "inputs_bytes": int(base),
                         "fused_inference_peak_bytes": int(inf_peak), "fused_training_peak_bytes": int(train_peak),
                         "materialising_inference_bytes": int(inf_peak + sim),
                         "materialising_training_bytes": int(train_peak + 2 * sim),
                         "ratio_inference": (inf_peak + sim) / inf_peak,
                         "ratio_training": (train_peak + 2 * sim) / train_peak})
        torch.cuda.empty_cache()
        # largest batch that fits the device: fused (linear fit of the measured peaks per document)
        # against materialising (S alone, and S plus its gradient)
        per_doc_inf = (rows[-1]["fused_inference_peak_bytes"] - rows[0]["fused_inference_peak_bytes"]) / (
            rows[-1]["B"] - rows[0]["B"])
        per_doc_train = (rows[-1]["fused_training_peak_bytes"] - rows[0]["fused_training_peak_bytes"]) / (
            rows[-1]["B"] - rows[0]["B"])
        sim_per_doc = 4 * self.nQ * self.nq * self.nd
        return {"device_bytes": int(cap), "sweep": rows,
                "max_B_fused_inference": int(cap / per_doc_inf),
                "max_B_fused_training": int(cap / per_doc_train),
                "max_B_materialising_inference": int(cap / (per_doc_inf + sim_per_doc)),
                "max_B_materialising_training": int(cap / (per_doc_train + 2 * sim_per_doc))}


def run_footprint(args, device):
    wl = Footprint(args, device, 0)
    res = wl.measure()
    line = {"metric": "peak device bytes of the fused MaxSim path against a materialising one",
            "value": res["sweep"][-1]["fused_training_peak_bytes"], "unit": "bytes", "n_gpus": 1,
            "higher_is_better": False, "dtype": "bf16", "data": "synthetic",
            "config": {"workload": wl.workload, "queries": wl.nQ, "Lq": wl.nq, "Ld": wl.nd, "d": wl.d,
                       "B_sweep": list(wl.SWEEP), "value": "fused training-step peak at the largest B"},
            "footprint": res}
    print(json.dumps(line), flush=True)


WORKLOADS = {"colbert_full": Headline, "colbert_lenmask": Headline, "varlen": Varlen, "pq": PQ, "i8": I8,
             "colpali_train": ColPaliTrain, "footprint": Footprint}


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
    ap.add_argument("--order", default="index", choices=["index", "length"],
                    help="padded workloads: walk documents in index order or length-bucketed order")
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


def max_over_ranks(ms, world, device):
    """Max of a per-rank time over all ranks (identity for one rank)."""
    if world <= 1:
        return float(ms)
    import torch.distributed as dist
    t = torch.tensor([float(ms)], device=device, dtype=torch.float64)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def whole_job_rate(units_per_rank, steps, world, elapsed_ms_max):
    """Weak scaling: every rank scores its own units; rate = all units / slowest rank's time."""
    return units_per_rank * steps * world / (elapsed_ms_max / 1e3)


def rank_seed(rank):
    """Each rank draws its own documents (seeds 1000 apart)."""
    return 1000 * rank


def cpu_baseline(wl, seconds):
    import oracle
    fn, n = wl.cpu_sample(2000 if getattr(wl, "nd", 128) * wl.d <= 128 * 128 else 500)
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
    if args.workload == "footprint":
        print(json.dumps({"impl": "reference", "unavailable": "the footprint sweep measures device memory only; "
                          "the oracle arm has no device footprint"}), flush=True)
        return
    import copy

    import oracle
    n = 1000 if args.nd * args.d <= 128 * 128 else 250
    sargs = copy.copy(args)
    sargs.B = min(args.B, n)          # the sample is drawn on the host; no GPU work in this arm
    wl = WORKLOADS[args.workload](sargs, "cpu", 0)
    full_B = args.B if args.B != 100_000 else getattr(WORKLOADS[args.workload], "default_B", args.B)
    wl.config = dict(wl.config, B=full_B, workload=re.sub(r"_B%d(?=_|$)" % wl.B, "_B%d" % full_B, wl.workload),
                     l2="host run: no GPU cache involved; each step scores a sample of the workload")
    if "tokens" in wl.config:
        wl.config["sample_tokens"] = wl.config.pop("tokens")   # the sample's, not the workload's
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
    if args.workload == "footprint":
        if rank == 0:
            run_footprint(args, device)
        return
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

    # Inputs smaller than 4x L2: flush L2 between steps (a 512 MB write, outside
    # the kernel events) and compute throughput from kernel time.
    in_bytes = getattr(wl, "hbm_bytes", wl.bytes_per_launch)
    flush = torch.empty(512 << 20, dtype=torch.uint8, device=device) if in_bytes < 4 * L2_BYTES else None
    if flush is not None:
        # first touch of fresh device memory is slow (~0.2 s for 512 MB): do it before the timed region
        flush.fill_(0)
        torch.cuda.synchronize()
        wl.config = dict(wl.config, l2="inputs %.3f GB < 4 x L2: L2 flushed (512 MB write) before every step; "
                         "value from kernel time" % (in_bytes / 1e9))
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
        if flush is not None:
            flush.fill_(i & 0xFF)
        wl.step(ev[i])             # events bracket the dominant kernel's call on this stream
    t_end.record(stream)
    barrier()
    time.sleep(0.25)
    clocks.active = False
    clocks.stop()
    elapsed_ms = t_start.elapsed_time(t_end)
    per_launch_ms = [a.elapsed_time(b) for a, b in ev]
    kernel_ms = sum(per_launch_ms) / len(per_launch_ms)
    elapsed_ms = max_over_ranks(elapsed_ms, world, device)
    st, flags = m.maxsim_device_status()
    if st != 0:
        raise SystemExit(f"device status after timed region: {st} flags {flags}")

    value = whole_job_rate(wl.units, args.steps, world, elapsed_ms)
    if flush is not None:
        value = wl.units * world / (kernel_ms / 1e3)

    # roofline of the dominant kernel
    peak_source = peaks["source"]
    if wl.bound == "hbm":
        achieved = wl.bytes_per_launch / (kernel_ms / 1e3) / 1e9
        peak, unit = peaks["hbm_gbs"], "GB/s"
    elif wl.bound == "alu" and getattr(wl, "alu_unit", "") == "ffma":
        # fp32 FFMA: FLOPs against the FP32 FMA peak derived from unit counts and clock
        achieved = wl.flops_per_launch / (kernel_ms / 1e3) / 1e12
        peak, unit = ffma_peak_tflops(device), "TFLOP/s"
        peak_source = "derived: 128 FP32 lanes per SM x 2 FLOP x SMs x maximum SM clock"
    elif wl.bound == "tensor":
        # a kernel timed inside a long step: the sustained bf16 figure
        achieved = wl.flops_per_launch / (kernel_ms / 1e3) / 1e12
        peak, unit = peaks["bf16_tflops_sustained"], "TFLOP/s"
    else:
        # on-chip shared-memory bound (PQ table lookups): bytes of table reads
        # against one 128-byte wavefront per SM per clock at the maximum SM clock
        achieved = wl.bytes_per_launch / (kernel_ms / 1e3) / 1e9
        peak, unit = smem_peak_gbs(device), "GB/s"
        peak_source = "derived: one 128-byte shared-memory wavefront per SM per clock at the maximum SM clock"
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
        e_ms = max_over_ranks(a.elapsed_time(b), world, device)
        e2e = {"value": wl.units * args.e2e_steps * world / (e_ms / 1e3), "unit": "docs/s",
               "h2d_bytes_per_step": int(wl.h2d), "d2h_bytes_per_step": int(wl.d2h),
               "ms_per_step": e_ms / args.e2e_steps}

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu:
        cpu = cpu_baseline(wl, args.cpu_seconds)

    if rank == 0:
        hbm_gbs = getattr(wl, "hbm_bytes", wl.bytes_per_launch) / (kernel_ms / 1e3) / 1e9
        line = {
            "metric": METRIC, "value": value, "unit": "docs/s", "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": elapsed_ms / args.steps, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": wl.dtype, "data": "synthetic",
            "config": wl.config,
            "hbm_gbs": hbm_gbs, "hbm_frac_of_measured_peak": hbm_gbs / peaks["hbm_gbs"],
            "roofline": {"bound": wl.bound, "achieved": achieved, "peak": peak, "unit": unit,
                         "frac": achieved / peak, "traffic": traffic, "kernel": wl.kernel,
                         "peak_source": peak_source,
                         "algorithmic_bytes_per_launch": wl.bytes_per_launch,
                         "kernel_ms": kernel_ms},
            "cpu_baseline": cpu, "e2e": e2e, "clocks": clocks.summary(),
            "gpu_launches": wl.launches_per_step * args.steps,
        }
        if hasattr(wl, "kernel_rooflines"):
            line["roofline_kernels"] = dict({wl.kernel: line["roofline"]}, **wl.kernel_rooflines(peaks))
        if hasattr(wl, "extra"):
            line["extra"] = wl.extra()
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
