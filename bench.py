#!/usr/bin/env python
"""GEMM throughput on one GB300 (or N, as independent replicas), following the
benchmark method of "ThunderKittens 2.0 GPU Kernel优化" §五: bit-identical
seeded inputs, W warm-up launches, K timed back-to-back launches between two
CUDA events, input groups rotated so that every launch reads cold L2
(groups = 1 if the inputs are >= 3x L2, else floor(3 L2 / size) + 1), clocks
sampled during the run.

Headline: BF16 D = A.B^T at M=N=K=16384 (the largest point of the BF16 square
sweep), TFLOP/s = 2MNK / t.  The same JSON line carries the rest of the BF16
sweep (512 .. 8192), the MXFP8 / NVFP4 GEMMs at 4096, 8192 and 16384 (operands
quantised on the GPU by the library's own quantisers), the skinny N=K=8192 shapes,
the quantisers, a grouped GEMM and the end-to-end host-buffer GEMM, each with
its roofline fraction.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

--impl reference times the CPU oracle (the plain FP64 reference GEMM) on the
host cores on a bounded sample of the same workload.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

PAGES_PEAK_TFLOPS = {"bf16": 2250.0, "mxfp8": 4500.0, "nvfp4": 9000.0}   # HGX B200 dense figures the pages list
PAGES_HBM_GBS = 8000.0                                                     # the HBM bandwidth in the same table
NOMINAL_RATIO = {"bf16": 1.0, "mxfp8": 2.0, "nvfp4": 6.0}                 # GB300 dense fp8/fp4 vs bf16 (4.5, 13.5 vs 2.25 PF)
SEEDS = {"bf16": 1001, "mxfp8": 1002, "nvfp4": 1003}                      # 1000 + workload index
PAUSE_S = [0.0]   # idle seconds before each timed workload (set from --sleep-ms after the headline)
QUEUE_DELAY_CYCLES_PER_STEP = 100000   # ~50 us of GPU delay per queued launch (host issue takes ~15 us)


def parse_args():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=100)
    ap.add_argument("--warmup", type=int, default=500)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--size", type=int, default=16384, help="headline M=N=K")
    ap.add_argument("--formats", default="bf16,mxfp8,nvfp4")
    ap.add_argument("--sweep", default="512,2048,4096,8192", help="extra BF16 sizes reported beside the headline")
    ap.add_argument("--sweep-scaled", default="4096,8192", help="extra MXFP8 / NVFP4 sizes reported beside 16384")
    ap.add_argument("--nontile", default="4000", help="M=N=K sizes that are not tile multiples, timed in BF16 and NVFP4")
    ap.add_argument("--sustained-s", type=float, default=1.0,
                    help="seconds of back-to-back headline launches timed after the headline loop (0: skip)")
    ap.add_argument("--no-vendor-peak", action="store_true",
                    help="skip timing the vendor library's MXFP8 / NVFP4 GEMM on the 16384 operands (measured peaks)")
    ap.add_argument("--e2e-steps", type=int, default=20)
    ap.add_argument("--cpu-rows", type=int, default=768, help="rows of the oracle's CPU-baseline sample")
    ap.add_argument("--head-format", default="bf16", choices=["bf16", "mxfp8", "nvfp4"],
                    help="format of the first (timed, clock-sampled) workload; profiling runs pick it")
    ap.add_argument("--skinny", default="1,16,128,1024",
                    help="M values of the skinny N=K=8192 GEMMs reported (1: batch-1 decode)")
    ap.add_argument("--no-cpu", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-list", action="store_true", help="skip the GEMM-list timings")
    ap.add_argument("--no-quant", action="store_true", help="skip the quantiser timings")
    ap.add_argument("--grouped-decode", default="8,16,4096,7168",
                    help="experts,rows per expert,N,K of the decode-regime grouped GEMM (empty: skip)")
    ap.add_argument("--grouped", default="8,16384,4096,7168",
                    help="grouped GEMM reported beside the headline: groups,total rows,N,K ('' to skip)")
    ap.add_argument("--l2", choices=["rotate", "flush"], default="rotate")
    ap.add_argument("--sleep-ms", type=int, default=500,
                    help="idle time before each timed workload after the headline (the pages' method: 500 ms)")
    ap.add_argument("--vendor", default="",
                    help="M=N=K sizes at which the vendor library's GEMMs (cuBLAS / cuBLASLt through torch) are timed "
                         "beside this library's on the same operands, as context (empty: skip)")
    return ap.parse_args()


# --------------------------------------------------------------------------- environment

def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return {"bf16": float(d["bf16_tflops"]), "bf16_sustained": float(d.get("bf16_tflops_sustained", 0) or 0),
                "hbm_gbs": float(d["hbm_gbs"]), "source": "measured"}
    return {"bf16": 1900.0, "bf16_sustained": 1700.0, "hbm_gbs": 6800.0, "source": "fallback"}


def _code_only(src: str) -> str:
    """C++ source without comments or blank lines: what the compiler sees, so a
    comment edit leaves recorded counters valid."""
    import re
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    src = re.sub(r"//[^\n]*", "", src)
    return "\n".join(line.rstrip() for line in src.splitlines() if line.strip())


def kernel_hash():
    h = hashlib.sha256()
    for f in ("ptx.cuh", "gemm_kernel.cuh", "host_common.cuh", "gemm_bf16.cu", "gemm_mxfp8.cu", "gemm_nvfp4.cu"):
        h.update(_code_only(open(os.path.join(ROOT, "dense_block_scaled_gb300", "csrc", f)).read()).encode())
    return h.hexdigest()[:16]


def recorded_traffic(workload):
    """DRAM bytes per launch recorded from an ncu capture, if taken on the current kernel source."""
    p = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(p):
        return None
    d = json.load(open(p)).get(workload)
    if not d or d.get("kernel_hash") != kernel_hash():
        return None
    return d.get("dram_bytes_per_launch")


class ClockSampler:
    """nvidia-smi sampled every 200 ms while the GPU is busy."""

    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap,"
              "clocks.mem,temperature.gpu")

    def __init__(self, device_uuid):
        self.uuid = device_uuid
        self.proc = None
        self.out = tempfile.NamedTemporaryFile(prefix="clk", suffix=".csv", delete=False)

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", self.uuid, f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "200"], stdout=self.out, stderr=subprocess.DEVNULL)
        except (OSError, ValueError):
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.out.close()
        rows = []
        for line in open(self.out.name):
            f = [x.strip() for x in line.split(",")]
            if len(f) < 8:
                continue
            try:
                mem = float(f[8]) if len(f) > 8 else float("nan")
                temp = float(f[9]) if len(f) > 9 else float("nan")
                rows.append((float(f[0]), float(f[1]), float(f[2]), f[4:8], mem, temp))
            except ValueError:
                continue
        os.unlink(self.out.name)
        if not rows:
            return None
        loaded = [r for r in rows if r[2] > 300.0] or rows
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in loaded for i, v in enumerate(r[3]) if v.lower() == "active"})
        return {"sm_mhz": statistics.median(r[0] for r in loaded), "sm_max_mhz": max(r[1] for r in rows),
                "mem_mhz": statistics.median(r[4] for r in loaded), "temp_c_max": max(r[5] for r in rows),
                "power_w_max": max(r[2] for r in rows), "samples": len(rows), "reasons": reasons}


# --------------------------------------------------------------------------- workloads

class Workload:
    """One GEMM (format, M=N=K=size) resident in HBM in `groups` identical copies."""

    def __init__(self, fmt, size, seed, l2_bytes, torch, tkg, synth, keep_host=False, mnk=None, keep_fp32=False):
        self.fmt, self.size = fmt, size
        self.m, self.n, self.k = mnk if mnk else (size, size, size)
        m, n, k = self.m, self.n, self.k
        t0 = time.time()
        a, b = synth.gemm_inputs_f32(m, n, k, seed)
        dev = torch.device("cuda")
        self.host = None
        self.fp32 = None
        if fmt == "bf16":
            ca, cb = synth.bf16_codes(a), synth.bf16_codes(b)
            del a, b
            A = torch.from_numpy(ca.view("int16")).view(torch.bfloat16)
            B = torch.from_numpy(cb.view("int16")).view(torch.bfloat16)
            ops = [A.to(dev), B.to(dev), None, None, None, None]
            if keep_host:
                self.host = (ca, cb)
        else:
            X = torch.from_numpy(a).to(dev)
            Y = torch.from_numpy(b).to(dev)
            del a, b
            bs = 32 if fmt == "mxfp8" else 16
            cols = k if fmt == "mxfp8" else k // 2
            QA = torch.empty((m, cols), dtype=torch.uint8, device=dev)
            QB = torch.empty((n, cols), dtype=torch.uint8, device=dev)
            SA = torch.empty((tkg.scale_bytes(m, k, bs),), dtype=torch.uint8, device=dev)
            SB = torch.empty((tkg.scale_bytes(n, k, bs),), dtype=torch.uint8, device=dev)
            if fmt == "mxfp8":
                tkg.quantize_mxfp8(X, QA, SA)
                tkg.quantize_mxfp8(Y, QB, SB)
                ops = [QA, QB, SA, SB, None, None]
            else:
                TA = torch.empty(1, dtype=torch.float32, device=dev)
                TB = torch.empty(1, dtype=torch.float32, device=dev)
                tkg.quantize_nvfp4(X, QA, SA, TA)
                tkg.quantize_nvfp4(Y, QB, SB, TB)
                ops = [QA, QB, SA, SB, TA, TB]
            if keep_fp32:
                self.fp32 = X
            del X, Y
            torch.cuda.synchronize()
        self.in_bytes = sum(int(o.numel() * o.element_size()) for o in ops if o is not None)
        self.out_bytes = self.m * self.n * 2
        self.groups = 1 if self.in_bytes >= 3 * l2_bytes else (3 * l2_bytes) // self.in_bytes + 1
        self.sets = [ops] + [[o.clone() if o is not None else None for o in ops] for _ in range(self.groups - 1)]
        self.D = [torch.empty((self.m, self.n), dtype=torch.bfloat16, device=dev) for _ in range(self.groups)]
        self.flop = 2.0 * self.m * self.n * self.k
        self.prep_s = time.time() - t0

    def launch(self, i, tkg):
        A, B, sa, sb, ta, tb = self.sets[i % self.groups]
        D = self.D[i % self.groups]
        if self.fmt == "bf16":
            tkg.gemm_bf16(A, B, D, 1.0)
        elif self.fmt == "mxfp8":
            tkg.gemm_mxfp8(A, B, sa, sb, D, 1.0)
        else:
            tkg.gemm_nvfp4(A, B, sa, sb, D, 1.0, ta=ta, tb=tb)


def time_launches(w, steps, warmup, torch, tkg, dist=None, l2_mode="rotate", flush_buf=None):
    """Seconds per launch: W untimed launches, then K timed back to back between
    two events on the launching stream (or one event pair per launch around an
    explicit L2 flush when l2_mode == 'flush').  The warm-up covers at least one
    pass over the rotated input copies, so that the timed launches find every
    copy's tensor maps already encoded (the headline, whose inputs exceed 3x L2,
    has one copy)."""
    if PAUSE_S[0] > 0:
        torch.cuda.synchronize()
        time.sleep(PAUSE_S[0])
    for i in range(max(warmup, getattr(w, "groups", 1))):
        w.launch(i, tkg)
    torch.cuda.synchronize()
    if dist is not None:
        dist.barrier()
    torch.cuda.synchronize()
    if l2_mode == "flush":
        total = 0.0
        for i in range(steps):
            flush_buf.zero_()
            e0 = torch.cuda.Event(enable_timing=True)
            e1 = torch.cuda.Event(enable_timing=True)
            e0.record()
            w.launch(i, tkg)
            e1.record()
            e1.synchronize()
            total += e0.elapsed_time(e1)
        ms = total
    else:
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        # A short GPU-side delay ahead of the start event (outside the timed
        # region) lets the host enqueue all K launches before the first one runs,
        # so launches of ~10 us are timed back to back rather than at the rate
        # the host issues them; the e2e figure keeps the host's costs.
        torch.cuda._sleep(QUEUE_DELAY_CYCLES_PER_STEP * min(steps, 400))
        e0.record()
        for i in range(steps):
            w.launch(i, tkg)
        e1.record()
        e1.synchronize()
        ms = e0.elapsed_time(e1)
    torch.cuda.synchronize()
    if dist is not None:
        dist.barrier()
    st = tkg.device_status()
    if st != tkg.OK:
        raise RuntimeError(f"device status after timing: {tkg.status_string(st)}")
    return ms / 1e3 / steps


def sustained_seconds(w, seconds, t_burst, torch, tkg, uuid):
    """Seconds per launch over a back-to-back run of at least `seconds` (the
    part settles at its power cap), with the clocks sampled during it."""
    n = max(10, int(seconds / max(t_burst, 1e-6)) + 1)
    clocks = ClockSampler(uuid)
    clocks.start()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record()
    for i in range(n):
        w.launch(i, tkg)
    e1.record()
    e1.synchronize()
    clk = clocks.stop()
    st = tkg.device_status()
    if st != tkg.OK:
        raise RuntimeError(f"device status after the sustained loop: {tkg.status_string(st)}")
    ms = e0.elapsed_time(e1)
    return ms / 1e3 / n, n, ms / 1e3, clk


def quant_timings(X, steps, warmup, torch, tkg, hbm_gbs):
    """Device time of the library's quantisers on one FP32 operand (rows x k,
    larger than L2, so no flush is needed between launches).  Algorithmic bytes
    per element: MXFP8 reads 4 and writes 1 + 1/32 (codes, scales); NVFP4 makes
    two passes, the tensor amax (4 read) and the quantisation (4 read, 1/2 + 1/16
    written)."""
    rows, k = X.shape
    dev = X.device
    out = {}
    for fmt, bs, cols, bpe in (("mxfp8", 32, k, 4 + 1 + 1 / 32), ("nvfp4", 16, k // 2, 8 + 0.5 + 1 / 16)):
        Q = torch.empty((rows, cols), dtype=torch.uint8, device=dev)
        S = torch.empty((tkg.scale_bytes(rows, k, bs),), dtype=torch.uint8, device=dev)
        T = torch.empty(1, dtype=torch.float32, device=dev)
        run = (lambda: tkg.quantize_mxfp8(X, Q, S)) if fmt == "mxfp8" else (lambda: tkg.quantize_nvfp4(X, Q, S, T))
        for _ in range(warmup):
            run()
        torch.cuda.synchronize()
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record()
        for _ in range(steps):
            run()
        e1.record()
        e1.synchronize()
        t = e0.elapsed_time(e1) / 1e3 / steps
        gbs = rows * k * bpe / t / 1e9
        out[fmt] = {"us": t * 1e6, "gbs": gbs, "frac_of_hbm": gbs / hbm_gbs, "bytes_per_elem": bpe,
                    "shape": [rows, k]}
        del Q, S, T
    return out


GROUPED_SEED = 1006


def grouped_sizes(groups, total, seed=GROUPED_SEED):
    """Group row counts of the mixture-of-experts workload: `total` rows dealt
    to `groups` experts by a seeded multinomial draw, in whole 128-row blocks
    (the padded layout in which each group starts on a scale block)."""
    import numpy as np
    rng = np.random.default_rng(seed)
    return [int(x) * 128 for x in rng.multinomial(total // 128, [1.0 / groups] * groups)]


LIST_CASES = [
    # label, format, shapes: independent GEMMs (own operands each) in one tkg_gemm_list_* launch
    ("BF16 8 x 512^3", "bf16", [(512, 512, 512)] * 8),
    ("BF16 8 x M=16 N=K=8192", "bf16", [(16, 8192, 8192)] * 8),
    ("NVFP4 8 x M=16 N=K=8192", "nvfp4", [(16, 8192, 8192)] * 8),
]
LIST_SEED = 1100


class ListWorkload:
    """Several independent GEMMs (seeded N(0,1) operands each; block-scaled ones
    quantised by the library's quantisers) run as one tkg_gemm_list launch, in
    identical copies rotated so that every launch reads cold L2."""

    def __init__(self, fmt, shapes, seed, l2_bytes, torch, tkg, synth):
        self.fmt, self.shapes = fmt, shapes
        dev = torch.device("cuda")
        base = []
        for i, (m, n, k) in enumerate(shapes):
            w = Workload(fmt, 0, seed + i, 0, torch, tkg, synth, mnk=(m, n, k))   # one copy (no rotation)
            base.append(w.sets[0] + [w.D[0]])
            del w
        self.in_bytes = sum(int(o.numel() * o.element_size()) for ops in base for o in ops[:6] if o is not None)
        self.out_bytes = sum(m * n * 2 for m, n, _ in shapes)
        self.groups = 1 if self.in_bytes >= 3 * l2_bytes else (3 * l2_bytes) // self.in_bytes + 1
        self.sets = [base] + [[[o.clone() if o is not None else None for o in ops] for ops in base]
                              for _ in range(self.groups - 1)]
        self.descs = []
        for st in self.sets:
            self.descs.append([tkg.gemm_desc(fmt, A, B, D, 1.0, sfa=sa, sfb=sb, ta=ta, tb=tb)
                               for A, B, sa, sb, ta, tb, D in st])
        self.flop = sum(2.0 * m * n * k for m, n, k in shapes)
        del dev

    def launch(self, i, tkg):
        tkg.gemm_list(self.fmt, self.descs[i % self.groups])


def list_timings(steps, warmup, l2, torch, tkg, synth, hbm_gbs, single):
    """Per case: time per list launch, per GEMM, TFLOP/s and the fraction of the
    HBM roofline over all operand and output bytes; `single` gives the same
    GEMM's one-launch time where the bench measured it."""
    out = {}
    for label, fmt, shapes in LIST_CASES:
        w = ListWorkload(fmt, shapes, LIST_SEED, l2, torch, tkg, synth)
        t = time_launches(w, steps, warmup, torch, tkg)
        byts = w.in_bytes + w.out_bytes
        e = {"us_per_launch": t * 1e6, "us_per_gemm": t * 1e6 / len(shapes), "tflops": w.flop / t / 1e12,
             "gbs": byts / t / 1e9, "frac_of_hbm": byts / t / 1e9 / hbm_gbs, "gemms": len(shapes),
             "input_groups": w.groups}
        tg = graph_seconds(w, steps, torch, tkg)
        e["us_per_launch_graph"] = tg * 1e6
        e["us_per_gemm_graph"] = tg * 1e6 / len(shapes)
        e["frac_of_hbm_graph"] = byts / tg / 1e9 / hbm_gbs
        one, one_graph = single.get(label, (None, None))
        if one:
            e["single_launch_us"] = one
            e["speedup_vs_single_launches"] = one * len(shapes) / (t * 1e6)
        if one_graph:
            e["single_launch_us_graph"] = one_graph
            e["speedup_vs_single_launches_graph"] = one_graph * len(shapes) / (tg * 1e6)
        out[label] = e
        del w
        torch.cuda.empty_cache()
    return out


def grouped_timings(formats, groups, total, n, k, steps, warmup, torch, tkg, synth):
    """TFLOP/s of the grouped GEMM over `groups` experts of n x k weights.
    Inputs are seeded N(0,1); MXFP8 / NVFP4 operands come from the library's
    quantisers (A as one tensor: with 128-row groups its tiled scales are the
    per-group layout; each expert's B as its own tensor)."""
    sizes = grouped_sizes(groups, total)
    a, b = synth.gemm_inputs_f32(total, groups * n, k, GROUPED_SEED)
    dev = torch.device("cuda")
    out = {"sizes": sizes, "n": n, "k": k}
    flop = 2.0 * total * n * k
    for fmt in formats:
        D = torch.empty((total, n), dtype=torch.bfloat16, device=dev)
        if fmt == "bf16":
            A = torch.from_numpy(synth.bf16_codes(a).view("int16")).view(torch.bfloat16).to(dev)
            B = torch.from_numpy(synth.bf16_codes(b).view("int16")).view(torch.bfloat16).to(dev).view(groups, n, k)
            run = lambda: tkg.gemm_grouped_bf16(sizes, A, B, D)
        else:
            bs = 32 if fmt == "mxfp8" else 16
            cols = k if fmt == "mxfp8" else k // 2
            X = torch.from_numpy(a).to(dev)
            A = torch.empty((total, cols), dtype=torch.uint8, device=dev)
            SA = torch.empty((tkg.scale_bytes(total, k, bs),), dtype=torch.uint8, device=dev)
            B = torch.empty((groups, n, cols), dtype=torch.uint8, device=dev)
            sfb_g = tkg.scale_bytes(n, k, bs)
            SB = torch.empty((groups * sfb_g,), dtype=torch.uint8, device=dev)
            TA = torch.empty(1, dtype=torch.float32, device=dev)
            TB = torch.empty(groups, dtype=torch.float32, device=dev)
            if fmt == "mxfp8":
                tkg.quantize_mxfp8(X, A, SA)
            else:
                tkg.quantize_nvfp4(X, A, SA, TA)
            del X
            for g in range(groups):
                Y = torch.from_numpy(b[g * n:(g + 1) * n]).to(dev)
                if fmt == "mxfp8":
                    tkg.quantize_mxfp8(Y, B[g], SB[g * sfb_g:(g + 1) * sfb_g])
                else:
                    tkg.quantize_nvfp4(Y, B[g], SB[g * sfb_g:(g + 1) * sfb_g], TB[g:g + 1])
            if fmt == "mxfp8":
                run = lambda: tkg.gemm_grouped_mxfp8(sizes, A, B, SA, SB, D)
            else:
                run = lambda: tkg.gemm_grouped_nvfp4(sizes, A, B, SA, SB, D, ta=TA, tb=TB)
        if PAUSE_S[0] > 0:
            torch.cuda.synchronize()
            time.sleep(PAUSE_S[0])
        for _ in range(warmup):
            run()
        torch.cuda.synchronize()
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record()
        for _ in range(steps):
            run()
        e1.record()
        e1.synchronize()
        t = e0.elapsed_time(e1) / 1e3 / steps
        if tkg.device_status() != tkg.OK:
            raise RuntimeError("device status after grouped timing")
        out[fmt] = {"us": t * 1e6, "tflops": flop / t / 1e12,
                    "frac_of_pages_peak": flop / t / 1e12 / PAGES_PEAK_TFLOPS[fmt]}
        del A, B, D
        torch.cuda.empty_cache()
    return out


def grouped_decode_timings(groups, rows, n, k, steps, warmup, torch, tkg, synth, hbm_gbs):
    """Grouped GEMM in the decode regime of a mixture-of-experts layer: `rows`
    rows per expert, bound by reading the experts' n x k weights from HBM.
    BF16, MXFP8 and NVFP4 (each group's A rows quantised into its own 128-row
    scale block; NVFP4 with one tensor scale for all of A); reported as time and
    fraction of the HBM roofline over all bytes."""
    sizes = [rows] * groups
    total = rows * groups
    a, b = synth.gemm_inputs_f32(total, groups * n, k, GROUPED_SEED + 1)
    dev = torch.device("cuda")
    out = {"groups": groups, "rows_per_group": rows, "n": n, "k": k}
    D = torch.empty((total, n), dtype=torch.bfloat16, device=dev)

    def timed(run):
        if PAUSE_S[0] > 0:
            torch.cuda.synchronize()
            time.sleep(PAUSE_S[0])
        for _ in range(warmup):
            run()
        torch.cuda.synchronize()
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record()
        for _ in range(steps):
            run()
        e1.record()
        e1.synchronize()
        if tkg.device_status() != tkg.OK:
            raise RuntimeError("device status after grouped decode timing")
        return e0.elapsed_time(e1) / 1e3 / steps

    A = torch.from_numpy(synth.bf16_codes(a).view("int16")).view(torch.bfloat16).to(dev)
    B = torch.from_numpy(synth.bf16_codes(b).view("int16")).view(torch.bfloat16).to(dev).view(groups, n, k)
    t = timed(lambda: tkg.gemm_grouped_bf16(sizes, A, B, D))
    byts = (groups * n * k + total * k) * 2 + total * n * 2
    out["bf16"] = {"us": t * 1e6, "gbs": byts / t / 1e9, "frac_of_hbm": byts / t / 1e9 / hbm_gbs}
    # the same with the group sizes in device memory (capacity = the rows present)
    sizes_dev = torch.tensor(sizes, dtype=torch.int32, device=dev)

    def dev_sfa(sa, bs):
        buf = torch.zeros((tkg.grouped_dev_scale_bytes(groups, total, k, bs),), dtype=torch.uint8, device=dev)
        buf[:sa.numel()] = sa
        return buf

    t = timed(lambda: tkg.gemm_grouped_dev_bf16(sizes_dev, A, B, D))
    out["bf16_device_sizes"] = {"us": t * 1e6, "gbs": byts / t / 1e9, "frac_of_hbm": byts / t / 1e9 / hbm_gbs}
    del A, B
    sfb = tkg.scale_bytes(n, k, 32)
    blk = tkg.scale_bytes(128, k, 32)
    A8 = torch.empty((total, k), dtype=torch.uint8, device=dev)
    SA8 = torch.zeros((tkg.grouped_scale_bytes(sizes, k, 32),), dtype=torch.uint8, device=dev)
    B8 = torch.empty((groups, n, k), dtype=torch.uint8, device=dev)
    SB8 = torch.empty((groups * sfb,), dtype=torch.uint8, device=dev)
    X = torch.from_numpy(a).to(dev)
    for g in range(groups):
        r0 = g * rows
        tkg.quantize_mxfp8(X[r0:r0 + rows].contiguous(), A8[r0:r0 + rows],
                           SA8[g * blk * ((rows + 127) // 128):][:tkg.scale_bytes(rows, k, 32)])
        tkg.quantize_mxfp8(torch.from_numpy(b[g * n:(g + 1) * n]).to(dev), B8[g], SB8[g * sfb:(g + 1) * sfb])
    del X
    t = timed(lambda: tkg.gemm_grouped_mxfp8(sizes, A8, B8, SA8, SB8, D))
    byts = groups * (n * k + sfb) + total * k + SA8.numel() + total * n * 2
    out["mxfp8"] = {"us": t * 1e6, "gbs": byts / t / 1e9, "frac_of_hbm": byts / t / 1e9 / hbm_gbs}
    SA8d = dev_sfa(SA8, 32)
    t = timed(lambda: tkg.gemm_grouped_dev_mxfp8(sizes_dev, A8, B8, SA8d, SB8, D))
    out["mxfp8_device_sizes"] = {"us": t * 1e6, "gbs": byts / t / 1e9, "frac_of_hbm": byts / t / 1e9 / hbm_gbs}
    del SA8d
    del A8, SA8, B8, SB8
    # NVFP4: one tensor scale for all of A (the experts' rows quantised together, each group into its own
    # 128-row scale block with the scale of the whole), one per expert for B
    sfb4 = tkg.scale_bytes(n, k, 16)
    blk4 = tkg.scale_bytes(128, k, 16)
    A4 = torch.empty((total, k // 2), dtype=torch.uint8, device=dev)
    SA4 = torch.zeros((tkg.grouped_scale_bytes(sizes, k, 16),), dtype=torch.uint8, device=dev)
    B4 = torch.empty((groups, n, k // 2), dtype=torch.uint8, device=dev)
    SB4 = torch.empty((groups * sfb4,), dtype=torch.uint8, device=dev)
    TA = torch.empty(1, dtype=torch.float32, device=dev)
    TB = torch.empty(groups, dtype=torch.float32, device=dev)
    X = torch.from_numpy(a).to(dev)
    whole_q = torch.empty((total, k // 2), dtype=torch.uint8, device=dev)
    whole_s = torch.empty((tkg.scale_bytes(total, k, 16),), dtype=torch.uint8, device=dev)
    tkg.quantize_nvfp4(X, whole_q, whole_s, TA)             # the tensor scale of all of A
    for g in range(groups):
        r0 = g * rows
        tkg.quantize_nvfp4_scaled(X[r0:r0 + rows], A4[r0:r0 + rows],
                                  SA4[g * blk4 * ((rows + 127) // 128):][:tkg.scale_bytes(rows, k, 16)], TA)
        tkg.quantize_nvfp4(torch.from_numpy(b[g * n:(g + 1) * n]).to(dev), B4[g], SB4[g * sfb4:(g + 1) * sfb4],
                           TB[g:g + 1])
    del X, whole_q, whole_s
    t = timed(lambda: tkg.gemm_grouped_nvfp4(sizes, A4, B4, SA4, SB4, D, ta=TA, tb=TB))
    byts = groups * (n * k // 2 + sfb4) + total * k // 2 + SA4.numel() + total * n * 2
    out["nvfp4"] = {"us": t * 1e6, "gbs": byts / t / 1e9, "frac_of_hbm": byts / t / 1e9 / hbm_gbs}
    SA4d = dev_sfa(SA4, 16)
    t = timed(lambda: tkg.gemm_grouped_dev_nvfp4(sizes_dev, A4, B4, SA4d, SB4, D, ta=TA, tb=TB))
    out["nvfp4_device_sizes"] = {"us": t * 1e6, "gbs": byts / t / 1e9, "frac_of_hbm": byts / t / 1e9 / hbm_gbs}
    del SA4d
    del A4, SA4, B4, SB4, TA, TB, D
    torch.cuda.empty_cache()
    return out


class VendorGemm:
    """The vendor library's GEMM on a Workload's resident operands (torch.mm for BF16, torch._scaled_mm
    for MXFP8 and NVFP4, which read the same tiled scale layout), launched like Workload.launch.  Context
    only: the headline and every other number on the line come from this library's kernels."""

    def __init__(self, w, torch):
        self.w, self.torch = w, torch
        self.groups, self.flop = w.groups, w.flop

    def launch(self, i, _tkg):
        torch, w = self.torch, self.w
        A, B, sa, sb, _, _ = w.sets[i % w.groups]
        D = w.D[i % w.groups]
        if w.fmt == "bf16":
            torch.mm(A, B.t(), out=D)
        elif w.fmt == "mxfp8":
            torch._scaled_mm(A.view(torch.float8_e4m3fn), B.view(torch.float8_e4m3fn).t(),
                             scale_a=sa.view(torch.float8_e8m0fnu), scale_b=sb.view(torch.float8_e8m0fnu),
                             out_dtype=torch.bfloat16, out=D)
        else:
            # per-tensor scales left out: alpha does not change the work
            torch._scaled_mm(A.view(torch.float4_e2m1fn_x2), B.view(torch.float4_e2m1fn_x2).t(),
                             scale_a=sa.view(torch.float8_e4m3fn), scale_b=sb.view(torch.float8_e4m3fn),
                             out_dtype=torch.bfloat16, out=D)


def vendor_timings(formats, sizes, steps, warmup, l2, torch, tkg, synth, l2_mode, flush_buf):
    """Per format and size: this library's GEMM and the vendor library's on the same operands, timed the
    same way (ours, vendor, ours again), and how many outputs of the two differ by more than BF16 rounding."""
    out = {}
    for fmt in formats:
        for s in sizes:
            key = f"{fmt} {s}"
            try:
                w = Workload(fmt, s, SEEDS[fmt], l2, torch, tkg, synth)
                v = VendorGemm(w, torch)
                w.launch(0, tkg)
                ours = w.D[0].float().clone()
                v.launch(0, tkg)
                theirs = w.D[0].float()
                if fmt == "nvfp4":
                    theirs = theirs * (w.sets[0][4] * w.sets[0][5])
                # outside the band one BF16 rounding step wide around ours (relative, plus the same of the
                # mean magnitude for outputs near zero): different summation orders stay inside it
                band = 2.0 ** -7 * (ours.abs() + ours.abs().mean())
                outside = int(((ours - theirs).abs() > band).sum())
                t0 = time_launches(w, steps, warmup, torch, tkg, None, l2_mode, flush_buf)
                tv = time_launches(v, steps, warmup, torch, tkg, None, l2_mode, flush_buf)
                t1 = time_launches(w, steps, min(warmup, 100), torch, tkg, None, l2_mode, flush_buf)
                out[key] = {"ours_tflops": w.flop / t0 / 1e12, "vendor_tflops": w.flop / tv / 1e12,
                            "ours_again_tflops": w.flop / t1 / 1e12, "input_groups": w.groups,
                            "outputs_outside_bf16_band": outside, "outputs": int(ours.numel())}
                del w, v, ours, theirs
                torch.cuda.empty_cache()
            except Exception as e:   # a vendor build without the format: reported, not fatal
                out[key] = {"error": repr(e)[:300]}
    return out


def graph_seconds(w, steps, torch, tkg):
    """Seconds per launch when the K launches are replayed from one captured CUDA
    graph: the same kernels without the per-call host work."""
    w.launch(0, tkg)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        for i in range(steps):
            w.launch(i, tkg)
    g.replay()
    torch.cuda.synchronize()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record()
    g.replay()
    e1.record()
    e1.synchronize()
    st = tkg.device_status()
    if st != tkg.OK:
        raise RuntimeError(f"device status after graph replay: {tkg.status_string(st)}")
    return e0.elapsed_time(e1) / 1e3 / steps


def e2e_seconds(w, steps, torch, tkg):
    """Per-step seconds through the public API with HOST buffers: every step
    copies its inputs from pinned host memory to the device and its output
    back, inside the timed region.  BF16 goes through tkg_gemm_bf16_from_host,
    which overlaps those copies with the GEMM; the block-scaled formats copy
    with torch and call the device GEMM."""
    A, B, sa, sb, ta, tb = w.sets[0]
    dev_ops = [A, B, sa, sb, ta, tb]
    host = [o.cpu().pin_memory() if o is not None else None for o in dev_ops]
    Dh = torch.empty((w.m, w.n), dtype=torch.bfloat16).pin_memory()
    h2d = sum(int(h.numel() * h.element_size()) for h in host if h is not None)
    d2h = int(Dh.numel() * Dh.element_size())

    def step():
        if w.fmt == "bf16":
            tkg.gemm_bf16_from_host(host[0], host[1], Dh, A, B, w.D[0])
            return
        for h, d in zip(host, dev_ops):
            if h is not None:
                d.copy_(h, non_blocking=True)
        w.launch(0, tkg)
        Dh.copy_(w.D[0], non_blocking=True)

    for _ in range(3):   # warm-up steps, as for the device timing
        step()
    torch.cuda.synchronize()
    evs = [torch.cuda.Event(enable_timing=True) for _ in range(steps + 1)]
    evs[0].record()
    for i in range(steps):
        step()
        evs[i + 1].record()
    evs[-1].synchronize()
    per_step = sorted(evs[i].elapsed_time(evs[i + 1]) for i in range(steps))
    total_ms = evs[0].elapsed_time(evs[-1])
    median_ms = per_step[len(per_step) // 2]
    spread = {"median_ms": median_ms, "mean_ms": total_ms / steps, "min_ms": per_step[0], "max_ms": per_step[-1]}
    return median_ms / 1e3, h2d, d2h, spread


def cpu_baseline(A, B, size, rows):
    """The oracle, as it stands, on a band of `rows` rows of the headline workload
    (A, B: its host BF16 codes)."""
    import oracle
    oracle.build()
    t0 = time.time()
    oracle.gemm("bf16", A[:rows], B)
    dt = time.time() - t0
    return {"value": 2.0 * rows * size * size / dt / 1e12, "unit": "TFLOP/s", "cores": oracle.num_threads(),
            "kind": "oracle", "sample": f"rows 0..{rows - 1} of A against all {size} rows of B, K={size} "
                                        f"(FP64, {dt:.1f} s)"}


# The oracle beside the GPU lines: (label, format, m, n, k, seed, rows timed).  Inputs are drawn from the
# same seeds and quantised by the oracle's own quantisers on the host; a band of rows bounds the larger ones.
CPU_SWEEP = [
    ("BF16 M=N=K=512", "bf16", 512, 512, 512, SEEDS["bf16"], 512),
    ("BF16 M=N=K=2048", "bf16", 2048, 2048, 2048, SEEDS["bf16"], 2048),
    ("BF16 M=N=K=4096", "bf16", 4096, 4096, 4096, SEEDS["bf16"], 256),
    ("MXFP8 M=N=K=4096", "mxfp8", 4096, 4096, 4096, SEEDS["mxfp8"], 256),
    ("NVFP4 M=N=K=4096", "nvfp4", 4096, 4096, 4096, SEEDS["nvfp4"], 256),
    ("BF16 M=16 N=K=8192", "bf16", 16, 8192, 8192, 1004, 16),
    ("NVFP4 M=16 N=K=8192", "nvfp4", 16, 8192, 8192, 1004, 16),
]


def cpu_oracle_sweep(configs=CPU_SWEEP):
    """The oracle, as it stands, timed on each listed configuration (its GEMM only, on `rows` rows of A
    against all of B), in GFLOP/s."""
    import oracle
    from dense_block_scaled_gb300 import synth
    oracle.build()
    out = {}
    for label, fmt, m, n, k, seed, rows in configs:
        a, b = synth.gemm_inputs_f32(m, n, k, seed)
        a = a[:rows]
        if fmt == "bf16":
            args = (synth.bf16_codes(a), synth.bf16_codes(b))
        elif fmt == "mxfp8":
            (qa, sa), (qb, sb) = oracle.quant_mxfp8(a), oracle.quant_mxfp8(b)
            args = (qa, qb, sa, sb)
        else:
            (qa, sa, ta), (qb, sb, tb) = oracle.quant_nvfp4(a), oracle.quant_nvfp4(b)
            args = (qa, qb, sa, sb, oracle.alpha_eff(1.0, ta, tb))
        del a, b
        t0 = time.time()
        oracle.gemm(fmt, *args)
        dt = time.time() - t0
        out[label] = {"gflops": 2.0 * rows * n * k / dt / 1e9, "rows": rows, "seconds": dt}
    return out


# --------------------------------------------------------------------------- arms

def headline_config(size, l2_desc):
    return {"workload": f"BF16 GEMM M=N=K={size}", "A": f"{size}x{size} bf16 N(0,1) seed {SEEDS['bf16']}",
            "B": f"{size}x{size} bf16 N(0,1)", "alpha": 1.0, "accumulate": "fp32", "output": "bf16",
            "l2": l2_desc}


def l2_description(groups, mode):
    if mode == "flush":
        return "explicit flush (2x L2 write) before every launch"
    return "inputs larger than 3x L2, no rotation needed" if groups == 1 else f"{groups} rotated input groups"


def config_table(by_format, nontile, skinny, size, lists=None):
    """The workload definition's configurations in one compact table (TFLOP/s or
    microseconds and the roofline fractions), for the headline line's roofline
    object."""
    name = {"bf16": "BF16", "mxfp8": "MXFP8", "nvfp4": "NVFP4"}
    keys = ("tflops", "frac_of_pages_peak", "frac_of_measured", "frac_of_nominal")
    out = {}
    for fmt, e in by_format.items():
        out[f"{name[fmt]} {size}^3"] = {k: e.get(k) for k in keys}
        if e.get("measured_peak_source"):
            out[f"{name[fmt]} {size}^3"]["measured_peak"] = e["measured_peak_tflops"]
    for key, e in nontile.items():
        fmt, s_ = key.split()
        out[f"{name[fmt]} {s_}^3"] = {k: e.get(k) for k in keys}
    for key, e in skinny.items():
        out[key.replace("bf16", "BF16").replace("nvfp4", "NVFP4")] = {
            "us": e["us"], "tflops": e["tflops"], "frac_of_hbm": e["frac_of_hbm"],
            "frac_of_pages_hbm": e.get("frac_of_pages_hbm"), "frac_of_roofline": e["frac_of_roofline"]}
    for key, e in (lists or {}).items():
        out["list " + key] = {"us_per_gemm": e["us_per_gemm"], "tflops": e["tflops"], "frac_of_hbm": e["frac_of_hbm"],
                              "speedup_vs_single_launches": e.get("speedup_vs_single_launches"),
                              "us_per_gemm_graph": e.get("us_per_gemm_graph"),
                              "speedup_vs_single_launches_graph": e.get("speedup_vs_single_launches_graph")}
    return out


def max_over_ranks(t, dist, torch, device):
    """The job's time: the slowest rank's (each rank times the same number of
    steps of its own replica)."""
    if dist is None:
        return t
    tt = torch.tensor([t], dtype=torch.float64, device=device)
    dist.all_reduce(tt, op=dist.ReduceOp.MAX)
    return float(tt.item())


def job_value(world, units_per_rank, t_max):
    """Whole-job throughput: the units every rank processed, over the job's time."""
    return world * units_per_rank / t_max


def run_reference(args):
    """CPU oracle on the host cores: each step = a sample of output elements."""
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return 0
    import numpy as np

    import oracle
    from dense_block_scaled_gb300 import synth
    size = args.size
    oracle.build()
    a_rows = 64
    a, b = synth.gemm_inputs_f32(size, size, size, SEEDS["bf16"])   # the whole workload, as the GPU arm
    A, B = synth.bf16_codes(a[:a_rows]), synth.bf16_codes(b)
    del a, b
    rng = np.random.default_rng(0)
    per_step = 256
    ii = rng.integers(0, a_rows, size=(args.warmup + args.steps, per_step))
    jj = rng.integers(0, size, size=(args.warmup + args.steps, per_step))
    for s in range(args.warmup):
        oracle.gemm_elems("bf16", A, B, None, None, 1.0, ii[s], jj[s])
    t0 = time.time()
    for s in range(args.warmup, args.warmup + args.steps):
        oracle.gemm_elems("bf16", A, B, None, None, 1.0, ii[s], jj[s])
    dt = (time.time() - t0) / max(args.steps, 1)
    value = 2.0 * per_step * size / dt / 1e12
    line = {
        "impl": "reference", "metric": "GEMM TFLOP/s (BF16 D=A.B^T, M=N=K=%d)" % size, "value": value,
        "unit": "TFLOP/s", "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": dt * 1e3, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "f64", "data": "synthetic",
        "config": dict(headline_config(size, l2_description(1 if size >= 8192 else 2, "rotate")),
                       sample_per_step=f"{per_step} output elements"),
        "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": oracle.num_threads(), "kind": "oracle",
                         "sample": f"{per_step} random output elements per step, each a K={size} FP64 dot product"},
        "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


def run_ours(args):
    import torch
    from dense_block_scaled_gb300 import build, synth, tkg

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    torch.cuda.set_device(local)
    dist = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    build.build()
    tkg.load()
    pk = peaks()
    props = torch.cuda.get_device_properties(local)
    l2 = int(getattr(props, "L2_cache_size", 0) or 0) or 126 * 2 ** 20
    uuid = "GPU-" + str(props.uuid) if hasattr(props, "uuid") else str(local)

    formats = [f for f in args.formats.split(",") if f]
    hf = args.head_format
    head = Workload(hf, args.size, SEEDS[hf], l2, torch, tkg, synth,
                    keep_host=(rank == 0 and not args.no_cpu and hf == "bf16"))
    flush_buf = torch.empty(2 * l2 // 4, dtype=torch.float32, device="cuda") if args.l2 == "flush" else None

    clocks = ClockSampler(uuid)
    clocks.start()
    t_head = time_launches(head, args.steps, args.warmup, torch, tkg, dist, args.l2, flush_buf)
    clk = clocks.stop()

    t_max = max_over_ranks(t_head, dist, torch, "cuda")
    value = job_value(world, head.flop, t_max) / 1e12
    achieved = head.flop / t_head / 1e12
    sustained = None
    if rank == 0 and args.sustained_s > 0:
        ts, ns, secs, sclk = sustained_seconds(head, args.sustained_s, t_head, torch, tkg, uuid)
        tf = head.flop / ts / 1e12
        sustained = {"tflops": tf, "launches": ns, "seconds": secs, "clocks": sclk,
                     "frac_of_sustained_peak": (tf / (pk["bf16_sustained"] * NOMINAL_RATIO[hf])
                                                if pk["bf16_sustained"] else None),
                     "frac_of_pages_peak": tf / PAGES_PEAK_TFLOPS[hf]}

    PAUSE_S[0] = max(args.sleep_ms, 0) / 1e3   # from here on every timed workload starts after an idle pause
    vendor_peak = {}   # the vendor library's same-loop TFLOP/s on the same operands: a measured per-format peak

    def fmt_entry(w, t):
        tf = w.flop / t / 1e12
        nominal = pk["bf16"] * NOMINAL_RATIO[w.fmt]
        if w.fmt == "bf16":
            peak_meas, src = pk["bf16"], f"{pk['source']} cuBLAS bf16 burst"
        elif w.fmt in vendor_peak:
            peak_meas, src = vendor_peak[w.fmt], "vendor library, same operands, same loop"
        else:
            peak_meas, src = None, None
        return {"tflops": tf, "ms": t * 1e3, "frac_of_pages_peak": tf / PAGES_PEAK_TFLOPS[w.fmt],
                "pages_peak_tflops": PAGES_PEAK_TFLOPS[w.fmt],
                "measured_peak_tflops": peak_meas, "frac_of_measured": tf / peak_meas if peak_meas else None,
                "measured_peak_source": src, "nominal_peak_tflops": nominal, "frac_of_nominal": tf / nominal,
                "input_groups": w.groups}

    by_format, sweep, sweep_scaled, skinny, quant, grouped, grouped_decode = {}, {}, {}, {}, {}, {}, {}
    nontile = {}
    lists = {}
    vendor = {}
    e2e = None
    if rank == 0:
        by_format[hf] = fmt_entry(head, t_head)
        for fmt in formats:
            if fmt == hf:
                continue
            w = Workload(fmt, args.size, SEEDS[fmt], l2, torch, tkg, synth,
                         keep_fp32=(fmt != "bf16" and not args.no_quant and not quant))
            tw = time_launches(w, args.steps, args.warmup, torch, tkg, None, args.l2, flush_buf)
            if fmt != "bf16" and not args.no_vendor_peak:
                try:
                    tv = time_launches(VendorGemm(w, torch), args.steps, args.warmup, torch, tkg, None, args.l2,
                                       flush_buf)
                    vendor_peak[fmt] = w.flop / tv / 1e12
                except Exception:   # a vendor build without the format: no measured peak
                    pass
            by_format[fmt] = fmt_entry(w, tw)
            if w.fp32 is not None:
                quant = quant_timings(w.fp32, 20, 3, torch, tkg, pk["hbm_gbs"])
            del w
            torch.cuda.empty_cache()
        for s in [int(x) for x in args.sweep.split(",") if x]:
            w = Workload("bf16", s, SEEDS["bf16"], l2, torch, tkg, synth)
            t = time_launches(w, args.steps, min(args.warmup, 500), torch, tkg, None, args.l2, flush_buf)
            tg = graph_seconds(w, args.steps, torch, tkg)
            sweep[str(s)] = {"tflops": w.flop / t / 1e12, "us": t * 1e6, "input_groups": w.groups,
                             "frac_of_pages_peak": w.flop / t / 1e12 / PAGES_PEAK_TFLOPS["bf16"],
                             "us_graph": tg * 1e6, "tflops_graph": w.flop / tg / 1e12}
            del w
            torch.cuda.empty_cache()
        for fmt in ("mxfp8", "nvfp4"):
            for s in [int(x) for x in args.sweep_scaled.split(",") if x]:
                w = Workload(fmt, s, SEEDS[fmt], l2, torch, tkg, synth)
                t = time_launches(w, args.steps, min(args.warmup, 500), torch, tkg, None, args.l2, flush_buf)
                sweep_scaled[f"{fmt} {s}"] = {"tflops": w.flop / t / 1e12, "us": t * 1e6, "input_groups": w.groups,
                                              "frac_of_pages_peak": w.flop / t / 1e12 / PAGES_PEAK_TFLOPS[fmt]}
                del w
                torch.cuda.empty_cache()
        for fmt in ("bf16", "nvfp4"):
            for s_ in [int(x) for x in args.nontile.split(",") if x]:
                w = Workload(fmt, s_, SEEDS[fmt], l2, torch, tkg, synth)
                t = time_launches(w, args.steps, min(args.warmup, 500), torch, tkg, None, args.l2, flush_buf)
                nontile[f"{fmt} {s_}"] = fmt_entry(w, t)
                del w
                torch.cuda.empty_cache()
        for fmt in ("bf16", "nvfp4"):
            for mm in [int(x) for x in args.skinny.split(",") if x]:
                w = Workload(fmt, 8192, 1004, l2, torch, tkg, synth, mnk=(mm, 8192, 8192))
                t = time_launches(w, args.steps, min(args.warmup, 500), torch, tkg, None, args.l2, flush_buf)
                tg = graph_seconds(w, args.steps, torch, tkg)
                byts = w.in_bytes + w.out_bytes
                tf = w.flop / t / 1e12
                roof = min(PAGES_PEAK_TFLOPS[fmt], w.flop / byts * pk["hbm_gbs"] / 1e3)
                skinny[f"{fmt} M={mm} N=K=8192"] = {
                    "us": t * 1e6, "tflops": tf, "gbs": byts / t / 1e9, "frac_of_hbm": byts / t / 1e9 / pk["hbm_gbs"],
                    "frac_of_pages_hbm": byts / t / 1e9 / PAGES_HBM_GBS,
                    "roofline_tflops": roof, "frac_of_roofline": tf / roof, "input_groups": w.groups,
                    "us_graph": tg * 1e6, "frac_of_roofline_graph": w.flop / tg / 1e12 / roof}
                del w
                torch.cuda.empty_cache()
        if not args.no_list:
            def us(d):
                return (d.get("us"), d.get("us_graph")) if d else (None, None)
            single = {"BF16 8 x 512^3": us(sweep.get("512")),
                      "BF16 8 x M=16 N=K=8192": us(skinny.get("bf16 M=16 N=K=8192")),
                      "NVFP4 8 x M=16 N=K=8192": us(skinny.get("nvfp4 M=16 N=K=8192"))}
            lists = list_timings(max(args.steps, 100), min(args.warmup, 50), l2, torch, tkg, synth, pk["hbm_gbs"],
                                 single)
        if args.grouped:
            gg, gt, gn, gk = [int(x) for x in args.grouped.split(",")]
            grouped = grouped_timings([f for f in ("bf16", "mxfp8", "nvfp4")], gg, gt, gn, gk,
                                      min(args.steps, 50), min(args.warmup, 20), torch, tkg, synth)
        if args.grouped_decode:
            dg, dr, dn, dk = [int(x) for x in args.grouped_decode.split(",")]
            grouped_decode = grouped_decode_timings(dg, dr, dn, dk, max(args.steps, 100), min(args.warmup, 50), torch,
                                                    tkg, synth, pk["hbm_gbs"])
        if args.vendor:
            vendor = vendor_timings(formats, [int(x) for x in args.vendor.split(",") if x], args.steps,
                                    min(args.warmup, 500), l2, torch, tkg, synth, args.l2, flush_buf)
        if not args.no_e2e:
            te, h2d, d2h, spread = e2e_seconds(head, args.e2e_steps, torch, tkg)
            # value: the median step.  The host link and host memory are shared with
            # other jobs on the machine, and a single step stalled by them (tens of ms)
            # moves the mean of 20 steps by up to 10x; the mean and the spread are kept
            e2e = {"value": world * head.flop / te / 1e12, "unit": "TFLOP/s", "h2d_bytes_per_step": h2d,
                   "d2h_bytes_per_step": d2h, "ms_per_step": te * 1e3, "stat": f"median of {args.e2e_steps} steps",
                   "step_ms": spread}

    cpu = None
    cpu_sweep = {}
    if rank == 0 and not args.no_cpu and head.host is not None:
        cpu = cpu_baseline(head.host[0], head.host[1], args.size, args.cpu_rows)
        cpu_sweep = cpu_oracle_sweep()

    if rank == 0:
        name = {"bf16": "BF16", "mxfp8": "MXFP8", "nvfp4": "NVFP4"}[hf]
        workload = f"{name} GEMM M=N=K={args.size}"
        peak = pk["bf16"] * NOMINAL_RATIO[hf]
        line = {
            "metric": f"GEMM TFLOP/s ({name} D=A.B^T, M=N=K={args.size})",
            "value": value, "unit": "TFLOP/s", "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": t_max * 1e3, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": hf, "data": "synthetic",
            "config": dict(headline_config(args.size, l2_description(head.groups, args.l2)) if hf == "bf16"
                           else {"workload": workload, "l2": l2_description(head.groups, args.l2)},
                           frac_of_pages_peak=value / world / PAGES_PEAK_TFLOPS[hf],
                           pages_peak_tflops=PAGES_PEAK_TFLOPS[hf], replicas=world),
            "roofline": {"bound": "tensor", "achieved": achieved, "peak": peak, "unit": "TFLOP/s",
                         "frac": achieved / peak, "traffic": recorded_traffic(workload),
                         "peak_source": f"{pk['source']} cuBLAS bf16 burst x {NOMINAL_RATIO[hf]:g} (nominal {hf}/bf16)",
                         "frac_of_sustained": (achieved / (pk["bf16_sustained"] * NOMINAL_RATIO[hf])
                                               if pk["bf16_sustained"] else None),
                         "sustained": sustained,
                         "configs": config_table(by_format, nontile, skinny, args.size, lists)},
            "cpu_baseline": cpu,
            "e2e": e2e,
            "gpu_launches": args.steps,
            "clocks": clk,
            "formats": by_format,
            "sweep_bf16": sweep,
            "sweep_scaled": sweep_scaled,
            "nontile": nontile,
            "gemm_list": lists,
            "skinny": skinny,
            "quantize": quant,
            "grouped": grouped,
            "grouped_decode": grouped_decode,
            "kernel_hash": kernel_hash(),
        }
        if vendor:
            line["vendor_library"] = vendor
        if cpu_sweep:
            line["cpu_oracle_sweep"] = cpu_sweep
        print(json.dumps(line), flush=True)
    if dist is not None:
        dist.barrier()
        dist.destroy_process_group()
    return 0


def main():
    args = parse_args()
    if args.impl == "reference":
        return run_reference(args)
    return run_ours(args)


if __name__ == "__main__":
    sys.exit(main())
