"""Benchmark of the BF16 MoE grouped GEMM backward on GB300.

One step = one pass of the whole hot path over one batch of seeded synthetic input:
the grouped dgrad GEMM fused with the dSwiGLU/dGeGLU epilogue (dprob, optional dbias)
followed by the grouped wgrad on the same expert ranges.  The default workload is the
DeepSeek-like layer (L=256 experts, hidden 7168, N 2048, 131072 tokens Zipf(1.0),
rounded to 256 per expert): the one workload that carries both halves.  Other
workloads (--workload mixtral | geglu | wgrad64 | tiny) time whichever halves they have.

By default the line also carries ``per_config``: the four other layers of the same
benchmark family (tiny, mixtral, geglu, wgrad64) timed the same way, each part with its
TFLOP/s, fraction of the measured dense BF16 peak, arithmetic intensity against the measured
ridge point, the roof that bounds it and the fraction of that attainable roof.

Usage: python bench.py [--gpus N] [--steps K] [--warmup W] [--impl mgg|reference] [--workload NAME]
Under torchrun every rank runs an independent replica (weak scaling); rank 0 prints
one JSON line.  ``--gpus N`` with N > 1 outside torchrun starts N local ranks itself.
"""
from __future__ import annotations

import argparse
import hashlib
import re
import glob
import json
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "grouped GEMM TFLOP/s (dGLU dgrad, wgrad) and % of GB300 dense BF16 peak"
WORKLOAD_TEXT = {
    "deepseek": "DeepSeek-like: L=256, K=hidden=7168, N=2048, 131072 tokens Zipf(1.0) rounded to 256 per expert "
                "(M=T=162304); dSwiGLU dgrad (dense K-major B, BF16 C/D_row, dprob) then wgrad on the same ranges "
                "(A' (7168,T) K-major tensor_ragged, B' (T,2048) N-major, discrete FP32 outputs, overwrite)",
    "mixtral": "Mixtral-like dSwiGLU dgrad: L=8, K=4096, N=14336, 32768 tokens uniform (M=33536), dense B, BF16 D_row",
    "geglu": "dGeGLU dgrad: L=16, K=2048, N=5632, 49152 tokens Zipf(1.1) (M=50688), discrete N-major B, "
             "C~N(0,4), FP32 D_row, dbias",
    "wgrad64": "grouped wgrad: L=64, hidden=2048, inter=1408, T=65536 Zipf(1.2), FP32 dense accumulate",
    "tiny": "tiny: L=4, counts [256,0,512,256], K=hidden=256, N=128",
    "mixtral_situ": "Mixtral-like shape with the dSiTU-GLU backward (beta1=4, beta2=25), C~N(0,4), BF16 D_row",
    "dsrelu": "Mixtral-like shape with the dsReLU backward: L=8, K=4096, N=14336, 32768 tokens uniform, "
              "C (M,N) BF16, BF16 D_row, dprob and per-expert Amax",
    "mixtral_s": "profiling copy of mixtral with L=2 experts, 8192 tokens",
    "geglu_s": "profiling copy of geglu with 12288 tokens",
    "deepseek_s": "profiling copy of deepseek with L=32 experts, 16384 tokens",
    "dsrelu_s": "profiling copy of dsrelu with L=2 experts, 8192 tokens",
}


def env_int(name, default):
    v = os.environ.get(name)
    return int(v) if v not in (None, "") else default


# ----------------------------------------------------------------------------------------
# clocks sampled during the timed region
# ----------------------------------------------------------------------------------------
class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.lines = []

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "100"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
        except (OSError, ValueError):
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self):
        if self.proc is None:
            return None
        time.sleep(0.15)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.thread.join(timeout=2)
        sm, smax, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                smax = float(parts[2])
            except ValueError:
                continue
            for n, v in zip(names, parts[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        if not sm:
            return None
        loaded = [s for s in sm if s > 0.5 * (smax or max(sm))] or sm
        return {"sm_mhz": statistics.median(loaded), "sm_max_mhz": smax, "reasons": sorted(reasons),
                "samples": len(sm)}


# ----------------------------------------------------------------------------------------
# peaks, traffic
# ----------------------------------------------------------------------------------------
def measured_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return {"bf16_tflops": d["bf16_tflops"], "bf16_tflops_sustained": d.get("bf16_tflops_sustained"),
                "hbm_gbs": d["hbm_gbs"], "source": "measured"}
    return {"bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0, "hbm_gbs": 6800.0, "source": "fallback"}


# The sources each recorded kernel is built from (its own translation unit, the shared headers,
# the host code that encodes its tensor maps, the ABI header).
KERNEL_SOURCES = {
    "dglu_bwd_kernel": ("dglu_bwd.cu",),
    "wgrad_kernel": ("wgrad.cu",),
}
SHARED_SOURCES = ("mgg_pipeline.cuh", "mgg_ptx.cuh", "mgg_internal.h", "mgg_api.cu")


_COMMENTS = re.compile(r"/\*.*?\*/|//[^\n]*", re.S)


def source_sha(kernel: str = None) -> str:
    """Hash of the code of the CUDA sources (all of them, or those `kernel` is built from) and of
    the ABI headers: comments and whitespace are left out, so that a profile stays matched to
    the code it measured when only the documentation changes."""
    h = hashlib.sha1()
    csrc = os.path.join(ROOT, "moe_grouped_gemm_persistent_gb300", "csrc")
    if kernel is None:
        files = glob.glob(os.path.join(csrc, "*"))
    else:
        files = [os.path.join(csrc, f) for f in KERNEL_SOURCES[kernel] + SHARED_SOURCES]
    files = sorted(files + glob.glob(os.path.join(ROOT, "include", "*.h")))
    for f in files:
        with open(f, encoding="utf-8", errors="replace") as fh:
            code = " ".join(_COMMENTS.sub(" ", fh.read()).split())
        h.update(os.path.basename(f).encode() + b"\0" + code.encode())
    return h.hexdigest()[:16]


def recorded_traffic(kernel: str, workload: str):
    """dram bytes per launch from a committed ncu summary, if it matches the current sources."""
    p = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(p):
        return None
    with open(p) as f:
        d = json.load(f)
    ent = d.get(f"{kernel}/{workload}")
    if not ent or kernel not in KERNEL_SOURCES or ent.get("source_sha") != source_sha(kernel):
        return None
    return ent.get("dram_bytes_per_launch")


def roofline_of(flops: float, algo_bytes: float, ms: float, peaks) -> dict:
    """Where one kernel launch sits against the measured roofs: its arithmetic intensity (FLOPs per
    algorithmic byte) against the ridge point (dense BF16 peak / HBM copy bandwidth) decides the
    binding roof, attainable = min(tensor peak, intensity x HBM bandwidth).  Work that would take
    under 10 us at the attainable rate is bound by launch latency, not by either roof."""
    peak_tf, bw = peaks["bf16_tflops"], peaks["hbm_gbs"]
    tf = flops / (ms * 1e-3) / 1e12
    ai = flops / algo_bytes
    ridge = peak_tf * 1e12 / (bw * 1e9)
    attainable = min(peak_tf, ai * bw * 1e9 / 1e12)
    bound = "tensor" if ai >= ridge else "hbm"
    if flops / (attainable * 1e12) < 10e-6:
        bound = "launch"
    return {"ms": round(ms, 4), "tflops": round(tf, 1), "frac_of_peak": round(tf / peak_tf, 4),
            "algorithmic_gb": round(algo_bytes / 1e9, 4), "achieved_gbs": round(algo_bytes / (ms * 1e-3) / 1e9, 1),
            "ai_flop_per_byte": round(ai, 1), "ridge_flop_per_byte": round(ridge, 1), "bound": bound,
            "attainable_tflops": round(attainable, 1), "frac_of_attainable": round(tf / attainable, 4)}


# ----------------------------------------------------------------------------------------
# the CUDA path
# ----------------------------------------------------------------------------------------
class Problem:
    """Device-resident inputs/outputs of one workload and the two ABI calls of a step."""

    def __init__(self, workload: str, dev, sched: str = "dynamic", cta: str = "auto"):
        import torch
        from moe_grouped_gemm_persistent_gb300 import api, synth
        self.api = api
        self.torch = torch
        self.dev = dev
        self.workload = workload
        self.sched = sched
        self.cta = cta
        self.dspec, self.wspec = synth.workload_specs(workload)
        self.d = self.w = None
        if self.dspec is not None:
            s = self.dspec
            x = synth.make_dglu_inputs(s, device=dev)
            self.d = x
            self.srelu = s.act == "dsrelu"
            cols = s.N if self.srelu else 2 * s.N
            self.d_row = torch.empty(s.M, cols, dtype=synth.torch_dtype(s.d_dtype), device=dev)
            self.amax = torch.zeros(s.L, dtype=torch.float32, device=dev) if self.srelu else None
            self.dprob = torch.zeros(s.M, dtype=torch.float32, device=dev)
            self.dbias = torch.zeros(s.L, 2 * s.N, dtype=torch.bfloat16, device=dev) if s.dbias else None
            if s.b_mode == "discrete":
                self.b_ptrs = api.pointer_array(x["b"], dev)
                self.b_kw = dict(b_ptrs=self.b_ptrs, b_major=s.b_major, N=s.N)
            else:
                self.b_kw = dict(b=x["b"])
            self.d_ws = api.new_workspace(api.dsrelu_bwd_workspace_size(s.L) if self.srelu
                                          else api.dglu_bwd_workspace_size(s.L, s.N), dev)
        if self.wspec is not None:
            s = self.wspec
            y = synth.make_wgrad_inputs(s, device=dev)
            self.w = y
            odt = synth.torch_dtype(s.out_dtype)
            self.w_out = torch.empty(s.L, s.hidden, s.inter, dtype=odt, device=dev)
            if s.accumulate:
                self.w_out.copy_(y["out_old"])
            if s.out_mode == "discrete":
                self.w_kw = dict(out_ptrs=api.pointer_array([self.w_out[e] for e in range(s.L)], dev),
                                 out_dtype=s.out_dtype)
            else:
                self.w_kw = dict(out=self.w_out)
            self.w_ws = api.new_workspace(api.wgrad_workspace_size(s.L), dev)
        torch.cuda.synchronize(dev)

    @property
    def launches_per_step(self) -> int:
        n = 0
        if self.dspec is not None:
            n += 2 + (1 if self.dspec.dbias else 0)
        if self.wspec is not None:
            n += 2
        return n

    def reset_outputs(self):
        """Zeroes the outputs the dgrad accumulates into (dprob, dbias), as a caller does before
        each step; the per-part timings leave this out, the step timing keeps it."""
        if self.dspec is not None:
            self.dprob.zero_()
            if self.dbias is not None:
                self.dbias.zero_()

    def dgrad_step(self):
        self.reset_outputs()
        self.dgrad()

    def dgrad(self):
        s, x = self.dspec, self.d
        if self.srelu:
            self.api.dsrelu_bwd(a=x["a"], c=x["c"], padded_offsets=x["padded_offsets"], alpha=x["alpha"],
                                prob=x["prob"], dprob=self.dprob, d_row=self.d_row, amax=self.amax,
                                workspace=self.d_ws, sched=self.sched, cta=self.cta, **self.b_kw)
            return
        self.api.dglu_bwd(a=x["a"], c=x["c"], padded_offsets=x["padded_offsets"], alpha=x["alpha"], beta=x["beta"],
                          prob=x["prob"], dprob=self.dprob, d_row=self.d_row, dbias=self.dbias, act=s.act,
                          workspace=self.d_ws, sched=self.sched, cta=self.cta, **self.b_kw)

    def wgrad(self):
        s, y = self.wspec, self.w
        self.api.wgrad(a=y["a"], b=y["b"], offsets=y["offsets"], hidden=s.hidden, inter=s.inter,
                       a_major=s.a_major, b_major=s.b_major, input_order=s.input_order, accumulate=s.accumulate,
                       workspace=self.w_ws, sched=self.sched, cta=self.cta, **self.w_kw)

    def flops(self):
        f = {}
        if self.dspec is not None:
            f["dgrad"] = self.dspec.flops
        if self.wspec is not None:
            f["wgrad"] = self.wspec.flops
        return f

    def algorithmic_bytes(self):
        """Compulsory HBM bytes per launch of each kernel (inputs read once, outputs written once)."""
        b = {}
        if self.dspec is not None:
            s = self.dspec
            esz = {"bf16": 2, "fp16": 2, "fp32": 4}
            nz = int((s.counts > 0).sum())
            cols = s.N if s.act == "dsrelu" else 2 * s.N
            b["dgrad"] = (s.M * s.K * 2 + nz * s.N * s.K * 2 + s.M * cols * (esz[s.c_dtype] + esz[s.d_dtype])
                          + s.M * 12)
        if self.wspec is not None:
            s = self.wspec
            esz = {"bf16": 2, "fp16": 2, "fp32": 4}[s.out_dtype]
            nz = int((s.counts > 0).sum())
            outs = s.L if not s.accumulate else nz
            b["wgrad"] = (s.hidden * s.T * 2 + s.T * s.inter * 2 +
                          outs * s.hidden * s.inter * esz * (2 if s.accumulate else 1))
        return b

    def check_status(self):
        if self.dspec is not None:
            assert self.api.read_device_status(self.d_ws) == 0, self.api.last_error()
        if self.wspec is not None:
            assert self.api.read_device_status(self.w_ws) == 0, self.api.last_error()


def time_steps(prob: "Problem", steps: int, warmup: int, world: int):
    import torch
    dev = prob.dev
    stream = torch.cuda.current_stream(dev)
    parts = [k for k in ("dgrad", "wgrad") if (prob.dspec if k == "dgrad" else prob.wspec) is not None]
    fns = {"dgrad": prob.dgrad, "wgrad": prob.wgrad}
    for _ in range(warmup):
        prob.reset_outputs()
        for k in parts:
            fns[k]()
    torch.cuda.synchronize(dev)
    prob.check_status()
    ev = {k: [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(steps)]
          for k in parts}
    start, stop = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    sampler = ClockSampler(dev.index if dev.index is not None else 0)
    sampler.start()
    time.sleep(0.3)
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize(dev)
    start.record(stream)
    for i in range(steps):
        prob.reset_outputs()
        for k in parts:
            ev[k][i][0].record(stream)
            fns[k]()
            ev[k][i][1].record(stream)
    stop.record(stream)
    torch.cuda.synchronize(dev)
    if world > 1:
        torch.distributed.barrier()
    clocks = sampler.stop()
    total_ms = start.elapsed_time(stop)
    per = {k: statistics.median(a.elapsed_time(b) for a, b in ev[k]) for k in parts}
    prob.check_status()
    return total_ms, per, clocks


def _io_parts(prob: "Problem"):
    """Per part of the step (dgrad, wgrad): the device inputs it reads, the outputs it writes and
    the call that runs it."""
    import torch
    parts = []
    if prob.dspec is not None:
        x = prob.d
        bs = [x["b"]] if isinstance(x["b"], torch.Tensor) else list(x["b"])
        ins = [x["a"], x["c"], x["alpha"], x["beta"], x["prob"], x["padded_offsets"], *bs]
        outs = [prob.d_row, prob.dprob] + ([prob.dbias] if prob.dbias is not None else [])
        parts.append((ins, outs, prob.dgrad_step))
    if prob.wspec is not None:
        y = prob.w
        parts.append(([y["a"], y["b"], y["offsets"]], [prob.w_out], prob.wgrad))
    return parts


def time_e2e(prob: "Problem", steps: int, warmup: int):
    """Same step through the public API with pinned host buffers: every step copies all its inputs
    host -> device and all its outputs device -> host inside the timed region.  The copies in and
    out and the ABI calls run on three CUDA streams, with two device buffer sets used by alternate
    steps, so step i's results leave while step i + 1's inputs arrive and compute (the host link
    carries both directions at once).  Each part waits only for its own inputs, and its outputs
    leave as soon as it is done.  The timed region runs from the first input copy to the end of
    the last output copy."""
    import torch
    dev = prob.dev
    sets = [prob, Problem(prob.workload, dev, prob.sched, prob.cta)]
    io = [_io_parts(p) for p in sets]
    host_in = [[torch.empty(t.shape, dtype=t.dtype, pin_memory=True) for t in ins] for ins, _, _ in io[0]]
    for hs, (ins, _, _) in zip(host_in, io[0]):
        for h, t in zip(hs, ins):
            h.copy_(t)
    host_out = [[torch.empty(t.shape, dtype=t.dtype, pin_memory=True) for t in outs] for _, outs, _ in io[0]]
    bi = sum(t.numel() * t.element_size() for ins, _, _ in io[0] for t in ins)
    bo = sum(t.numel() * t.element_size() for _, outs, _ in io[0] for t in outs)
    s_in, s_cmp, s_out = (torch.cuda.Stream(dev) for _ in range(3))
    nparts = len(io[0])

    def run(n):
        # per part and buffer set: the last compute and the last output copy issued on it
        cmp_done = [[None, None] for _ in range(nparts)]
        out_done = [[None, None] for _ in range(nparts)]
        for i in range(n):
            k = i % 2
            in_done = []
            with torch.cuda.stream(s_in):
                for j, (ins, _, _) in enumerate(io[k]):
                    if cmp_done[j][k] is not None:  # step i - 2 has finished reading these inputs
                        s_in.wait_event(cmp_done[j][k])
                    for h, t in zip(host_in[j], ins):
                        t.copy_(h, non_blocking=True)
                    e = torch.cuda.Event()
                    e.record(s_in)
                    in_done.append(e)
            with torch.cuda.stream(s_cmp):
                for j, (_, _, fn) in enumerate(io[k]):
                    s_cmp.wait_event(in_done[j])
                    if out_done[j][k] is not None:  # step i - 2's outputs have left this set
                        s_cmp.wait_event(out_done[j][k])
                    fn()
                    cmp_done[j][k] = torch.cuda.Event()
                    cmp_done[j][k].record(s_cmp)
            with torch.cuda.stream(s_out):
                for j, (_, outs, _) in enumerate(io[k]):
                    s_out.wait_event(cmp_done[j][k])
                    for h, t in zip(host_out[j], outs):
                        h.copy_(t, non_blocking=True)
                    out_done[j][k] = torch.cuda.Event()
                    out_done[j][k].record(s_out)

    run(max(warmup, 2))
    torch.cuda.synchronize(dev)
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record(s_in)
    run(steps)
    b.record(s_out)
    torch.cuda.synchronize(dev)
    for p in sets:
        p.check_status()
    ms = a.elapsed_time(b) / steps
    del host_in, host_out, io, sets
    torch.cuda.empty_cache()
    return ms, bi, bo


# ----------------------------------------------------------------------------------------
# the oracle on the host cores (cpu_baseline and the reference arm)
# ----------------------------------------------------------------------------------------
def oracle_sample(prob_or_specs, dev, budget_s: float, seed: int = 0, max_experts=None):
    """Times the CPU oracle on whole experts of the workload, in a seeded order, until
    `budget_s` seconds of oracle time are spent.  Returns (TFLOP/s, seconds, sample text)."""
    import numpy as np
    import torch

    import oracle
    from moe_grouped_gemm_persistent_gb300 import synth

    dspec, wspec = prob_or_specs.dspec, prob_or_specs.wspec
    rng = np.random.default_rng(seed)
    f64 = lambda t: t.detach().to("cpu", torch.float64).numpy()
    spent, flops, done = 0.0, 0.0, []
    for part, spec in (("dgrad", dspec), ("wgrad", wspec)):
        if spec is None:
            continue
        part_budget = budget_s / (2 if (dspec is not None and wspec is not None) else 1)
        part_spent = 0.0
        offs = np.cumsum(spec.counts)
        ranges = oracle.expert_ranges(offs)
        cand = [e for e in rng.permutation(spec.L).tolist() if spec.counts[e] > 0]
        # prefer experts whose single evaluation fits the budget
        cand.sort(key=lambda e: 0 if spec.counts[e] <= 2048 else 1)
        for e in cand[: (max_experts or len(cand))]:
            lo, hi = ranges[e]
            if part == "dgrad":
                x = prob_or_specs.d
                a = f64(x["a"][lo:hi])
                bm = x["b"][e] if isinstance(x["b"], torch.Tensor) else x["b"][e]
                b_g = f64(bm) if (spec.b_mode == "dense" or spec.b_major == "k") else f64(bm).T
                c = f64(x["c"][lo:hi])
                offs_local = np.zeros(spec.L, dtype=np.int64)
                offs_local[e:] = hi - lo
                alpha, beta = x["alpha"].cpu().numpy(), x["beta"].cpu().numpy()
                pr = x["prob"][lo:hi].cpu().numpy()
                t0 = time.perf_counter()
                if spec.act == "dsrelu":
                    oracle.dsrelu_bwd(a, lambda g: b_g, c, offs_local, alpha, pr)
                else:
                    oracle.dglu_bwd(a, lambda g: b_g, c, offs_local, alpha, beta, pr, act=spec.act)
                dt = time.perf_counter() - t0
                fl = 2.0 * (hi - lo) * spec.N * spec.K
            else:
                y = prob_or_specs.w
                h, i = spec.hidden, spec.inter
                if spec.input_order == "tensor_ragged" and spec.a_major == "k":
                    a_blk = f64(y["a"][lo * h:hi * h])
                else:
                    a_blk = f64(y["a"].view(h, spec.T)[:, lo:hi]).reshape(-1)
                b_blk = f64(y["b"].view(spec.T, i)[lo:hi])
                offs_local = np.array([hi - lo], dtype=np.int64)
                old = None
                if spec.accumulate:
                    old = [f64(y["out_old"][e])]
                t0 = time.perf_counter()
                oracle.wgrad(a_blk, b_blk.reshape(-1), offs_local, h, i, a_major="k", b_major="n",
                             input_order="tensor2d", accumulate=spec.accumulate, out_old=old)
                dt = time.perf_counter() - t0
                fl = 2.0 * h * (hi - lo) * i
            spent += dt
            part_spent += dt
            flops += fl
            done.append((part, e, hi - lo))
            if part_spent >= part_budget:
                break
    text = []
    for part in ("dgrad", "wgrad"):
        sel = [(e, n) for p, e, n in done if p == part]
        if sel:
            unit = "rows" if part == "dgrad" else "tokens"
            text.append(f"{part}: {len(sel)} experts, {sum(n for _, n in sel)} {unit} (first: "
                        + ", ".join(f"e{e}" for e, _ in sel[:6]) + (", ..." if len(sel) > 6 else "") + ")")
    return flops / spent / 1e12, spent, "; ".join(text)


# ----------------------------------------------------------------------------------------
def max_over_ranks(value: float, dev) -> float:
    """The largest of every rank's value (the slowest rank's time decides a step)."""
    import torch
    t = torch.tensor([float(value)], dtype=torch.float64, device=dev)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return float(t.item())


PER_CONFIG = ("tiny", "mixtral", "geglu", "wgrad64")


def time_per_config(dev, args, peaks) -> dict:
    """The other layers of the benchmark family, each timed like the headline (warm-up, then
    `steps` steps between CUDA events, per-part events), with the roofline of every part."""
    import torch
    out = {}
    for name in PER_CONFIG:
        prob = Problem(name, dev, args.sched, args.cta)
        steps = max(args.steps, 50) if name == "tiny" else args.steps
        total_ms, per, clocks = time_steps(prob, steps, args.warmup, 1)
        flops, algo = prob.flops(), prob.algorithmic_bytes()
        out[name] = {"description": WORKLOAD_TEXT[name], "steps": steps, "ms_per_step": round(total_ms / steps, 4),
                     "parts": {k: roofline_of(flops[k], algo[k], ms, peaks) for k, ms in per.items()},
                     "clocks": clocks}
        del prob
        torch.cuda.empty_cache()
    return out


def spawn_local_ranks(n: int) -> int:
    """`--gpus N` outside torchrun: start N local ranks (one per GPU) with the same arguments."""
    import socket
    with socket.socket() as sk:
        sk.bind(("127.0.0.1", 0))
        port = sk.getsockname()[1]
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", f"--nproc-per-node={n}",
           "--master-addr", "127.0.0.1", "--master-port", str(port), os.path.abspath(__file__), *sys.argv[1:]]
    return subprocess.call(cmd, cwd=ROOT)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=10)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", default="mgg", choices=["mgg", "reference"])
    ap.add_argument("--workload", default="deepseek", choices=sorted(WORKLOAD_TEXT))
    ap.add_argument("--e2e-steps", type=int, default=16)
    ap.add_argument("--sched", default="dynamic", choices=["static", "dynamic"])
    ap.add_argument("--cta", default="auto", choices=["auto", "single", "pair"],
                    help="tile-to-SM mapping: one CTA per 128-row tile, or a CTA pair per 256-row tile")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-seconds", type=float, default=12.0)
    ap.add_argument("--no-per-config", action="store_true",
                    help="time only --workload (by default an N=1 run also times tiny, mixtral, geglu, wgrad64)")
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3

    if args.gpus > 1 and os.environ.get("WORLD_SIZE") in (None, ""):
        return spawn_local_ranks(args.gpus)
    world = env_int("WORLD_SIZE", 1)
    if world != args.gpus:
        print(f"bench.py: --gpus {args.gpus} but WORLD_SIZE={world}: launch one rank per GPU", file=sys.stderr)
        return 2
    rank = env_int("RANK", 0)
    local_rank = env_int("LOCAL_RANK", 0)

    if args.impl == "reference":
        return run_reference(args, world, rank)

    import torch
    if world > 1:
        torch.distributed.init_process_group("nccl")
    dev = torch.device("cuda", local_rank)
    torch.cuda.set_device(dev)
    from moe_grouped_gemm_persistent_gb300.build import build
    if rank == 0:
        build()
    if world > 1:
        torch.distributed.barrier()
    build()

    prob = Problem(args.workload, dev, args.sched, args.cta)
    total_ms, per, clocks = time_steps(prob, args.steps, args.warmup, world)
    if world > 1:
        total_ms = max_over_ranks(total_ms, dev)
    ms_step = total_ms / args.steps
    flops = prob.flops()
    step_flops = sum(flops.values())
    value = step_flops * world / (ms_step * 1e-3) / 1e12
    peaks = measured_peaks()

    algo = prob.algorithmic_bytes()
    parts = {k: roofline_of(flops[k], algo[k], ms, peaks) for k, ms in per.items()}
    dom = max(per, key=lambda k: per[k])
    kernel_name = {"dgrad": "dglu_bwd_kernel", "wgrad": "wgrad_kernel"}[dom]
    d = parts[dom]
    tensor_side = {"tflops": d["tflops"], "tensor_peak_tflops": peaks["bf16_tflops"],
                   "frac_of_tensor_peak": d["frac_of_peak"],
                   "frac_of_sustained_tensor_peak": round(d["tflops"] / (peaks["bf16_tflops_sustained"]
                                                                         or peaks["bf16_tflops"]), 4),
                   "ai_flop_per_byte": d["ai_flop_per_byte"], "ridge_flop_per_byte": d["ridge_flop_per_byte"],
                   "attainable_tflops": d["attainable_tflops"], "frac_of_attainable": d["frac_of_attainable"]}
    if d["bound"] == "hbm":  # algorithmic bytes per launch / launch time against the measured copy rate
        roofline = {"kernel": kernel_name, "bound": "hbm", "achieved": d["achieved_gbs"], "peak": peaks["hbm_gbs"],
                    "unit": "GB/s", "frac": round(d["achieved_gbs"] / peaks["hbm_gbs"], 4)}
    else:
        roofline = {"kernel": kernel_name, "bound": "tensor", "achieved": d["tflops"], "peak": peaks["bf16_tflops"],
                    "unit": "TFLOP/s", "frac": d["frac_of_peak"]}
    roofline.update({"traffic": recorded_traffic(kernel_name, args.workload),
                     "algorithmic_bytes": int(algo[dom]), "flops": flops[dom],
                     "peak_source": f"{peaks['source']} (MEASURED_PEAKS.json: bf16 burst, HBM copy)", **tensor_side})

    e2e = None
    if not args.no_e2e:
        ms_e2e, bi, bo = time_e2e(prob, args.e2e_steps, 1)
        if world > 1:
            ms_e2e = max_over_ranks(ms_e2e, dev)
        e2e = {"value": round(step_flops * world / (ms_e2e * 1e-3) / 1e12, 2), "unit": "TFLOP/s",
               "ms_per_step": round(ms_e2e, 3), "h2d_bytes_per_step": bi, "d2h_bytes_per_step": bo,
               "steps": args.e2e_steps,
               "overlap": "input copies, ABI calls and output copies on three streams, two device buffer sets"}

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        tf, spent, sample = oracle_sample(prob, dev, args.cpu_seconds)
        cpu = {"value": tf, "unit": "TFLOP/s", "cores": os.cpu_count(), "kind": "oracle",
               "seconds": round(spent, 2), "sample": f"whole experts, seeded order: {sample}"}
    launches = prob.launches_per_step * args.steps

    per_config = None
    if world == 1 and args.workload == "deepseek" and not args.no_per_config:
        del prob
        torch.cuda.empty_cache()
        per_config = time_per_config(dev, args, peaks)

    if rank == 0:
        line = {
            "metric": METRIC, "value": round(value, 2), "unit": "TFLOP/s", "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": round(ms_step, 4), "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
            "config": {"workload": args.workload, "description": WORKLOAD_TEXT[args.workload],
                       "flops_per_step": step_flops, "l2": "inputs larger than L2 (no flush)"
                       if args.workload not in ("tiny",) else "inputs fit in L2 (tiny)",
                       "parallelism": f"replicas x{world}", "sched": args.sched, "cta": args.cta},
            "parts": parts, "roofline": roofline, "frac_of_peak": round(value / world / peaks["bf16_tflops"], 4),
            "clocks": clocks, "e2e": e2e, "cpu_baseline": cpu, "gpu_launches": launches,
            "per_config": per_config,
        }
        print(json.dumps(line))
    if world > 1:
        torch.distributed.destroy_process_group()


def run_reference(args, world, rank):
    """The oracle, as it stands, on the host cores: each step a bounded sample of the workload."""
    if world > 1 and rank != 0:
        return
    import torch
    have_gpu = torch.cuda.is_available()
    dev = torch.device("cuda", 0) if have_gpu else torch.device("cpu")

    class Specs:
        pass

    from moe_grouped_gemm_persistent_gb300 import synth
    sp = Specs()
    sp.dspec, sp.wspec = synth.workload_specs(args.workload)
    # inputs of the sampled experts only are needed; generate them where the product would
    if sp.dspec is not None:
        sp.d = synth.make_dglu_inputs(sp.dspec, device=dev)
    if sp.wspec is not None:
        sp.w = synth.make_wgrad_inputs(sp.wspec, device=dev)
    per_step_budget = max(0.5, min(6.0, 150.0 / (args.steps + args.warmup)))
    for i in range(args.warmup):
        oracle_sample(sp, dev, per_step_budget, seed=i, max_experts=2)
    vals, secs, samples = [], 0.0, []
    for i in range(args.steps):
        tf, spent, sample = oracle_sample(sp, dev, per_step_budget, seed=1000 + i, max_experts=2)
        vals.append(tf)
        secs += spent
        samples.append(sample)
    value = statistics.median(vals)
    line = {
        "impl": "reference", "metric": METRIC, "value": round(value, 6), "unit": "TFLOP/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(secs / args.steps * 1e3, 2),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": args.workload, "description": WORKLOAD_TEXT[args.workload]},
        "cpu_baseline": {"kind": "oracle", "cores": os.cpu_count(), "value": round(value, 6), "unit": "TFLOP/s",
                         "sample": f"per step up to 2 whole experts per part (seeded): {samples[0]}"},
        "e2e": {"value": round(value, 6), "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line))


if __name__ == "__main__":
    sys.exit(main())
