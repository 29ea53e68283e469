"""Benchmark of the chunked gated delta rule forward on GB300.

One step = one full forward (every kernel of the path) over the workload's
synthetic batch.  Default workload: GDN, bf16, B=4, T=32768, H=HV=32,
K=V=128, chunk 64, in-kernel QK L2 norm, no initial state, final state out.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                    [--workload NAME] [--algo auto|chunked|fused]

Prints one JSON line (rank 0).  The metric is tokens/s (B*T tokens per step,
all heads).  ``value`` times the forward with inputs resident in HBM (inputs
are 4.3 GB, far larger than the 129 MB L2, so no flush is needed); ``e2e``
times the public host-buffer call (pinned host -> device copies, the forward,
device -> host copies of o and ht) every step.  ``--impl reference`` times the
fp64 CPU oracle on a bounded sample of the same workload.  On one GPU the line
also carries ``bwd``: the backward timed on the KDA varlen workload (lengths
700/324/3072/12288, HV 32, K 128, V 256), against the FP32 CUDA-core peak;
``decode``: one decode step of the per-token form (256 sequences x 1 token,
32 heads, K = V = 128, state in place) against HBM bandwidth; and ``split``:
the intra-sequence split on one 32768-token fp32 sequence with 4 heads,
beside the unsplit chunked form; and ``configs``: the forward on each other
configuration (fp32 T=128 K=V=64; bf16 K=V=60 with grouped values; the varlen
400/624 pair; the KDA varlen case), each against the method's roofline, with
its chunked-form kernels timed one by one where that form serves it.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import torch  # noqa: E402

import workloads as wl  # noqa: E402

METRIC = "gated-delta-rule fwd tokens/s on 1 GB300; achieved % of HBM/tensor roofline"
UNIT = "tokens/s"
NOMINAL_HBM_GBS = 8000.0   # bytes roofline of the method's stated definition
FALLBACK = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0}


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            p = json.load(f)
        return {"hbm_gbs": float(p["hbm_gbs"]), "bf16_tflops": float(p["bf16_tflops"]),
                "bf16_tflops_sustained": float(p.get("bf16_tflops_sustained", p["bf16_tflops"])),
                "source": "measured"}
    return {**FALLBACK, "bf16_tflops_sustained": 1700.0, "source": "fallback"}


def recorded_traffic(w: wl.Workload, kernel: str):
    """DRAM bytes per launch from the committed ncu record, if it still describes
    the kernel as built (same source hash) and this workload; else None."""
    path = os.path.join(ROOT, "profiles", "gdr_fused_kernel_traffic.json")
    if kernel != "gdr_fused" or w.name != wl.GDN_BF16_LARGE.name or not os.path.exists(path):
        return None
    import hashlib
    rec = json.load(open(path))
    h = hashlib.sha256()
    for f in ("gdr_fused.cu", "gdr_fused_common.cuh", "gdr_sm100.cuh"):
        with open(os.path.join(ROOT, "chunked_gated_delta_08_gb300", "csrc", f), "rb") as fh:
            h.update(fh.read())
    if h.hexdigest() != rec.get("kernel_source_sha256"):
        return None
    return rec.get("traffic_bytes_per_launch_bench_workload")


# ------------------------------------------------------------------ algorithmic work
def algorithmic_bytes(w: wl.Workload) -> int:
    """Inputs read once, outputs written once (per step, whole workload)."""
    e = 2 if w.dtype == torch.bfloat16 else 4
    tok = w.B * w.T
    qk = 2 * tok * w.H * w.K * e
    vo = 2 * tok * w.HV * w.V * e
    g = tok * w.HV * (w.K if w.gate_per_k else 1) * 4
    beta = tok * w.HV * e
    state = w.N * w.HV * w.K * w.V * 4 * ((1 if w.h0_scale is not None else 0) + 1)
    return qk + vo + g + beta + state


def algorithmic_flops(w: wl.Workload) -> int:
    """3CK + 2CV + 6KV per token per value head (causal triangles counted as half)."""
    C = w.chunk_size
    return w.B * w.T * w.HV * (3 * C * w.K + 2 * C * w.V + 6 * w.K * w.V)


def bwd_algorithmic_flops(w: wl.Workload) -> int:
    """10CK + 5CV + 16KV per token per value head: the chunk-form backward's
    products (forward recompute included, causal triangles counted as half)."""
    C = w.chunk_size
    return w.B * w.T * w.HV * (10 * C * w.K + 5 * C * w.V + 16 * w.K * w.V)


def fp32_alu_tflops(sm_mhz: float) -> float:
    """FP32 FMA peak: 152 SMs x 128 lanes x 2 FLOP x the SM clock."""
    return 152 * 128 * 2 * sm_mhz * 1e6 / 1e12


# ------------------------------------------------------------------ clocks
class ClockSampler:
    """Samples nvidia-smi clocks and throttle reasons while the timed region runs."""
    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.rows = []
        self.proc = None
        self.thread = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", f"--id={self.index}", f"--query-gpu={self.Q}",
                                          "--format=csv,noheader,nounits", "-lms", "100"],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
            time.sleep(0.3)
        except (OSError, FileNotFoundError):
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) >= 9:
                self.rows.append(parts)

    def __exit__(self, *exc):
        if self.proc is not None:
            time.sleep(0.2)
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
        return False

    def summary(self):
        if not self.rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"], "samples": 0}
        sm = [float(r[1]) for r in self.rows if r[1].replace(".", "").isdigit()]
        mx = [float(r[2]) for r in self.rows if r[2].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in self.rows for i in range(4) if r[5 + i].lower() == "active"})
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": reasons, "samples": len(self.rows)}


# ------------------------------------------------------------------ distributed plumbing
def dist_setup(n_gpus: int):
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        if torch.cuda.is_available():
            torch.cuda.set_device(local)
        dist.init_process_group(backend)
    elif torch.cuda.is_available():
        torch.cuda.set_device(local)
    return world, rank, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(x: float, world: int) -> float:
    if world <= 1:
        return x
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64, device="cuda" if torch.cuda.is_available() else "cpu")
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


# ------------------------------------------------------------------ CPU oracle legs
def oracle_sample(w: wl.Workload, x: dict, n_units: int, threads: int):
    """Runs the oracle over ``n_units`` whole (sequence, head) units; returns
    (tokens equivalent, seconds, sample description)."""
    import oracle
    units = [(i % w.N, (i * 7) % w.HV) for i in range(n_units)]
    t0 = time.perf_counter()
    oracle.gdr_fwd_ref_units(x["q"], x["k"], x["v"], x["g"], x["beta"], units, h0=x["h0"],
                             cu_seqlens=x["cu_seqlens"], use_qk_l2norm=w.use_qk_l2norm, threads=threads)
    dt = time.perf_counter() - t0
    lens = w.lengths if w.lengths else [w.T] * w.N
    token_heads = sum(lens[n] for n, _ in units)
    return token_heads / w.HV, dt, (f"{n_units} whole (sequence, value head) units = {token_heads} token-heads "
                                    f"of {w.name}; tokens counted as token-heads / HV")


def run_reference(args, w, world, rank):
    if rank != 0:
        return
    x = wl.make_inputs(w)
    cores = os.cpu_count() or 1
    n_units = max(1, min(cores, w.N * w.HV))
    for _ in range(args.warmup):
        oracle_sample(w, x, n_units, cores)
    tok = 0.0
    secs = 0.0
    desc = ""
    for _ in range(args.steps):
        t, dt, desc = oracle_sample(w, x, n_units, cores)
        tok += t
        secs += dt
    value = tok / secs
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * secs / args.steps,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic", "config": config_of(w, args),
            "cpu_baseline": {"value": value, "unit": UNIT, "cores": cores, "kind": "oracle", "sample": desc},
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def config_of(w, args):
    return {"workload": w.name, "B": w.B, "T": w.T, "H": w.H, "HV": w.HV, "K": w.K, "V": w.V,
            "chunk_size": w.chunk_size, "varlen_lengths": list(w.lengths) if w.lengths else None,
            "gate": "per_key" if w.gate_per_k else "scalar", "use_qk_l2norm": w.use_qk_l2norm,
            "initial_state": w.h0_scale is not None, "final_state": True, "algo": args.algo,
            "l2_flush": "inputs larger than L2 (no flush)", "parallelism": f"replicas{args.gpus}"}


# ------------------------------------------------------------------ our arm
def stage_timings(gdr, w, d, steps):
    """Per-kernel durations of the chunked form, CUDA events on the launching stream."""
    s = torch.cuda.current_stream()
    names = (["chunk_index"] if w.lengths else []) + ["prepare", "fwd_h", "fwd_o"]
    tot = {n: 0.0 for n in names}
    import ctypes
    desc = gdr.make_desc(d["q"], d["v"], d["g"], d["cu_seqlens"], "chunked")
    sz = gdr.chunked_sizes(desc, w.chunk_size, w.lengths is not None)
    f32 = dict(dtype=torch.float32, device="cuda")
    B, T, HV, K, V, N = w.B, w.T, w.HV, w.K, w.V, w.N
    ci = torch.empty(max(1, sz.nt_max), 2, dtype=torch.int64, device="cuda")
    co = torch.empty(N + 1, dtype=torch.int64, device="cuda")
    gcum = torch.empty(*d["g"].shape, **f32)
    wt = torch.empty(B, T, HV, K, **f32)
    u = torch.empty(B, T, HV, V, **f32)
    h = torch.empty(sz.nt_max, HV, K, V, **f32)
    vn = torch.empty(B, T, HV, V, **f32)
    ht = torch.empty(N, HV, K, V, **f32)
    o = torch.empty(B, T, HV, V, dtype=d["q"].dtype, device="cuda")
    P = gdr._ptr
    sp = gdr._stream_ptr(s)
    cu = d["cu_seqlens"]
    C, l2 = w.chunk_size, int(w.use_qk_l2norm)
    lib = gdr.lib()
    for _ in range(steps):
        ev = [torch.cuda.Event(enable_timing=True) for _ in range(len(names) + 1)]
        ev[0].record(s)
        i = 1
        if w.lengths:
            gdr._check(lib.gdr_chunk_index(ctypes.byref(desc), P(cu), C, P(ci), P(co), sp))
            ev[i].record(s)
            i += 1
        gdr._check(lib.gdr_chunk_prepare(ctypes.byref(desc), P(d["k"]), P(d["v"]), P(d["g"]), P(d["beta"]), P(cu),
                                         P(ci) if cu is not None else None, C, l2, P(gcum), P(wt), P(u), sp))
        ev[i].record(s)
        i += 1
        gdr._check(lib.gdr_chunk_fwd_h(ctypes.byref(desc), P(d["k"]), P(wt), P(u), P(gcum), P(d["h0"]), P(cu),
                                       P(co) if cu is not None else None, C, l2, P(h), P(vn), P(ht), sp))
        ev[i].record(s)
        i += 1
        gdr._check(lib.gdr_chunk_fwd_o(ctypes.byref(desc), P(d["q"]), P(d["k"]), P(vn), P(h), P(gcum), P(cu),
                                       P(ci) if cu is not None else None, C, l2, P(o), sp))
        ev[i].record(s)
        s.synchronize()
        for j, n in enumerate(names):
            tot[n] += ev[j].elapsed_time(ev[j + 1])
    avg_ms = {n: t / steps for n, t in tot.items()}
    # bytes each kernel must move through its own interface (fp32 intermediates)
    e = 2 if w.dtype == torch.bfloat16 else 4
    tok, gw = B * T, (K if w.gate_per_k else 1)
    nt = sz.nt_max
    kbytes = {
        "chunk_index": 8 * (N + 1) + 16 * nt,
        "prepare": tok * w.H * K * e + tok * HV * (V * e + gw * 4 + e) + tok * HV * (K + V + gw) * 4,
        "fwd_h": tok * w.H * K * e + tok * HV * (K + V + gw) * 4 + nt * HV * K * V * 4 + tok * HV * V * 4,
        "fwd_o": 2 * tok * w.H * K * e + tok * HV * (V * 4 + gw * 4 + V * e) + nt * HV * K * V * 4,
    }
    return avg_ms, kbytes


def bwd_measurement(gdr, steps: int, warmup: int = 3):
    """The backward on the KDA varlen workload (its graded configuration),
    inputs resident, CUDA events on the launching stream."""
    w = wl.KDA_BF16_VARLEN
    x = {k: (None if t is None else t.cuda()) for k, t in wl.make_inputs(w).items()}
    s = torch.cuda.current_stream()
    outs = (torch.empty_like(x["q"]), torch.empty_like(x["k"]), torch.empty_like(x["v"]),
            torch.empty_like(x["g"]), torch.empty_like(x["beta"]),
            torch.empty(w.N, w.HV, w.K, w.V, dtype=torch.float32, device="cuda"))

    def call():
        gdr.bwd(x["q"], x["k"], x["v"], x["g"], x["beta"], x["do"], dht=x["dht"], h0=x["h0"],
                cu_seqlens=x["cu_seqlens"], chunk_size=w.chunk_size, use_qk_l2norm=w.use_qk_l2norm, out=outs)

    for _ in range(warmup):
        call()
    torch.cuda.synchronize()
    l0 = gdr.launch_count()
    with ClockSampler(torch.cuda.current_device()) as clk:
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(s)
        for _ in range(steps):
            call()
        e1.record(s)
        torch.cuda.synchronize()
    if gdr.device_status() != 0:
        raise RuntimeError(f"device status after the backward: {gdr.last_error()}")
    ms = e0.elapsed_time(e1) / steps
    flops = bwd_algorithmic_flops(w)
    clocks = clk.summary()
    sm_mhz = clocks.get("sm_max_mhz") or 2070.0
    peak = fp32_alu_tflops(sm_mhz)
    achieved = flops / (ms * 1e-3) / 1e12
    return {"workload": w.name, "value": w.B * w.T / (ms * 1e-3), "unit": UNIT, "ms_per_step": ms, "steps": steps,
            "gpu_launches_per_step": (gdr.launch_count() - l0) / steps, "clocks": clocks,
            "roofline": {"bound": "alu", "kernel": "whole backward", "achieved": achieved,
                         "peak": peak, "unit": "TFLOP/s", "frac": achieved / peak, "traffic": None,
                         "algorithmic_flops_per_step": flops,
                         "peak_source": "FP32 FMA: 152 SMs x 128 lanes x 2 x max SM clock"}}


def decode_measurement(gdr, steps: int, warmup: int = 3):
    """One decode step (the per-token form) on 256 sequences x 1 token, state
    updated in place; L2 is flushed between steps by a 256 MB write."""
    w = wl.GDN_BF16_DECODE
    x = {k: (None if t is None else t.cuda()) for k, t in wl.make_inputs(w).items()}
    state = x["h0"].clone()
    o = torch.empty(w.B, w.T, w.HV, w.V, dtype=w.dtype, device="cuda")
    flush = torch.empty(64 << 20, dtype=torch.float32, device="cuda")
    s = torch.cuda.current_stream()

    def call():
        gdr.fwd(x["q"], x["k"], x["v"], x["g"], x["beta"], h0=state, use_qk_l2norm=True, algo="recurrent",
                out=o, final_state=state)

    for _ in range(warmup):
        call()
    torch.cuda.synchronize()
    l0 = gdr.launch_count()
    ms = []
    for _ in range(steps):
        flush.zero_()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(s)
        call()
        e1.record(s)
        torch.cuda.synchronize()
        ms.append(e0.elapsed_time(e1))
    if gdr.device_status() != 0:
        raise RuntimeError(f"device status after decode: {gdr.last_error()}")
    avg = statistics.mean(ms)
    byt = algorithmic_bytes(w)
    pk = peaks()
    achieved = byt / (avg * 1e-3) / 1e9
    return {"workload": w.name, "value": w.B * w.T / (avg * 1e-3), "unit": UNIT, "ms_per_step": avg,
            "steps": steps, "gpu_launches_per_step": (gdr.launch_count() - l0) / steps,
            "l2_flush": "256 MB write between steps",
            "roofline": {"bound": "hbm", "kernel": "recurrent_fwd_kernel", "achieved": achieved,
                         "peak": pk["hbm_gbs"], "unit": "GB/s", "frac": achieved / pk["hbm_gbs"], "traffic": None,
                         "algorithmic_bytes_per_launch": byt}}


def split_measurement(gdr, steps: int, warmup: int = 3):
    """The intra-sequence split against the unsplit chunked form on one long
    sequence with four heads (fp32), inputs resident, CUDA events."""
    w = wl.GDN_FP32_LONG_FEW
    x = {k: (None if t is None else t.cuda()) for k, t in wl.make_inputs(w).items()}
    s = torch.cuda.current_stream()
    res = {}
    for algo in ("split", "chunked"):
        def call():
            gdr.fwd(x["q"], x["k"], x["v"], x["g"], x["beta"], h0=x["h0"], use_qk_l2norm=True, algo=algo)
        for _ in range(warmup):
            call()
        torch.cuda.synchronize()
        l0 = gdr.launch_count()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(s)
        for _ in range(steps):
            call()
        e1.record(s)
        torch.cuda.synchronize()
        res[algo] = (e0.elapsed_time(e1) / steps, (gdr.launch_count() - l0) / steps)
    if gdr.device_status() != 0:
        raise RuntimeError(f"device status after split: {gdr.last_error()}")
    ms, launches = res["split"]
    byt = algorithmic_bytes(w)
    pk = peaks()
    achieved = byt / (ms * 1e-3) / 1e9
    return {"workload": w.name, "value": w.B * w.T / (ms * 1e-3), "unit": UNIT, "ms_per_step": ms,
            "steps": steps, "gpu_launches_per_step": launches, "chunked_ms_per_step": res["chunked"][0],
            "speedup_vs_chunked": res["chunked"][0] / ms,
            "roofline": {"bound": "hbm", "kernel": "whole split forward", "achieved": achieved,
                         "peak": pk["hbm_gbs"], "unit": "GB/s", "frac": achieved / pk["hbm_gbs"], "traffic": None,
                         "algorithmic_bytes_per_launch": byt}}


def configs_measurement(gdr, steps: int, warmup: int = 3):
    """The forward on every other configuration (the fp32 small case, K = V = 60
    with grouped values, the varlen pair, the KDA varlen case), each with its
    roofline by the method's definition and against measured HBM, and, where
    the chunked form serves it, the duration of each of its kernels.  Inputs
    resident; L2 flushed by a 256 MB write before every timed step (these
    inputs fit in L2)."""
    pk = peaks()
    flush = torch.empty(64 << 20, dtype=torch.float32, device="cuda")
    s = torch.cuda.current_stream()
    out = {}
    for w in (wl.GDN_FP32_SMALL, wl.GDN_BF16_GVA_K60, wl.GDN_BF16_VARLEN, wl.KDA_BF16_VARLEN):
        x = wl.make_inputs(w)
        d = {k: (None if t is None else t.cuda()) for k, t in x.items()}
        o = torch.empty(w.B, w.T, w.HV, w.V, dtype=w.dtype, device="cuda")
        ht = torch.empty(w.N, w.HV, w.K, w.V, dtype=torch.float32, device="cuda")

        def call():
            gdr.fwd(d["q"], d["k"], d["v"], d["g"], d["beta"], h0=d["h0"], cu_seqlens=d["cu_seqlens"],
                    chunk_size=w.chunk_size, use_qk_l2norm=w.use_qk_l2norm, out=o, final_state=ht)

        for _ in range(warmup):
            call()
        torch.cuda.synchronize()
        l0 = gdr.launch_count()
        ms = []
        for _ in range(steps):
            flush.zero_()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(s)
            call()
            e1.record(s)
            torch.cuda.synchronize()
            ms.append(e0.elapsed_time(e1))
        launches = (gdr.launch_count() - l0) / steps
        if gdr.device_status() != 0:
            raise RuntimeError(f"device status after {w.name}: {gdr.last_error()}")
        avg = statistics.median(ms)
        byt, flops = algorithmic_bytes(w), algorithmic_flops(w)
        spec_us = max(byt / (NOMINAL_HBM_GBS * 1e9), flops / (pk["bf16_tflops"] * 1e12)) * 1e6
        kernels = None
        if launches > 1.0 + 1e-9:
            kernels, _ = stage_timings(gdr, w, d, 3)
        out[w.name] = {"value": w.B * w.T / (avg * 1e-3), "unit": UNIT, "ms_per_step": avg, "steps": steps,
                       "gpu_launches_per_step": launches, "form": "fused" if launches <= 1.0 + 1e-9 else "chunked",
                       "l2_flush": "256 MB write before every step", "kernel_ms": kernels,
                       "roofline_spec": {"bytes": byt, "flops": flops, "roofline_us": spec_us,
                                         "frac": spec_us / (avg * 1e3),
                                         "frac_of_measured_hbm": (byt / (pk["hbm_gbs"] * 1e9)) / (avg * 1e-3)}}
        del d, o, ht
    return out


def profile_pass(gdr):
    """Every form once on a mid-size workload, for a per-kernel ncu capture:
    fused, chunked and split forwards on one 32768-token GDN sequence with 32
    heads; the recurrent decode step; the KDA backward on one 8192-token
    sequence.  Inputs are freed between forms so a multi-pass capture saves and
    restores little device memory."""
    runs = []
    w = wl.GDN_BF16_PROFILE
    x = {k: (None if t is None else t.cuda()) for k, t in wl.make_inputs(w).items()}
    for algo in ("fused", "chunked", "split"):
        gdr.fwd(x["q"], x["k"], x["v"], x["g"], x["beta"], h0=x["h0"], use_qk_l2norm=True, algo=algo)
        runs.append(f"{w.name}:{algo}")
    del x
    torch.cuda.synchronize()
    torch.cuda.empty_cache()
    w = wl.GDN_BF16_DECODE
    x = {k: (None if t is None else t.cuda()) for k, t in wl.make_inputs(w).items()}
    gdr.fwd(x["q"], x["k"], x["v"], x["g"], x["beta"], h0=x["h0"], use_qk_l2norm=True, algo="recurrent",
            final_state=x["h0"])
    runs.append(f"{w.name}:recurrent")
    del x
    torch.cuda.synchronize()
    torch.cuda.empty_cache()
    w = wl.KDA_BF16_PROFILE
    x = {k: (None if t is None else t.cuda()) for k, t in wl.make_inputs(w).items()}
    gdr.bwd(x["q"], x["k"], x["v"], x["g"], x["beta"], x["do"], dht=x["dht"], h0=x["h0"],
            cu_seqlens=x["cu_seqlens"], use_qk_l2norm=True)
    runs.append(f"{w.name}:bwd")
    torch.cuda.synchronize()
    if gdr.device_status() != 0:
        raise RuntimeError(f"device status after the profile pass: {gdr.last_error()}")
    return {"runs": runs, "launches": gdr.launch_count()}


def run_ours(args, w, world, rank, local):
    import chunked_gated_delta_08_gb300 as gdr
    pk = peaks()
    x = wl.make_inputs(w)
    d = {k: (None if t is None else t.cuda()) for k, t in x.items()}
    s = torch.cuda.current_stream()
    o = torch.empty(w.B, w.T, w.HV, w.V, dtype=w.dtype, device="cuda")
    ht = torch.empty(w.N, w.HV, w.K, w.V, dtype=torch.float32, device="cuda")

    def step():
        gdr.fwd(d["q"], d["k"], d["v"], d["g"], d["beta"], h0=d["h0"], cu_seqlens=d["cu_seqlens"],
                chunk_size=w.chunk_size, use_qk_l2norm=w.use_qk_l2norm, algo=args.algo, out=o, final_state=ht)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    if gdr.device_status() != 0:
        raise RuntimeError(f"device status after warm-up: {gdr.last_error()}")

    # ---- timed region: inputs resident in HBM
    launches0 = gdr.launch_count()
    barrier(world)
    torch.cuda.synchronize()
    with ClockSampler(local) as clk:
        evs = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps + 1)]
        evs[0].record(s)
        for i in range(args.steps):
            step()
            evs[i + 1].record(s)
        torch.cuda.synchronize()
    barrier(world)
    launches = gdr.launch_count() - launches0
    step_ms = [evs[i].elapsed_time(evs[i + 1]) for i in range(args.steps)]
    total_s = max_over_ranks(sum(step_ms) / 1e3, world)
    tokens = w.B * w.T
    value = world * tokens * args.steps / total_s
    ms_per_step = 1e3 * total_s / args.steps
    if gdr.device_status() != 0:
        raise RuntimeError(f"device status after timed region: {gdr.last_error()}")

    # ---- dominant kernel and roofline
    byt, flops = algorithmic_bytes(w), algorithmic_flops(w)
    launches_per_step = launches / args.steps
    if launches_per_step <= 1.0 + 1e-9:
        kname, kms, kbytes = "gdr_fused", statistics.mean(step_ms), byt
    else:
        avg_ms, kb = stage_timings(gdr, w, d, max(2, min(args.steps, 5)))
        kname = max(avg_ms, key=avg_ms.get)
        kms, kbytes = avg_ms[kname], kb[kname]
    achieved = kbytes / (kms * 1e-3) / 1e9
    roofline = {"bound": "hbm", "kernel": kname, "achieved": achieved, "peak": pk["hbm_gbs"], "unit": "GB/s",
                "frac": achieved / pk["hbm_gbs"], "traffic": recorded_traffic(w, kname), "peak_source": pk["source"],
                "algorithmic_bytes_per_launch": kbytes, "avg_launch_ms": kms}
    spec_us = max(byt / (NOMINAL_HBM_GBS * 1e9), flops / (pk["bf16_tflops"] * 1e12)) * 1e6
    roofline_spec = {"definition": "max(bytes / 8 TB/s, FLOPs / dense bf16 peak) for the whole step",
                     "bytes": byt, "flops": flops, "roofline_us": spec_us, "step_us": ms_per_step * 1e3,
                     "frac": spec_us / (ms_per_step * 1e3),
                     "frac_of_measured_hbm": (byt / (pk["hbm_gbs"] * 1e9)) / (ms_per_step * 1e-3)}

    # ---- end to end through the host-buffer call
    pinned = {k: (None if t is None else t.pin_memory()) for k, t in x.items()}
    bufs = {}
    o_h = torch.empty(o.shape, dtype=o.dtype, pin_memory=True)
    ht_h = torch.empty(ht.shape, dtype=ht.dtype, pin_memory=True)

    def e2e_step():
        gdr.fwd_host(pinned["q"], pinned["k"], pinned["v"], pinned["g"], pinned["beta"], h0=pinned["h0"],
                     cu_seqlens=pinned["cu_seqlens"], chunk_size=w.chunk_size, use_qk_l2norm=w.use_qk_l2norm,
                     algo=args.algo, out_host=o_h, final_state_host=ht_h, dev_buffers=bufs)

    e2e_step()
    barrier(world)
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    n_e2e = max(1, min(args.steps, 5))
    for _ in range(n_e2e):
        e2e_step()
    e2e_s = max_over_ranks((time.perf_counter() - t0) / n_e2e, world)
    h2d = sum(t.numel() * t.element_size() for t in pinned.values() if t is not None)
    d2h = o_h.numel() * o_h.element_size() + ht_h.numel() * ht_h.element_size()
    del bufs

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        cores = os.cpu_count() or 1
        tok_s, dt, desc = oracle_sample(w, x, max(1, min(cores, w.N * w.HV)), cores)
        cpu = {"value": tok_s / dt, "unit": UNIT, "cores": cores, "kind": "oracle", "sample": desc}

    bwd = decode = None
    if rank == 0 and world == 1 and not args.no_bwd:
        bwd = bwd_measurement(gdr, steps=max(1, min(args.steps, 5)))
    if rank == 0 and world == 1 and not args.no_decode:
        decode = decode_measurement(gdr, steps=max(3, min(args.steps, 20)))
    split = None
    if rank == 0 and world == 1 and not args.no_split:
        split = split_measurement(gdr, steps=max(1, min(args.steps, 3)))
    configs = None
    if rank == 0 and world == 1 and not args.no_configs:
        configs = configs_measurement(gdr, steps=max(3, min(args.steps, 10)))

    if rank == 0:
        line = {"metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
                "warmup": args.warmup, "ms_per_step": ms_per_step, "higher_is_better": True, "scaling": "weak",
                "vs_baseline": None, "dtype": "bf16" if w.dtype == torch.bfloat16 else "f32",
                "data": "synthetic", "config": config_of(w, args), "clocks": clk.summary(),
                "e2e": {"value": world * tokens / e2e_s, "unit": UNIT, "h2d_bytes_per_step": h2d,
                        "d2h_bytes_per_step": d2h},
                "gpu_launches": launches, "roofline": roofline, "roofline_spec": roofline_spec,
                "cpu_baseline": cpu, "step_ms": {"min": min(step_ms), "median": statistics.median(step_ms)},
                "bwd": bwd, "decode": decode, "split": split, "configs": configs}
        print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=10)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default=wl.GDN_BF16_LARGE.name, choices=sorted(wl.BY_NAME))
    ap.add_argument("--algo", default="auto", choices=["auto", "chunked", "fused"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-bwd", action="store_true", help="skip the backward measurement")
    ap.add_argument("--no-decode", action="store_true", help="skip the decode-step measurement")
    ap.add_argument("--no-split", action="store_true", help="skip the intra-sequence split measurement")
    ap.add_argument("--no-configs", action="store_true", help="skip the forward on the other configurations")
    ap.add_argument("--mode", default="fwd", choices=["fwd", "bwd", "decode", "split", "configs", "profile"],
                    help="bwd / decode: run only that measurement and print it alone")
    args = ap.parse_args()
    args.warmup = max(3, args.warmup)  # at least three untimed warm-up steps
    w = wl.BY_NAME[args.workload]
    if args.mode != "fwd":  # one measurement alone (used for the profiles); one GPU
        import chunked_gated_delta_08_gb300 as gdr
        if args.mode == "profile":
            print(json.dumps({"mode": "profile", **profile_pass(gdr)}), flush=True)
            return
        fn = {"bwd": bwd_measurement, "decode": decode_measurement, "split": split_measurement,
              "configs": configs_measurement}[args.mode]
        res = fn(gdr, steps=args.steps, warmup=args.warmup)
        print(json.dumps({"mode": args.mode, **res}), flush=True)
        return
    world, rank, local = dist_setup(args.gpus)
    if args.impl == "reference":
        run_reference(args, w, world, rank)
    else:
        run_ours(args, w, world, rank, local)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
