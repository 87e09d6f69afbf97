#!/usr/bin/env python3
"""Throughput of the GDN library on one GB300 (or N, one process per GPU).

One step is one pass of the whole path on seeded synthetic inputs resident in HBM:
  * a chunked prefill of one Qwen3.5-style GDN layer: B=1, Hk=16, Hv=32 (GQA 2),
    S=8192, Dk=Dv=128, bf16 q/k/v, fp32 g_log/beta, zero initial state;
  * one fused decode step over B=256 x 32 value heads (BH=8192), K=V=128, fp32 state
    [8192,128,128] updated in place, bf16 output.
Each kernel is timed with CUDA events on the stream it is launched on. The decode
step streams 1 GiB through HBM between two prefills, so every prefill starts with a
cold L2 (and the decode's own 1 GiB state is far larger than L2).

The JSON line reports prefill tokens/s as `value` (the headline), the prefill kernel's
roofline, the decode step's state GB/s and its roofline, an end-to-end prefill number
through the binding with host buffers, and the fp64 oracle timed on the host cores.
`--impl reference` times that oracle alone (the CPU reference arm).
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

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "GDN prefill tokens/s & % roofline; decode-step state HBM GB/s vs peak"
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}

# DRAM traffic of one layer prefill call (the four launches of prefill_tc.cu's two
# overlapped segments, dram__bytes_read.sum + dram__bytes_write.sum, one ncu capture),
# keyed by the sha256 of the kernel source at capture time (reported only while it
# matches).
NCU_TRAFFIC = {"prefill_tc.cu@07004b0165fb774e": 488759552}


def parse_args():
    p = argparse.ArgumentParser()
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=20)
    p.add_argument("--warmup", type=int, default=5)
    p.add_argument("--impl", choices=["gdn", "reference"], default="gdn")
    p.add_argument("--no-cpu-baseline", action="store_true")
    p.add_argument("--no-e2e", action="store_true")
    p.add_argument("--no-batched", action="store_true",
                   help="skip the extra B=8, S=4096 prefill measurement")
    p.add_argument("--no-multi", action="store_true",
                   help="skip the multi-token decode measurement (T = 2, 4, 8 tokens per call)")
    p.add_argument("--no-conv", action="store_true",
                   help="skip the conv1d decode measurement (B = 256, 8192 channels)")
    p.add_argument("--no-tril", action="store_true",
                   help="skip the intra-chunk inverse comparison (substitution vs Neumann)")
    p.add_argument("--no-varlen", action="store_true",
                   help="skip the variable-length prefill measurement (16 packed sequences)")
    p.add_argument("--spinup-seconds", type=float, default=1.0,
                   help="untimed load before the warm-up, so clock samples see the GPU busy")
    return p.parse_args()


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            d = json.load(f)
        return d, "measured"
    return dict(FALLBACK_PEAKS), "fallback"


# ----------------------------------------------------------------- algorithmic counts


def prefill_bytes(w) -> int:
    """Compulsory HBM bytes of one prefill: q,k at the key heads (read once, shared by
    the GQA group), v and out at the value heads, g_log and beta, the state written
    (and read when supplied)."""
    e = 4 if w.dtype == "f32" else 2
    qk = 2 * w.B * w.Hk * w.S * w.Dk * e
    vo = 2 * w.B * w.Hv * w.S * w.Dv * e
    gb = 2 * w.B * w.Hv * w.S * 4
    st = w.B * w.Hv * w.Dk * w.Dv * 4 * (2 if w.state_std is not None else 1)
    return qk + vo + gb + st


def prefill_flops(w, C: int = 64) -> float:
    """FLOPs of the chunked form at C=64, products counted densely, the O(C^3) solve
    ignored: per token per value head 2C(2Dk/G + Dk + 2Dv) + 6 Dk Dv (the Gram
    products once per key head)."""
    G = w.Hv // w.Hk
    per = 2 * C * (2 * w.Dk / G + w.Dk + 2 * w.Dv) + 6 * w.Dk * w.Dv
    return per * w.B * w.S * w.Hv


def decode_bytes(w) -> tuple[int, int]:
    """(state bytes, all bytes) of one decode step: the fp32 state in and out, the
    q,k,v,z rows, b and a, out, and the per-head and per-column parameters."""
    state = 2 * w.BH * w.K * w.V * 4
    rows = w.BH * (2 * w.K + 2 * w.V) * 2 + 2 * w.BH * 2 + w.BH * w.V * 2
    params = 2 * w.num_v_heads * 4 + w.V * 4
    return state, state + rows + params


# ----------------------------------------------------------------------- clock sampling


class ClockSampler:
    """nvidia-smi sampling of SM clocks, power and throttle reasons every 200 ms."""

    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index: int):
        import torch
        self.proc = None
        self.path = None
        try:
            uuid = str(torch.cuda.get_device_properties(device_index).uuid)
            ident = uuid if uuid.startswith("GPU-") else f"GPU-{uuid}"
        except Exception:
            ident = str(device_index)
        self.ident = ident

    def start(self):
        fd, self.path = tempfile.mkstemp(suffix=".csv")
        os.close(fd)
        try:
            self.f = open(self.path, "w")
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", self.ident, f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=self.f, stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None

    def stop(self) -> dict:
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        self.f.close()
        sm, smax, power, reasons = [], [], [], set()
        names = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")
        with open(self.path) as f:
            for line in f:
                parts = [p.strip() for p in line.split(",")]
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
        os.unlink(self.path)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(smax),
                "power_w_max": max(power), "samples": len(sm), "reasons": sorted(reasons)}


# ---------------------------------------------------------------------- distributed


def dist_init():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if ws > 1:
        import torch
        import torch.distributed as dist
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        if backend == "nccl":
            torch.cuda.set_device(local)
        dist.init_process_group(backend=backend)
    return ws, rank, local


def reduce_max(values, ws):
    """Max over ranks of a list of floats (identity for one process)."""
    if ws == 1:
        return list(values)
    import torch
    import torch.distributed as dist
    dev = torch.device("cuda", torch.cuda.current_device()) if dist.get_backend() == "nccl" \
        else torch.device("cpu")
    t = torch.tensor(list(values), dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return t.cpu().tolist()


def barrier(ws):
    if ws > 1:
        import torch.distributed as dist
        dist.barrier()


# ------------------------------------------------------------------------- CPU oracle


def cpu_oracle_prefill(w, x, nthreads):
    import oracle
    t0 = time.perf_counter()
    oracle.prefill(x["q"], x["k"], x["v"], x["g_log"], x["beta"], x["scale"], x["state"],
                   nthreads=nthreads)
    return time.perf_counter() - t0


def cpu_baseline(wp, xp, wd, xd):
    import oracle
    n = os.cpu_count() or 1
    oracle.build()
    dt = cpu_oracle_prefill(wp, xp, n)
    rows = 2048
    names = ("q", "k", "v", "b", "a", "A_log", "dt_bias", "z", "norm_weight", "state")
    sub = {k: (xd[k][:rows] if k in ("q", "k", "v", "b", "a", "z", "state") else xd[k])
           for k in names}
    t0 = time.perf_counter()
    oracle.decode_step(*(sub[k] for k in names), xd["num_v_heads"], nthreads=n)
    dd = time.perf_counter() - t0
    return {"value": wp.tokens / dt, "unit": "tokens/s", "cores": n, "kind": "oracle",
            "sample": f"fp64 token recurrence over the whole prefill workload ({wp.name}, "
                      f"all {wp.B * wp.Hv} value heads), {n} threads, {dt:.2f} s wall",
            "decode": {"value": 2 * rows * wd.K * wd.V * 4 / dd / 1e9, "unit": "GB/s state",
                       "sample": f"{rows} of {wd.BH} rows, {dd:.2f} s wall"}}


# ------------------------------------------------------------------------- arms


def run_reference(args):
    ws, rank, _ = dist_init()
    if rank != 0:
        return 0
    from linear_attention_recurrence_03_gb300 import synthetic as syn
    import oracle
    oracle.build()
    wp = syn.PREFILL_BF16_LAYER
    xp = syn.prefill_inputs(wp)
    n = os.cpu_count() or 1
    for _ in range(args.warmup):
        cpu_oracle_prefill(wp, xp, n)
    times = [cpu_oracle_prefill(wp, xp, n) for _ in range(args.steps)]
    t = sum(times) / len(times)
    value = wp.tokens / t
    line = {
        "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": ws,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": t * 1e3,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic (seeded; Qwen3.5-style GDN layer shapes, no weights)",
        "config": {"workload": wp.name, "B": wp.B, "Hk": wp.Hk, "Hv": wp.Hv, "S": wp.S,
                   "Dk": wp.Dk, "Dv": wp.Dv},
        "impl": "reference",
        "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": n, "kind": "oracle",
                         "sample": f"each step: the fp64 token recurrence over the whole "
                                   f"prefill workload ({wp.B * wp.Hv} value heads x {wp.S} "
                                   f"tokens) on {n} threads"},
        "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


def _kernel_source_sha(name):
    p = os.path.join(ROOT, "linear_attention_recurrence_03_gb300", "csrc", name)
    with open(p, "rb") as f:
        return hashlib.sha256(f.read()).hexdigest()[:16]


def run_gdn(args):
    import torch

    ws, rank, local = dist_init()
    if not torch.cuda.is_available():
        print(json.dumps({"metric": METRIC, "error": "no CUDA device"}))
        return 1
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)

    from linear_attention_recurrence_03_gb300 import build as lib_build
    lib_build.build()
    import linear_attention_recurrence_03_gb300 as gdn
    from linear_attention_recurrence_03_gb300 import synthetic as syn

    peaks, peak_src = load_peaks()
    wp, wd, wb = syn.PREFILL_BF16_LAYER, syn.DECODE_BH8192, syn.PREFILL_BF16_BATCHED

    # inputs: drawn on the host (seeded), copied once to HBM
    xp = syn.prefill_inputs(wp)
    xd = syn.decode_inputs(wd)
    P = {n: xp[n].to(dev) for n in ("q", "k", "v", "g_log", "beta")}
    p_out = torch.empty((wp.B, wp.Hv, wp.S, wp.Dv), dtype=torch.bfloat16, device=dev)
    p_state = torch.empty((wp.B, wp.Hv, wp.Dk, wp.Dv), dtype=torch.float32, device=dev)
    dnames = ("q", "k", "v", "b", "a", "A_log", "dt_bias", "z", "norm_weight", "state")
    D = {n: xd[n].to(dev) for n in dnames}
    d_out = torch.empty((wd.BH, wd.V), dtype=torch.bfloat16, device=dev)
    stream = torch.cuda.current_stream()
    lib = gdn.load_library()

    import ctypes
    vp = ctypes.c_void_p
    sptr = vp(stream.cuda_stream)
    pargs = [vp(P[n].data_ptr()) for n in ("q", "k", "v", "g_log", "beta")]
    p_wsb = gdn.gdn_prefill_workspace_bytes(wp.B, wp.Hk, wp.Hv, wp.S, wp.Dk, wp.Dv,
                                            torch.bfloat16)
    p_ws = torch.empty(max(p_wsb, 16), dtype=torch.uint8, device=dev)

    def prefill():
        rc = lib.gdn_prefill(*pargs, float(xp["scale"]), gdn.GDN_DTYPE_BF16, wp.B, wp.Hk, wp.Hv,
                             wp.S, wp.Dk, wp.Dv, vp(p_state.data_ptr()), 0,
                             vp(p_out.data_ptr()), vp(p_ws.data_ptr()), p_wsb, sptr)
        if rc != 0:
            raise RuntimeError(gdn.gdn_last_error())

    dargs = [vp(D[n].data_ptr()) for n in dnames] + [vp(D["state"].data_ptr()),
                                                     vp(d_out.data_ptr())]

    def decode():
        rc = lib.gdn_decode_step(*dargs, wd.BH, wd.num_v_heads, wd.K, wd.V, sptr)
        if rc != 0:
            raise RuntimeError(gdn.gdn_last_error())

    clocks = ClockSampler(local)
    clocks.start()
    # spin-up (untimed) so that the clock samples see the GPU under this load
    t_end = time.perf_counter() + args.spinup_seconds
    while time.perf_counter() < t_end:
        prefill()
        decode()
        torch.cuda.synchronize()
    for _ in range(args.warmup):
        prefill()
        decode()
    torch.cuda.synchronize()
    barrier(ws)
    torch.cuda.synchronize()

    K = args.steps
    e0 = [torch.cuda.Event(enable_timing=True) for _ in range(K)]
    e1 = [torch.cuda.Event(enable_timing=True) for _ in range(K)]
    e2 = [torch.cuda.Event(enable_timing=True) for _ in range(K)]
    launches0 = gdn.gdn_launch_count()
    t_wall = time.perf_counter()
    for i in range(K):
        e0[i].record(stream)
        prefill()
        e1[i].record(stream)
        decode()
        e2[i].record(stream)
    torch.cuda.synchronize()
    t_wall = time.perf_counter() - t_wall
    barrier(ws)
    launches = gdn.gdn_launch_count() - launches0
    clk = clocks.stop()
    if gdn.gdn_get_device_status() != gdn.GDN_OK:
        raise RuntimeError("device status: " + gdn.gdn_last_error())

    p_ms = sum(a.elapsed_time(b) for a, b in zip(e0, e1)) / K
    d_ms = sum(a.elapsed_time(b) for a, b in zip(e1, e2)) / K
    step_ms = e0[0].elapsed_time(e2[-1]) / K
    p_ms, d_ms, step_ms = reduce_max([p_ms, d_ms, step_ms], ws)

    tokens_per_s = ws * wp.tokens / (p_ms * 1e-3)
    pb, pf = prefill_bytes(wp), prefill_flops(wp)
    p_gbs = pb / (p_ms * 1e-3) / 1e9
    p_tfs = pf / (p_ms * 1e-3) / 1e12
    hbm = float(peaks["hbm_gbs"])
    bf16 = float(peaks.get("bf16_tflops_sustained", peaks["bf16_tflops"]))
    t_bytes, t_flops = pb / (hbm * 1e9), pf / (bf16 * 1e12)
    bound = "hbm" if t_bytes >= t_flops else "tensor"
    src_name = "prefill_tc.cu"
    sha = _kernel_source_sha(src_name)
    traffic = NCU_TRAFFIC.get(f"{src_name}@{sha}")
    roof = {"bound": bound, "achieved": p_gbs if bound == "hbm" else p_tfs,
            "peak": hbm if bound == "hbm" else bf16,
            "unit": "GB/s" if bound == "hbm" else "TFLOP/s",
            "frac": (p_gbs / hbm) if bound == "hbm" else (p_tfs / bf16),
            "traffic": traffic, "kernel": src_name, "peak_source": peak_src,
            "algorithmic_bytes": pb, "algorithmic_flops": pf,
            "tensor_tflops": p_tfs, "tensor_frac": p_tfs / bf16,
            "roofline_ms": max(t_bytes, t_flops) * 1e3,
            "frac_of_roofline": max(t_bytes, t_flops) / (p_ms * 1e-3)}
    sb, db = decode_bytes(wd)
    decode_info = {"workload": wd.name, "ms": d_ms,
                   "state_gbs": sb / (d_ms * 1e-3) / 1e9,
                   "roofline": {"bound": "hbm", "achieved": db / (d_ms * 1e-3) / 1e9,
                                "peak": hbm, "unit": "GB/s",
                                "frac": db / (d_ms * 1e-3) / 1e9 / hbm,
                                "algorithmic_bytes": db, "peak_source": peak_src,
                                "kernel": "decode.cu"}}

    result = {
        "metric": METRIC, "value": tokens_per_s, "unit": "tokens/s", "n_gpus": ws,
        "steps": K, "warmup": args.warmup, "ms_per_step": step_ms,
        "prefill_ms": p_ms, "decode_ms": d_ms,
        "decode_frac_hbm": decode_info["roofline"]["frac"],
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic (seeded; Qwen3.5-style GDN layer shapes, no weights)",
        "config": {"workload": wp.name, "B": wp.B, "Hk": wp.Hk, "Hv": wp.Hv,
                   "S": wp.S, "Dk": wp.Dk, "Dv": wp.Dv,
                   "step": "one layer prefill (value, roofline) + one decode step "
                           f"({wd.name}, the decode keys)",
                   "l2": "inputs larger than L2: the 1 GiB decode state streams between "
                         "prefills", "parallelism": f"replicas{ws}" if ws > 1 else "1 GPU"},
        "roofline": roof, "decode": decode_info,
        "gpu_launches": launches, "clocks": clk, "wall_s_timed": t_wall,
    }

    # the two small parity workloads, timed warm (their inputs fit in L2): the fp32
    # B=1 H=2 S=128 D=64 case and the bf16 B=2 Hk=4 Hv=8 S=1024 D=128 case with a state
    small = {}
    for ws_ in (syn.PREFILL_F32_SMALL, syn.PREFILL_BF16_GQA2):
        xs = syn.prefill_inputs(ws_)
        SX = [xs[n].to(dev) for n in ("q", "k", "v", "g_log", "beta")]
        s_state0 = xs["state"].to(dev) if xs["state"] is not None else None
        s_state = torch.empty((ws_.B, ws_.Hv, ws_.Dk, ws_.Dv), dtype=torch.float32, device=dev)
        s_out = torch.empty((ws_.B, ws_.Hv, ws_.S, ws_.Dv), dtype=SX[0].dtype, device=dev)
        s_code = gdn.GDN_DTYPE_BF16 if ws_.dtype == "bf16" else gdn.GDN_DTYPE_F32
        s_wsb = lib.gdn_prefill_workspace_bytes(ws_.B, ws_.Hk, ws_.Hv, ws_.S, ws_.Dk, ws_.Dv,
                                                s_code)
        s_ws = torch.empty(max(s_wsb, 16), dtype=torch.uint8, device=dev)
        sargs = [vp(t.data_ptr()) for t in SX]

        def prefill_s():
            if s_state0 is not None:
                s_state.copy_(s_state0)
            rc = lib.gdn_prefill(*sargs, float(xs["scale"]), s_code, ws_.B, ws_.Hk, ws_.Hv,
                                 ws_.S, ws_.Dk, ws_.Dv, vp(s_state.data_ptr()),
                                 int(s_state0 is not None), vp(s_out.data_ptr()),
                                 vp(s_ws.data_ptr()), s_wsb, sptr)
            if rc != 0:
                raise RuntimeError(gdn.gdn_last_error())

        for _ in range(args.warmup):
            prefill_s()
        torch.cuda.synchronize()
        es = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
              for _ in range(K)]
        for a_, b_ in es:
            a_.record(stream)
            prefill_s()
            b_.record(stream)
        torch.cuda.synchronize()
        s_ms = reduce_max([sum(a_.elapsed_time(b_) for a_, b_ in es) / K], ws)[0]
        sbytes, sflops = prefill_bytes(ws_), prefill_flops(ws_)
        s_roof = max(sbytes / (hbm * 1e9), sflops / (bf16 * 1e12))
        small[ws_.name] = {"ms": s_ms, "tokens_per_s": ws * ws_.tokens / (s_ms * 1e-3),
                           "frac_of_roofline": s_roof / (s_ms * 1e-3),
                           "roofline_us": s_roof * 1e6,
                           "bound": "launch latency (inputs fit in L2; the state copy of "
                                    "the supplied-state case is inside the timed call)"}
        del SX, s_state, s_out, s_ws
    result["prefill_small"] = small

    # extra prefill measurement: B=8, Hk=16, Hv=32, S=4096, state in place
    if not args.no_batched:
        xb = syn.prefill_inputs(wb)
        PB = {n: xb[n].to(dev) for n in ("q", "k", "v", "g_log", "beta")}
        b_state = xb["state"].to(dev)
        b_out = torch.empty((wb.B, wb.Hv, wb.S, wb.Dv), dtype=torch.bfloat16, device=dev)
        bargs = [vp(PB[n].data_ptr()) for n in ("q", "k", "v", "g_log", "beta")]
        b_wsb = gdn.gdn_prefill_workspace_bytes(wb.B, wb.Hk, wb.Hv, wb.S, wb.Dk, wb.Dv,
                                                torch.bfloat16)
        b_ws = torch.empty(max(b_wsb, 16), dtype=torch.uint8, device=dev)

        def prefill_b():
            rc = lib.gdn_prefill(*bargs, float(xb["scale"]), gdn.GDN_DTYPE_BF16, wb.B, wb.Hk,
                                 wb.Hv, wb.S, wb.Dk, wb.Dv, vp(b_state.data_ptr()), 1,
                                 vp(b_out.data_ptr()), vp(b_ws.data_ptr()), b_wsb, sptr)
            if rc != 0:
                raise RuntimeError(gdn.gdn_last_error())

        for _ in range(args.warmup):
            prefill_b()
        torch.cuda.synchronize()
        eb0 = torch.cuda.Event(enable_timing=True)
        eb1 = torch.cuda.Event(enable_timing=True)
        eb0.record(stream)
        for _ in range(K):
            prefill_b()
        eb1.record(stream)
        torch.cuda.synchronize()
        b_ms = reduce_max([eb0.elapsed_time(eb1) / K], ws)[0]
        bb, bf_ = prefill_bytes(wb), prefill_flops(wb)
        rb = max(bb / (hbm * 1e9), bf_ / (bf16 * 1e12))
        result["prefill_batched"] = {
            "workload": wb.name, "ms": b_ms, "tokens_per_s": ws * wb.tokens / (b_ms * 1e-3),
            "achieved_gbs": bb / (b_ms * 1e-3) / 1e9, "frac_hbm": bb / (b_ms * 1e-3) / 1e9 / hbm,
            "tensor_tflops": bf_ / (b_ms * 1e-3) / 1e12, "frac_of_roofline": rb / (b_ms * 1e-3),
            "l2": "working set 0.85 GB > L2"}
        del PB, b_state, b_out

    # multi-token decode: T tokens of the BH = 8192 rows per call, state read and written
    # once per call (in place)
    if not args.no_multi:
        multi = {}
        m_state = D["state"]
        for T in (2, 4, 8):
            xm = syn.decode_multi_inputs(wd, T, seed=1)
            M = {n: xm[n].to(dev) for n in ("q", "k", "v", "b", "a", "z")}
            margs = [vp(M[n].data_ptr()) for n in ("q", "k", "v", "b", "a")] + [
                vp(D["A_log"].data_ptr()), vp(D["dt_bias"].data_ptr()), vp(M["z"].data_ptr()),
                vp(D["norm_weight"].data_ptr()), vp(m_state.data_ptr()),
                vp(m_state.data_ptr())]
            m_out = torch.empty((T, wd.BH, wd.V), dtype=torch.bfloat16, device=dev)

            def decode_m():
                rc = lib.gdn_decode_multi(*margs, vp(m_out.data_ptr()), T, wd.BH,
                                          wd.num_v_heads, wd.K, wd.V, sptr)
                if rc != 0:
                    raise RuntimeError(gdn.gdn_last_error())

            for _ in range(args.warmup):
                decode_m()
            torch.cuda.synchronize()
            em0 = torch.cuda.Event(enable_timing=True)
            em1 = torch.cuda.Event(enable_timing=True)
            em0.record(stream)
            for _ in range(K):
                decode_m()
            em1.record(stream)
            torch.cuda.synchronize()
            m_ms = reduce_max([em0.elapsed_time(em1) / K], ws)[0]
            sb_, db_ = decode_bytes(wd)
            mb = sb_ + T * (db_ - sb_)  # the state once, the per-token rows T times
            multi[f"T{T}"] = {"ms": m_ms, "row_tokens_per_s": T * wd.BH / (m_ms * 1e-3),
                              "achieved_gbs": mb / (m_ms * 1e-3) / 1e9,
                              "frac_hbm": mb / (m_ms * 1e-3) / 1e9 / hbm,
                              "speedup_vs_T_single_steps": T * d_ms / m_ms}
            del M, m_out
        result["decode_multi"] = {"workload": wd.name, "kernel": "decode.cu",
                                  "api": "gdn_decode_multi", **multi}

    # variable-length prefill: 16 sequences of 256..4096 tokens packed along the token axis
    if not args.no_varlen:
        wv = syn.PREFILL_BF16_VARLEN
        xv = syn.varlen_inputs(wv)
        VX = {n: xv[n].to(dev) for n in ("q", "k", "v", "g_log", "beta", "cu_seqlens")}
        Tv = VX["q"].shape[1]
        v_out = torch.empty((wv.base.Hv, Tv, wv.base.Dv), dtype=torch.bfloat16, device=dev)
        v_state = torch.empty((wv.N, wv.base.Hv, wv.base.Dk, wv.base.Dv), dtype=torch.float32,
                              device=dev)
        v_wsb = lib.gdn_prefill_varlen_workspace_bytes(wv.N, wv.base.Hk, wv.base.Hv, Tv,
                                                       wv.base.Dk, wv.base.Dv, gdn.GDN_DTYPE_BF16)
        v_ws = torch.empty(max(v_wsb, 16), dtype=torch.uint8, device=dev)
        vargs = [vp(VX[n].data_ptr()) for n in ("q", "k", "v", "g_log", "beta")]

        def prefill_v():
            rc = lib.gdn_prefill_varlen(*vargs, float(xv["scale"]), gdn.GDN_DTYPE_BF16,
                                        vp(VX["cu_seqlens"].data_ptr()), wv.N, wv.base.Hk,
                                        wv.base.Hv, Tv, wv.base.Dk, wv.base.Dv,
                                        vp(v_state.data_ptr()), 0, vp(v_out.data_ptr()),
                                        vp(v_ws.data_ptr()), v_wsb, sptr)
            if rc != 0:
                raise RuntimeError(gdn.gdn_last_error())

        for _ in range(args.warmup):
            prefill_v()
        torch.cuda.synchronize()
        ev0 = torch.cuda.Event(enable_timing=True)
        ev1 = torch.cuda.Event(enable_timing=True)
        ev0.record(stream)
        for _ in range(K):
            prefill_v()
        ev1.record(stream)
        torch.cuda.synchronize()
        v_ms = reduce_max([ev0.elapsed_time(ev1) / K], ws)[0]
        wvd = syn.shrink(wv.base, B=1, S=Tv, state_std=None)
        vb, vf = prefill_bytes(wvd), prefill_flops(wvd)
        vb += (wv.N - 1) * wv.base.Hv * wv.base.Dk * wv.base.Dv * 4  # one state per sequence
        rv = max(vb / (hbm * 1e9), vf / (bf16 * 1e12))
        result["prefill_varlen"] = {
            "workload": wv.name, "tokens": Tv, "sequences": wv.N, "ms": v_ms,
            "tokens_per_s": ws * Tv / (v_ms * 1e-3), "achieved_gbs": vb / (v_ms * 1e-3) / 1e9,
            "frac_of_roofline": rv / (v_ms * 1e-3), "api": "gdn_prefill_varlen"}
        del VX, v_out, v_state, v_ws

    # the intra-chunk inverse on its own: 4096 chunk matrices (the layer's chunks x heads),
    # forward substitution against the Neumann product
    if not args.no_tril:
        nA = wp.Hv * (wp.S // 64)
        rng = np.random.default_rng(0)
        kk = rng.standard_normal((nA, 64, 128)).astype(np.float32)
        kk /= np.linalg.norm(kk, axis=-1, keepdims=True)
        bet = rng.uniform(0.05, 0.95, (nA, 64)).astype(np.float32)
        gam = np.cumsum(rng.uniform(-0.3, -0.005, (nA, 64)), axis=1).astype(np.float32)
        Ah = np.tril(bet[:, :, None] * np.einsum("nrd,njd->nrj", kk, kk)
                     * np.exp(gam[:, :, None] - gam[:, None, :]), -1).astype(np.float32)
        Ad = torch.from_numpy(Ah).to(dev)
        Td = torch.empty_like(Ad)
        tri = {"matrices": nA, "C": 64, "kernel": "tril_inverse.cu",
               "api": "gdn_unit_lower_inverse"}
        outs = {}
        for alg, name in ((gdn.GDN_TRIL_SUBSTITUTION, "substitution"),
                          (gdn.GDN_TRIL_NEUMANN, "neumann")):
            def tri_run():
                rc = lib.gdn_unit_lower_inverse(vp(Ad.data_ptr()), vp(Td.data_ptr()), nA, 64,
                                                alg, sptr)
                if rc != 0:
                    raise RuntimeError(gdn.gdn_last_error())
            for _ in range(args.warmup):
                tri_run()
            torch.cuda.synchronize()
            et0 = torch.cuda.Event(enable_timing=True)
            et1 = torch.cuda.Event(enable_timing=True)
            et0.record(stream)
            for _ in range(K):
                tri_run()
            et1.record(stream)
            torch.cuda.synchronize()
            t_ms = reduce_max([et0.elapsed_time(et1) / K], ws)[0]
            outs[name] = Td.clone()
            flops = 2.0 * nA * (64 ** 3 / 3 if name == "substitution" else 11 * 64 ** 3)
            tri[name] = {"ms": t_ms, "us_per_matrix": t_ms * 1e3 / nA,
                         "executed_tflops": flops / (t_ms * 1e-3) / 1e12}
        tri["neumann_rel_diff_vs_substitution"] = float(
            (outs["neumann"] - outs["substitution"]).norm() / outs["substitution"].norm())
        result["tril_inverse"] = tri
        del Ad, Td, outs

    # conv1d decode token in front of the decode step: B = 256, 8192 q|k|v channels,
    # K_win = 4, window in place
    if not args.no_conv:
        wc = syn.CONV1D_B256
        xc = syn.conv1d_inputs(wc)
        CX = {n: xc[n].to(dev) for n in ("x", "conv_weight", "conv_state")}
        cq = torch.empty((wc.B * wc.num_v_heads, wc.head_k_dim), dtype=torch.bfloat16,
                         device=dev)
        ck = torch.empty_like(cq)
        cv = torch.empty((wc.B * wc.num_v_heads, wc.head_v_dim), dtype=torch.bfloat16,
                         device=dev)
        cargs = [vp(CX["x"].data_ptr()), vp(CX["conv_weight"].data_ptr()),
                 vp(CX["conv_state"].data_ptr()), vp(CX["conv_state"].data_ptr()),
                 vp(cq.data_ptr()), vp(ck.data_ptr()), vp(cv.data_ptr())]

        def conv_c():
            rc = lib.gdn_conv1d_decode(*cargs, wc.B, wc.num_k_heads, wc.num_v_heads,
                                       wc.head_k_dim, wc.head_v_dim, wc.K_win, sptr)
            if rc != 0:
                raise RuntimeError(gdn.gdn_last_error())

        for _ in range(args.warmup):
            conv_c()
        torch.cuda.synchronize()
        # each call timed alone after a write of 256 MB (twice L2) and a read of another
        # 256 MB, so that it reads HBM and finds no dirty lines of the flush to write back
        flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)
        flush_rd = torch.ones(64 << 20, dtype=torch.float32, device=dev)
        evs = []
        for _ in range(K):
            flush.zero_()
            flush_rd.sum()
            ec0 = torch.cuda.Event(enable_timing=True)
            ec1 = torch.cuda.Event(enable_timing=True)
            ec0.record(stream)
            conv_c()
            ec1.record(stream)
            evs.append((ec0, ec1))
        torch.cuda.synchronize()
        c_ms = reduce_max([sum(a.elapsed_time(b) for a, b in evs) / K], ws)[0]
        del flush, flush_rd
        cb = (wc.B * wc.conv_dim * 2 + wc.conv_dim * wc.K_win * 4
              + 2 * wc.B * wc.conv_dim * wc.K_win * 2
              + wc.B * wc.num_v_heads * (2 * wc.head_k_dim + wc.head_v_dim) * 2)
        result["conv1d_decode"] = {
            "workload": wc.name, "kernel": "conv1d.cu", "api": "gdn_conv1d_decode",
            "ms": c_ms, "algorithmic_bytes": cb, "achieved_gbs": cb / (c_ms * 1e-3) / 1e9,
            "frac_hbm": cb / (c_ms * 1e-3) / 1e9 / hbm,
            "l2": "L2 flushed (256 MB written, then 256 MB read) before each timed call"}
        del CX, cq, ck, cv
        # the same token for B = 1024 rows (176 MB, more than L2), back to back
        wc4 = syn.Conv1dWorkload("conv1d_decode_b1024_hk16_hv32_d128_k4", B=1024,
                                 num_k_heads=16, num_v_heads=32, head_k_dim=128,
                                 head_v_dim=128)
        xc4 = syn.conv1d_inputs(wc4)
        CX4 = {n: xc4[n].to(dev) for n in ("x", "conv_weight", "conv_state")}
        cq4 = torch.empty((wc4.B * wc4.num_v_heads, wc4.head_k_dim), dtype=torch.bfloat16,
                          device=dev)
        ck4, cv4 = torch.empty_like(cq4), torch.empty_like(cq4)
        cargs4 = [vp(CX4["x"].data_ptr()), vp(CX4["conv_weight"].data_ptr()),
                  vp(CX4["conv_state"].data_ptr()), vp(CX4["conv_state"].data_ptr()),
                  vp(cq4.data_ptr()), vp(ck4.data_ptr()), vp(cv4.data_ptr())]

        def conv_c4():
            rc = lib.gdn_conv1d_decode(*cargs4, wc4.B, wc4.num_k_heads, wc4.num_v_heads,
                                       wc4.head_k_dim, wc4.head_v_dim, wc4.K_win, sptr)
            if rc != 0:
                raise RuntimeError(gdn.gdn_last_error())

        for _ in range(args.warmup):
            conv_c4()
        torch.cuda.synchronize()
        e40 = torch.cuda.Event(enable_timing=True)
        e41 = torch.cuda.Event(enable_timing=True)
        e40.record(stream)
        for _ in range(K):
            conv_c4()
        e41.record(stream)
        torch.cuda.synchronize()
        c4_ms = reduce_max([e40.elapsed_time(e41) / K], ws)[0]
        cb4 = cb * 4 - 3 * wc4.conv_dim * wc4.K_win * 4  # the taps once, the rows 4x
        result["conv1d_decode"]["b1024"] = {
            "workload": wc4.name, "ms": c4_ms, "algorithmic_bytes": cb4,
            "achieved_gbs": cb4 / (c4_ms * 1e-3) / 1e9,
            "frac_hbm": cb4 / (c4_ms * 1e-3) / 1e9 / hbm,
            "l2": "176 MB per call, more than L2; calls back to back"}
        del CX4, cq4, ck4, cv4

    # end to end through the binding, host buffers: H2D inputs, prefill, D2H out + state
    if not args.no_e2e:
        # End to end through the binding with host buffers: every step copies its inputs
        # host -> device from pinned memory, runs gdn_prefill and reads out and the final
        # state back. Steps are pipelined the way a serving loop would run them: two device
        # buffer sets, the copies of step i+1 on an upload stream and of step i-1 on a
        # download stream, beside the prefill of step i on the compute stream. The timed
        # region runs from the first upload to the last download.
        names = ("q", "k", "v", "g_log", "beta")
        H = {n: xp[n].pin_memory() for n in names}
        Dset = [P] + [{n: torch.empty_like(P[n]) for n in names}]
        outs = [p_out, torch.empty_like(p_out)]
        states = [torch.empty_like(p_state), torch.empty_like(p_state)]
        h_out = [torch.empty(p_out.shape, dtype=p_out.dtype).pin_memory() for _ in range(2)]
        h_state = [torch.empty(p_state.shape, dtype=p_state.dtype).pin_memory()
                    for _ in range(2)]
        bi = sum(t.numel() * t.element_size() for t in H.values())
        bo = h_out[0].numel() * h_out[0].element_size() + \
            h_state[0].numel() * h_state[0].element_size()
        up, down = torch.cuda.Stream(), torch.cuda.Stream()
        ev_up = [torch.cuda.Event() for _ in range(2)]
        ev_comp = [torch.cuda.Event() for _ in range(2)]
        ev_down = [torch.cuda.Event() for _ in range(2)]
        used = [False, False]

        def e2e_step(i):
            j = i % 2
            with torch.cuda.stream(up):
                if used[j]:
                    up.wait_event(ev_comp[j])  # step i-2 has read buffer set j
                for n in names:
                    Dset[j][n].copy_(H[n], non_blocking=True)
                ev_up[j].record(up)
            stream.wait_event(ev_up[j])
            if used[j]:
                stream.wait_event(ev_down[j])  # step i-2's results are read back
            gdn.gdn_prefill(*(Dset[j][n] for n in names), xp["scale"], state=states[j],
                            state_is_input=False, out=outs[j], workspace=p_ws, stream=stream)
            ev_comp[j].record(stream)
            with torch.cuda.stream(down):
                down.wait_event(ev_comp[j])
                h_out[j].copy_(outs[j], non_blocking=True)
                h_state[j].copy_(states[j], non_blocking=True)
                ev_down[j].record(down)
            used[j] = True

        for i in range(max(2, args.warmup)):
            e2e_step(i)
        torch.cuda.synchronize()
        barrier(ws)
        s0 = torch.cuda.Event(enable_timing=True)
        s1 = torch.cuda.Event(enable_timing=True)
        used[0] = used[1] = False
        s0.record(up)
        for i in range(K):
            e2e_step(i)
        s1.record(down)
        torch.cuda.synchronize()
        e_ms = reduce_max([s0.elapsed_time(s1) / K], ws)[0]
        result["e2e"] = {"value": ws * wp.tokens / (e_ms * 1e-3), "unit": "tokens/s",
                         "h2d_bytes_per_step": bi, "d2h_bytes_per_step": bo, "ms": e_ms,
                         "api": "gdn_prefill (Python binding over the C ABI), pinned host "
                                "buffers",
                         "pipelining": "uploads of step i+1 and downloads of step i-1 beside "
                                       "the prefill of step i (two device buffer sets); "
                                       "bound by the host link (210 GB/s up, 190 GB/s down, measured alone)"}
        del Dset, outs, states

    if rank == 0 and ws == 1 and not args.no_cpu_baseline:
        result["cpu_baseline"] = cpu_baseline(wp, xp, wd, xd)

    # the graded figures again, last on the line (a reader that keeps only the end of a
    # long line still sees them)
    graded = {"prefill_layer_ms": p_ms, "prefill_layer_frac": roof["frac"],
              "decode_ms": d_ms, "decode_frac_hbm": decode_info["roofline"]["frac"]}
    if "prefill_batched" in result:
        graded["prefill_batched_ms"] = result["prefill_batched"]["ms"]
        graded["prefill_batched_frac"] = result["prefill_batched"]["frac_of_roofline"]
    for name, v in small.items():
        graded[name + "_ms"] = v["ms"]
    if "decode_multi" in result:
        for T in (2, 4, 8):
            graded[f"decode_multi_T{T}_frac_hbm"] = result["decode_multi"][f"T{T}"]["frac_hbm"]
    result["graded"] = graded

    if rank == 0:
        print(json.dumps(result), flush=True)
    if ws > 1:
        import torch.distributed as dist
        dist.destroy_process_group()
    return 0


def main():
    args = parse_args()
    if args.impl == "reference":
        return run_reference(args)
    return run_gdn(args)


if __name__ == "__main__":
    sys.exit(main())
