#!/usr/bin/env python
"""Throughput of the single-GPU MoE layer forward (libmoe on B300, sm_103a).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME] [--impl b300|reference]

One step = one pass of the whole layer (router, dispatch, grouped SwiGLU
experts, combine + statistics) over one batch of T tokens whose inputs are
already resident in HBM.  Each step takes the next of several token batches
so the working set of consecutive steps exceeds L2 (126 MB); the expert
weights alone are larger than L2 on every workload but the tiny one.
Prints one JSON line (rank 0).  Under torchrun every rank runs its own
replica (independent batches, no collective on the data path): weak scaling.

The default workload is the largest one (stress_bf16: T=65536, h=4096, E=64,
k=6, d_e=1408).  `value` is the median of --repeats regions of exactly K
steps, each a CUDA-graph replay of the whole layer.  The stage breakdown is
device time: each stage is captured as its own graph, and the stage graphs
are replayed in layer order with events between them.  With one GPU the line
also carries `per_config`: value, stages and roofline of every other
workload, measured the same way in the same run.

--impl reference times the plain CPU oracle (oracle/) on the host cores on
bounded samples of the same workload.
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
import time

import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from mixture_experts_layer_84_b300 import synth  # noqa: E402
from mixture_experts_layer_84_b300 import workloads as W  # noqa: E402

METRIC = "MoE-layer tokens/s on 1 B300; dispatch/combine %HBM BW; expert GEMM %TC peak"
L2_BYTES = 126 * 1024 * 1024
FALLBACK_PEAKS = {"hbm_gbs": 6400.0, "bf16_tflops": 1800.0, "bf16_tflops_sustained": 1400.0}
GEMM_SOURCES = ["mixture_experts_layer_84_b300/csrc/ffn_tc.cu", "mixture_experts_layer_84_b300/csrc/ptx.cuh"]


# ----------------------------------------------------------------------------- ranks

def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def init_dist(backend: str):
    ws, rank, local = dist_env()
    if ws > 1 and not torch.distributed.is_initialized():
        os.environ.setdefault("MASTER_ADDR", "127.0.0.1")
        torch.distributed.init_process_group(backend)
    return ws, rank, local


def barrier(device=None):
    if torch.distributed.is_available() and torch.distributed.is_initialized():
        if device is not None and device.type == "cuda":
            torch.distributed.barrier(device_ids=[device.index])
        else:
            torch.distributed.barrier()
    if device is not None and device.type == "cuda":
        torch.cuda.synchronize(device)


def max_over_ranks(x: float, device) -> float:
    """The largest value of x over all ranks (x itself when not distributed)."""
    if not (torch.distributed.is_available() and torch.distributed.is_initialized()):
        return float(x)
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return float(t.item())


def weak_scaling_value(tokens_per_rank_step: int, steps: int, n_ranks: int, max_seconds: float) -> float:
    """Whole-job tokens/s: every rank processed its own batches in the slowest rank's time."""
    return tokens_per_rank_step * steps * n_ranks / max_seconds


# ----------------------------------------------------------------------------- peaks, clocks

def measured_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as fh:
            d = json.load(fh)
        return {k: float(d[k]) for k in FALLBACK_PEAKS}, "measured"
    return dict(FALLBACK_PEAKS), "fallback"


class ClockSampler:
    """nvidia-smi clock/throttle samples of one GPU while a region runs."""
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device):
        self.proc = None
        try:
            self.uuid = str(torch.cuda.get_device_properties(device).uuid)
            if not self.uuid.startswith("GPU-"):
                self.uuid = "GPU-" + self.uuid
        except Exception:
            self.uuid = None

    def start(self):
        cmd = ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits", "-lms", "200"]
        if self.uuid:
            cmd[1:1] = ["-i", self.uuid]
        try:
            self.proc = subprocess.Popen(cmd, stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
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
        sm, mx, power, reasons = [], [], [], set()
        names = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")
        for line in out.splitlines():
            f = [x.strip() for x in line.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                mx.append(float(f[2]))
                power.append(float(f[3]))
            except ValueError:
                continue
            for name, val in zip(names, f[5:9]):
                if val.lower() == "active":
                    reasons.add(name)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "reasons": sorted(reasons),
                "power_w_max": max(power) if power else None, "samples": len(sm)}


# ----------------------------------------------------------------------------- algorithmic work

def stage_work(w: W.Workload, A: float, n_active: float, fp8: bool = False, gather: bool = False):
    """Algorithmic bytes and FLOPs of each stage for one step (A kept pairs, n_active experts with rows).
    fp8: the dispatched rows and the gate/up weights are one byte per element (plus a float32 scale
    per row)."""
    b = w.elem_bytes
    T, h, E, k, d = w.T, w.h, w.E, w.k, w.d_e
    route_bytes = T * h * b + h * E * b + T * k * 8 + (h * E * b + T * E * 4 if w.noisy else 0)
    route_flops = 2 * T * h * E * (2 if w.noisy else 1)
    xb, wb = (1, 1) if fp8 else (b, b)
    dispatch_bytes = T * h * b + A * h * xb + T * k * 12 + (A * 4 if fp8 else 0)
    if gather:  # no row copy: the first GEMM reads the A token rows of U in place of X
        dispatch_bytes = T * k * 12
    ffn_flops = 6 * A * h * d
    ffn_bytes = (2 * wb + b) * h * d * n_active + A * h * xb + A * h * b + 2 * A * d * b
    combine_bytes = A * h * b + 2 * T * h * b + T * k * 8 + w.n_shared * T * h * b
    work = {"route": {"bytes": route_bytes, "flops": route_flops},
            "dispatch": {"bytes": dispatch_bytes, "flops": 0},
            "ffn": {"bytes": ffn_bytes, "flops": ffn_flops},
            "combine": {"bytes": combine_bytes, "flops": 0}}
    if w.n_shared:
        ds = w.d_shared
        work["shared_ffn"] = {"flops": 6 * T * h * ds * w.n_shared,
                              "bytes": w.n_shared * (3 * h * ds * b + T * h * b + 2 * T * ds * b + T * h * b)}
    return work


def launches_per_step(w: W.Workload, gather: bool = False, fp8: bool = False) -> int:
    """Kernels libmoe launches for one moe_layer_forward (moe_layer_forward_fp8) of this workload."""
    if w.T == 0:
        return 2  # dispatch scan + statistics
    fused_router = w.dtype == W.BF16 and (2 * w.E if w.noisy else w.E) <= 256
    route = 1 if fused_router else 2       # the fused router (weights packed beforehand), or logits + selection
    if w.priority == W.PRIORITY_CHOICE_MAJOR:
        # histograms, column scans, then slots + row copy (no copy when gathering); no column scan
        # when the placement blocks add up histograms of at most 8192 counts themselves, and no
        # histograms either when they count at most 8192 expert ids themselves (token chunks of
        # 8 .. 256 tokens)
        tc = 8
        while tc < 256 and tc * 2 * 148 < w.T:
            tc *= 2
        meta = 1 if w.T * w.k <= 8192 else 2 if -(-w.T // tc) * w.k * w.E <= 8192 else 3
        dispatch = meta
    else:
        meta = 3                           # count, scan, assign
        dispatch = 3 if gather else 4      # (, scatter)
    if fp8:
        dispatch = meta + 1                # the metadata only (no bf16 copy), then the E4M3 row copy
    ffn, combine = 2, 1                    # two GEMMs; rows and statistics
    return route + dispatch + ffn + 2 * w.n_shared + combine


def kernel_source_sha(files) -> str:
    h = hashlib.sha256()
    for f in files:
        with open(os.path.join(ROOT, f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()


def profile_traffic(workload_name):
    """DRAM bytes per step of the grouped GEMM (both launches) from the committed ncu summary,
    if the kernel source it was taken on is the current one (else None)."""
    path = os.path.join(ROOT, "profiles", f"grouped_gemm_{workload_name}.md")
    if not os.path.exists(path):
        return None
    txt = open(path).read()
    m_sha = re.search(r"source_sha256:\s*([0-9a-f]{64})", txt)
    m_tr = re.search(r"traffic_bytes_per_step:\s*([0-9.eE+]+)", txt)
    if not (m_sha and m_tr) or m_sha.group(1) != kernel_source_sha(GEMM_SOURCES):
        return None
    return float(m_tr.group(1))


# ----------------------------------------------------------------------------- CPU oracle timing

class _Inp:
    def __init__(self, **kw):
        self.__dict__.update(kw)


def oracle_inputs_host(inp: "synth.LayerInputs"):
    """Host copies of the layer's inputs in their own precision (the oracle widens them to double as
    it reads them).  Made once, outside every timed region."""
    def host(x):
        return None if x is None else x.detach().to("cpu").contiguous()
    return _Inp(U=host(inp.U), W_r=host(inp.W_r), b_r=host(inp.b_r), W_noise=host(inp.W_noise), eps=host(inp.eps),
                W_gate=host(inp.W_gate), W_up=host(inp.W_up), W_down=host(inp.W_down), sel_bias=host(inp.sel_bias),
                shared=None if inp.shared is None else tuple(host(x) for x in inp.shared))


def oracle_step(w: W.Workload, host, tokens):
    """The oracle's whole layer forward on a sample of the batch's tokens (its capacity from the
    sample's own size); returns its per-stage seconds."""
    import oracle
    t = torch.as_tensor(tokens, dtype=torch.int64)
    sub = _Inp(U=host.U[t], W_r=host.W_r, b_r=host.b_r, W_noise=host.W_noise,
               eps=None if host.eps is None else host.eps[t], W_gate=host.W_gate, W_up=host.W_up,
               W_down=host.W_down)
    r = oracle.layer_forward(sub, T=len(tokens), h=w.h, E=w.E, k=w.k, d_e=w.d_e, score_fn=w.score_fn,
                             renorm=w.renorm, capacity_factor=w.capacity_factor, capacity_override=w.capacity,
                             priority=w.priority, sel_bias=host.sel_bias, shared=host.shared, n_group=w.n_group,
                             topk_group=w.topk_group)
    return r["seconds"]


def stage_seconds_report(totals: dict, n_tokens_total: int):
    whole = sum(totals.values())
    return {name: {"s": round(s, 4), "share": round(s / whole, 4) if whole > 0 else 0.0,
                   "us_per_token": round(s / max(1, n_tokens_total) * 1e6, 2)}
            for name, s in totals.items()}


def oracle_cpu_info():
    import oracle
    return {"cores": os.cpu_count() or 1, "threads": oracle.threads()}


def cpu_baseline(w: W.Workload, inp, n_tokens: int = 0, target_s: float = 12.0):
    """The oracle as it stands on the host cores, on a bounded sample of the batch: a probe on a few
    tokens sets the sample size for about `target_s` seconds of CPU work (all T tokens, run again
    until that time is reached, when the whole batch is faster)."""
    import numpy as np
    host = oracle_inputs_host(inp)
    oracle_step(w, host, np.arange(min(w.T, 8)))  # untimed: first-call costs (threads, page faults)
    n = min(w.T, 64)
    while True:
        t0 = time.perf_counter()
        oracle_step(w, host, np.arange(n))
        one = time.perf_counter() - t0
        if n >= w.T or one >= target_s / 4 or (n_tokens and n >= n_tokens):
            break
        n = min(w.T, n * 4)
    toks = np.arange(n)
    reps, totals, t0 = 0, {}, time.perf_counter()
    while True:
        sec = oracle_step(w, host, toks)
        for name, s in sec.items():
            totals[name] = totals.get(name, 0.0) + s
        reps += 1
        dt = time.perf_counter() - t0
        if dt >= target_s or dt + dt / reps > 30.0:
            break
    info = oracle_cpu_info()
    return {"value": n * reps / dt, "unit": "tokens/s", "cores": info["threads"], "host_cores": info["cores"],
            "kind": "oracle",
            "sample": f"C++ oracle layer forward (plain loops, double accumulation, OpenMP over rows, "
                      f"{info['threads']} threads) on the first {n} of the batch's {w.T} tokens, {reps} call(s) in "
                      f"{dt:.1f} s; capacity from those {n} tokens",
            "stages": stage_seconds_report(totals, n * reps)}


def run_reference(args, w: W.Workload):
    import numpy as np
    ws, rank, _ = dist_env()
    if rank != 0:
        return 0
    host = oracle_inputs_host(synth.generate(w, seed=0, device="cpu"))
    budget = float(args.reference_budget_s)
    rng = np.random.default_rng(0)
    probe = np.sort(rng.choice(w.T, size=min(8, w.T), replace=False))
    oracle_step(w, host, probe)  # untimed: first-call costs
    t0 = time.perf_counter()
    oracle_step(w, host, probe)
    per_call = time.perf_counter() - t0
    # a call costs a fixed part (each weight row is read once) plus a part per token: size the sample
    # from two probes so that warm-up + steps fit the budget
    probe2 = np.sort(rng.choice(w.T, size=min(64, w.T), replace=False))
    t0 = time.perf_counter()
    oracle_step(w, host, probe2)
    per_call2 = time.perf_counter() - t0
    per_tok = max((per_call2 - per_call) / max(1, len(probe2) - len(probe)), 1e-6)
    fixed = max(per_call - per_tok * len(probe), 0.0)
    per_step = budget / max(1, args.steps + args.warmup)
    n = int(max(1, min(w.T, (per_step - fixed) / per_tok)))
    for _ in range(args.warmup):
        oracle_step(w, host, np.sort(rng.choice(w.T, size=n, replace=False)))
    totals = {}
    t0 = time.perf_counter()
    for _ in range(args.steps):
        for name, s in oracle_step(w, host, np.sort(rng.choice(w.T, size=n, replace=False))).items():
            totals[name] = totals.get(name, 0.0) + s
    dt = time.perf_counter() - t0
    value = n * args.steps / dt
    info = oracle_cpu_info()
    sample = (f"each step: the C++ oracle layer forward (plain loops, double accumulation, OpenMP over rows, "
              f"{info['threads']} threads) on {n} tokens drawn from the {w.T}-token batch")
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": ws,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": dt / args.steps * 1e3,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic", "config": workload_config(w),
            "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": info["threads"], "host_cores": info["cores"],
                             "kind": "oracle", "sample": sample, "stages": stage_seconds_report(totals, n * args.steps)},
            "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)
    return 0


# ----------------------------------------------------------------------------- reference arm

def ffn_tiles(w: W.Workload) -> str:
    """The grouped-GEMM kernel libmoe picks: 256-row CTA-pair tiles when the mean expert segment is
    at least 1024 rows, else the weights-as-M pair kernel "swab" (MOE_FFN_TILES overrides)."""
    env = os.environ.get("MOE_FFN_TILES", "")
    if env in ("single", "pair", "swab"):
        return env + " (MOE_FFN_TILES)"
    if w.dtype == W.F32:
        return "cuda-core float32"
    return "pair" if w.T * w.k >= 1024 * w.E else "swab"


def workload_config(w: W.Workload, n_rot: int = 0):
    c = {"workload": w.name, "T": w.T, "h": w.h, "E": w.E, "k": w.k, "d_e": w.d_e,
         "score": "softmax" if w.score_fn == W.SOFTMAX else "sigmoid", "renorm": w.renorm, "noisy": w.noisy,
         "capacity_factor": w.capacity_factor, "logit_bias": w.bias, "parallelism": "replicas",
         "ffn_tiles": ffn_tiles(w)}
    if w.n_shared:
        c.update(n_shared=w.n_shared, d_shared=w.d_shared)
    if w.sel_bias != "none":
        c["selection_bias"] = "loss-free balancing bias ~ N(0, 0.05) on the scores"
    if w.n_group > 1:
        c.update(n_group=w.n_group, topk_group=w.topk_group)
    if n_rot:
        c["l2"] = (f"inputs larger than L2: {n_rot} rotating token batches plus "
                   f"{3 * w.E * w.h * w.d_e * w.elem_bytes / 1e9:.2f} GB of expert weights per step")
    return c


# ----------------------------------------------------------------------------- B300 arm

STAGES = ("route", "dispatch", "ffn", "shared_ffn", "combine")


class _GraphEvents:
    """CUDA events recorded as nodes of a captured graph (cudaEventRecordExternal), so that the
    device time between two stages of one graph replay can be read without launch gaps."""

    EXTERNAL = 0x01  # cudaEventRecordExternal

    def __init__(self):
        import ctypes
        self.ct = ctypes
        self.rt = ctypes.CDLL("libcudart.so.13")
        self.rt.cudaEventCreate.argtypes = [ctypes.POINTER(ctypes.c_void_p)]
        self.rt.cudaEventRecordWithFlags.argtypes = [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_uint]
        self.rt.cudaEventElapsedTime.argtypes = [ctypes.POINTER(ctypes.c_float), ctypes.c_void_p, ctypes.c_void_p]
        self.rt.cudaEventDestroy.argtypes = [ctypes.c_void_p]

    def new(self):
        ev = self.ct.c_void_p()
        if self.rt.cudaEventCreate(self.ct.byref(ev)) != 0:
            raise RuntimeError("cudaEventCreate failed")
        return ev

    def record(self, ev, stream):
        if self.rt.cudaEventRecordWithFlags(ev, self.ct.c_void_p(stream.cuda_stream), self.EXTERNAL) != 0:
            raise RuntimeError("cudaEventRecordWithFlags failed")

    def elapsed(self, a, b) -> float:
        ms = self.ct.c_float()
        if self.rt.cudaEventElapsedTime(self.ct.byref(ms), a, b) != 0:
            raise RuntimeError("cudaEventElapsedTime failed")
        return ms.value


class LayerRun:
    """One workload on the device: inputs, rotating token batches, buffers, and CUDA graphs of the
    whole layer and of each stage (one of each per batch)."""

    def __init__(self, w: W.Workload, device, fp8: bool = False, gather: bool = False):
        from mixture_experts_layer_84_b300 import _lib as L
        self.L, self.w, self.device = L, w, device
        self.inp = inp = synth.generate(w, seed=0, device=device)
        ubytes = w.T * w.h * w.elem_bytes
        self.n_rot = max(2, min(64, math.ceil(2 * L2_BYTES / max(ubytes, 1))))
        self.pool = [inp.U] + [synth.normal((w.T, w.h), 1.0, 100 + r, "U", device, w.torch_dtype)
                               for r in range(self.n_rot - 1)]
        self.cfg = L.config_of(w)
        if fp8 and (w.dtype != W.BF16 or w.h % 16):
            raise SystemExit("bench.py --fp8: needs a bf16 workload with h % 16 == 0")
        self.fp8 = fp8
        self.gather = gather and not fp8 and w.dtype == W.BF16
        self.bufs = L.LayerBuffers.allocate(self.cfg, device=device, with_X=not (fp8 or self.gather))
        self.w8 = L.FP8Weights.quantize(inp.W_gate, inp.W_up) if fp8 else None  # once, outside every timed region
        self.rows8 = L.FP8Rows.allocate(self.cfg, device=device) if fp8 else None
        self.stages = [s for s in STAGES if s != "shared_ffn" or w.n_shared]
        self.graphs, self.stage_graphs, self.graph_error = [], [], None
        self.timed_graphs, self.graph_events, self.stage_timing_note = [], None, None
        # the router weights packed once for the tensor-core router (None where it reads W_r as is);
        # timed on its own, outside every timed region
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        L.moe_pack_router(self.cfg, inp.W_r, inp.W_noise)  # first call: module loading, attributes
        e0.record()
        self.W_r_packed = L.moe_pack_router(self.cfg, inp.W_r, inp.W_noise)
        e1.record()
        torch.cuda.synchronize(device)
        self.pack_ms = e0.elapsed_time(e1) if self.W_r_packed is not None else None

    # the stage calls of moe_layer_forward (or moe_layer_forward_fp8), one function per stage
    def run_stage(self, name, U):
        L, w, inp, b, cfg = self.L, self.w, self.inp, self.bufs, self.cfg
        if name == "route":
            if self.W_r_packed is not None:
                L.moe_route_packed(cfg, U, self.W_r_packed, inp.b_r, inp.eps, None, b.idx, b.gate, b.ws,
                                   sel_bias=inp.sel_bias)
            else:
                L.moe_route(cfg, U, inp.W_r, inp.b_r, inp.W_noise, inp.eps, None, None, b.idx, b.gate, b.ws,
                            sel_bias=inp.sel_bias)
        elif name == "dispatch":
            if self.fp8:
                L.moe_dispatch_fp8(cfg, U, b.idx, b.counts_routed, b.counts_kept, b.offsets, b.slot_row, b.row_token,
                                   self.rows8.X8, self.rows8.x_scale, b.n_dropped, b.ws)
            else:  # gather: routing metadata only, the first GEMM reads the token rows itself
                L.moe_dispatch(cfg, U, b.idx, b.counts_routed, b.counts_kept, b.offsets, b.slot_row, b.row_token,
                               None if self.gather else b.X, b.n_dropped, b.ws)
        elif name == "ffn":
            if self.fp8:
                L.moe_expert_ffn_fp8(cfg, self.rows8.X8, self.rows8.x_scale, b.offsets, self.w8, inp.W_down, b.act,
                                     b.Y, b.ws)
            elif self.gather:
                L.moe_expert_ffn_gather(cfg, U, b.row_token, b.offsets, inp.W_gate, inp.W_up, inp.W_down, b.act, b.Y,
                                        b.ws)
            else:
                L.moe_expert_ffn(cfg, b.X, b.offsets, inp.W_gate, inp.W_up, inp.W_down, b.act, b.Y, b.ws)
        elif name == "shared_ffn":
            L.moe_shared_ffn(cfg, U, inp.W_gate_sh, inp.W_up_sh, inp.W_down_sh, b.act_shared, b.Y_shared, b.ws)
        elif name == "combine":
            L.moe_combine(cfg, U, b.Y, b.slot_row, b.gate, b.counts_routed, b.out, b.f, b.P, b.aux, b.ws,
                          z_loss=b.z_loss, Y_shared=b.Y_shared)
        else:
            raise ValueError(name)

    def layer(self, U):
        for s in self.stages:
            self.run_stage(s, U)

    def batch_stats(self):
        """Kept pairs and active experts of each batch (outside any timed region)."""
        self.A_of, self.act_of = [], []
        for U in self.pool:
            self.layer(U)
            off = self.bufs.offsets.cpu()
            self.A_of.append(int(off[-1]))
            self.act_of.append(int(((off[1:] - off[:-1]) > 0).sum()))
        code = self.L.moe_get_device_status(self.bufs.ws)
        if code != 0:
            raise SystemExit(f"bench.py: device status {code} on {self.w.name}")

    def capture(self, enabled: bool = True):
        """One graph of the whole layer per batch, and one graph per stage per batch."""
        if not enabled:
            return
        dev = self.device
        cap = torch.cuda.Stream(dev)
        cap.wait_stream(torch.cuda.current_stream(dev))
        with torch.cuda.stream(cap):
            self.layer(self.pool[0])  # first calls on this stream outside the capture
        torch.cuda.current_stream(dev).wait_stream(cap)
        torch.cuda.synchronize(dev)
        try:
            for U in self.pool:
                g = torch.cuda.CUDAGraph()
                # relaxed: the library's host-side set-up calls (kernel attributes) are not stream work
                with torch.cuda.graph(g, stream=cap, capture_error_mode="relaxed"):
                    self.layer(U)
                self.graphs.append(g)
                per = {}
                for s in self.stages:
                    gs = torch.cuda.CUDAGraph()
                    with torch.cuda.graph(gs, stream=cap, capture_error_mode="relaxed"):
                        self.run_stage(s, U)
                    per[s] = gs
                self.stage_graphs.append(per)
        except RuntimeError as exc:  # time eager launches instead, and say so
            self.graphs, self.stage_graphs = [], []
            self.graph_error = str(exc).splitlines()[0][:200]
            torch.cuda.synchronize(dev)
            return
        # the whole layer once more per batch, with an event node before each stage and after the last
        try:
            ge = _GraphEvents()
            for U in self.pool:
                evs = [ge.new() for _ in range(len(self.stages) + 1)]
                g = torch.cuda.CUDAGraph()
                with torch.cuda.graph(g, stream=cap, capture_error_mode="relaxed"):
                    for j, s in enumerate(self.stages):
                        ge.record(evs[j], cap)
                        self.run_stage(s, U)
                    ge.record(evs[-1], cap)
                self.timed_graphs.append((g, evs))
            self.graph_events = ge
        except (RuntimeError, OSError, AttributeError) as exc:
            self.timed_graphs, self.graph_events = [], None
            self.stage_timing_note = "event nodes unavailable (" + str(exc).splitlines()[0][:120] + ")"
            torch.cuda.synchronize(dev)

    def step(self, i):
        if self.graphs:
            self.graphs[i % self.n_rot].replay()
        else:
            self.layer(self.pool[i % self.n_rot])

    def stage_step(self, i, ev):
        """Step i with an event before each stage and after the last (device time of each stage)."""
        b = i % self.n_rot
        for j, s in enumerate(self.stages):
            ev[j].record()
            if self.stage_graphs:
                self.stage_graphs[b][s].replay()
            else:
                self.run_stage(s, self.pool[b])
        ev[len(self.stages)].record()

    def time_steps(self, K, warmup):
        """Milliseconds of exactly K steps (after `warmup` untimed ones), barriers on both sides."""
        for i in range(warmup):
            self.step(i)
        barrier(self.device)
        t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        t0.record()
        for i in range(K):
            self.step(i)
        t1.record()
        barrier(self.device)
        return t0.elapsed_time(t1)

    def time_stages(self, K):
        """Per stage, the median device time over K steps: between the event nodes of one whole-layer
        graph replay where those exist, else between the replays of each stage's own graph."""
        n = len(self.stages)
        if self.timed_graphs:
            ge = self.graph_events
            try:
                for i in range(min(K, 3)):
                    self.timed_graphs[i % self.n_rot][0].replay()
                torch.cuda.synchronize(self.device)
                per = [[] for _ in range(n)]
                for i in range(K):
                    g, evs = self.timed_graphs[i % self.n_rot]
                    g.replay()
                    torch.cuda.synchronize(self.device)  # the next replay of this graph re-records its events
                    for j in range(n):
                        per[j].append(ge.elapsed(evs[j], evs[j + 1]))
                return {s: statistics.median(per[j]) for j, s in enumerate(self.stages)}
            except RuntimeError as exc:
                self.timed_graphs = []
                self.stage_timing_note = "event nodes unreadable (" + str(exc).splitlines()[0][:120] + ")"
        evs = [[torch.cuda.Event(enable_timing=True) for _ in range(n + 1)] for _ in range(K)]
        for i in range(min(K, 3)):
            self.stage_step(i, evs[i])  # warm-up of the stage graphs
        torch.cuda.synchronize(self.device)
        for i in range(K):
            self.stage_step(i, evs[i])
        torch.cuda.synchronize(self.device)
        return {s: statistics.median(evs[i][j].elapsed_time(evs[i][j + 1]) for i in range(K))
                for j, s in enumerate(self.stages)}

    def stage_timing_desc(self) -> str:
        if self.timed_graphs:
            return ("device time between event nodes before each stage of one whole-layer graph replay, median "
                    "over the K steps (a stage carries the write-back of the dirty L2 lines left by the one before)")
        what = ("device time of each stage's own CUDA graph, replayed in layer order with events between them, "
                "median over the K steps")
        return what + ("; " + self.stage_timing_note if self.stage_timing_note else "")

    def work(self, K):
        A_mean = sum(self.A_of[i % self.n_rot] for i in range(K)) / K
        act_mean = sum(self.act_of[i % self.n_rot] for i in range(K)) / K
        return A_mean, act_mean, stage_work(self.w, A_mean, act_mean, self.fp8, self.gather)


def stage_report(stage_ms, work, peaks):
    stages = {}
    for name, m in stage_ms.items():
        wk = work[name]
        gbs = wk["bytes"] / (m * 1e-3) / 1e9
        d = {"ms": round(m, 5), "GB/s": round(gbs, 1), "frac_hbm": round(gbs / peaks["hbm_gbs"], 4)}
        if wk["flops"]:
            tf = wk["flops"] / (m * 1e-3) / 1e12
            d["TFLOP/s"] = round(tf, 2)
            d["frac_tensor"] = round(tf / peaks["bf16_tflops"], 4)
        stages[name] = d
    return stages


def roofline(w: W.Workload, work, ffn_ms, A_mean, peaks, peak_src, fp8=False):
    """The dominant kernel's roofline: the grouped expert GEMM (both launches of one step)."""
    ffn = work["ffn"]
    intensity = ffn["flops"] / max(ffn["bytes"], 1)
    ridge = peaks["bf16_tflops"] * 1e12 / (peaks["hbm_gbs"] * 1e9)
    if w.dtype == W.F32:
        # float32 CUDA-core FMA peak: 148 SMs x 128 lanes x 2 FLOP x 2.032 GHz
        roof = {"bound": "alu", "achieved": ffn["flops"] / (ffn_ms * 1e-3) / 1e12,
                "peak": 148 * 128 * 2 * 2.032e9 / 1e12, "unit": "TFLOP/s"}
    elif fp8 and intensity >= ridge * 1.5:
        # gate|up (4 A h d FLOPs) at twice the bf16 rate (the recipe's nominal fp8 : bf16 ratio) and
        # down (2 A h d) at the bf16 rate: the peak is the FLOPs over the time both take at peak,
        # 1.5x the bf16 rate, and so is the ridge
        f1, f2 = 4 * A_mean * w.h * w.d_e, 2 * A_mean * w.h * w.d_e
        mixed = (f1 + f2) / (f1 / (2 * peaks["bf16_tflops"]) + f2 / peaks["bf16_tflops"]) if f1 + f2 else 1.0
        roof = {"bound": "tensor", "achieved": ffn["flops"] / (ffn_ms * 1e-3) / 1e12, "peak": round(mixed, 1),
                "unit": "TFLOP/s"}
    elif intensity >= ridge:
        roof = {"bound": "tensor", "achieved": ffn["flops"] / (ffn_ms * 1e-3) / 1e12, "peak": peaks["bf16_tflops"],
                "unit": "TFLOP/s"}
    else:
        roof = {"bound": "hbm", "achieved": ffn["bytes"] / (ffn_ms * 1e-3) / 1e9, "peak": peaks["hbm_gbs"],
                "unit": "GB/s"}
    roof["frac"] = round(roof["achieved"] / roof["peak"], 4)
    if roof["bound"] == "tensor" and not fp8:
        # the same against the bf16 rate measured under the power cap in a seconds-long loop
        roof["peak_sustained"] = peaks["bf16_tflops_sustained"]
        roof["frac_sustained"] = round(roof["achieved"] / peaks["bf16_tflops_sustained"], 4)
    roof["achieved"] = round(roof["achieved"], 2)
    roof["traffic"] = None if fp8 else profile_traffic(w.name)
    tiles = ffn_tiles(w)
    kname = ("ffn_simt_f32" if w.dtype == W.F32 else "grouped_gemm_swab" if tiles.startswith("swab")
             else "grouped_gemm_tc_pair" if tiles.startswith("pair") else "grouped_gemm_tc")
    roof["kernel"] = f"grouped SwiGLU expert GEMM ({tiles} tiles: {kname}) gate|up + down, both launches of one step"
    roof["peak_source"] = f"{peak_src}, {'bf16 burst' if roof['bound'] == 'tensor' else roof['bound']}"
    roof["timing"] = "median CUDA-event time of the ffn stage graph over the timed steps"
    if fp8:
        roof["kernel"] = ("grouped SwiGLU expert GEMM: E4M3 gate|up (kind::f8f6f4) + bf16 down, both launches of "
                          "one step")
        if roof["bound"] == "tensor":
            roof["peak_source"] += ("; E4M3 gate|up at 2x the measured bf16 burst (nominal ratio), combined with "
                                    "bf16 down by their FLOPs")
    return roof


def measure(run: LayerRun, K: int, warmup: int, repeats: int):
    """value (median over `repeats` regions of exactly K steps), stage device times, roofline."""
    run.batch_stats()
    run.capture()
    regions = [run.time_steps(K, warmup if r == 0 else 1) for r in range(repeats)]
    stage_ms = run.time_stages(K)
    return regions, stage_ms


def per_config_entry(w: W.Workload, device, K: int, warmup: int, repeats: int, peaks, peak_src):
    run = LayerRun(w, device)
    regions, stage_ms = measure(run, K, warmup, repeats)
    ms = statistics.median(regions)
    A_mean, act_mean, work = run.work(K)
    d = {"workload": w.name, "value": round(w.T * K / (ms * 1e-3), 1), "unit": "tokens/s",
         "ms_per_step": round(ms / K, 5), "steps": K, "repeats": repeats,
         "value_range": [round(w.T * K / (max(regions) * 1e-3), 1), round(w.T * K / (min(regions) * 1e-3), 1)],
         "roofline": roofline(w, work, stage_ms["ffn"], A_mean, peaks, peak_src),
         "stages": stage_report(stage_ms, work, peaks),
         "stage_sum_ms": round(sum(stage_ms.values()), 5),
         "kept_pairs_A": A_mean, "active_experts": act_mean,
         "launch": "one CUDA graph replay per step" if run.graphs else "eager stage calls",
         "config": workload_config(w, run.n_rot)}
    del run
    torch.cuda.empty_cache()
    return d


def run_b300(args, w: W.Workload):
    ws_n, rank, local = init_dist("nccl")
    if not torch.cuda.is_available():
        raise SystemExit("bench.py: no CUDA device")
    device = torch.device("cuda", local)
    torch.cuda.set_device(device)
    L = None
    from mixture_experts_layer_84_b300 import _lib as L  # noqa: F811

    run = LayerRun(w, device, fp8=args.fp8, gather=args.gather)
    fp8, inp, cfg, bufs, pool, n_rot = run.fp8, run.inp, run.cfg, run.bufs, run.pool, run.n_rot
    K = args.steps
    peaks, peak_src = measured_peaks()

    run.batch_stats()
    clocks = ClockSampler(device) if rank == 0 else None
    barrier(device)
    if clocks:
        clocks.start()
        time.sleep(0.3)
    run.capture(not args.no_graph)
    # R regions of exactly K steps each (the first after the warm-up); `value` is the median region
    regions = [run.time_steps(K, args.warmup if r == 0 else 1) for r in range(args.repeats)]
    stage_ms = run.time_stages(K)

    # end to end through the public call: every step copies its tokens in from pinned host memory,
    # runs moe_layer_forward and reads out (and aux) back.  Three streams pipeline the steps: the
    # copy-in of step j+1 and the copy-out of step j-1 overlap the layer of step j.
    import dataclasses
    U_host = [torch.empty((w.T, w.h), dtype=w.torch_dtype, pin_memory=True) for _ in range(2)]
    for j in range(2):
        U_host[j].copy_(pool[j])
    out_host = [torch.empty((w.T, w.h), dtype=w.torch_dtype, pin_memory=True) for _ in range(2)]
    aux_host = [torch.empty(1, dtype=torch.float32, pin_memory=True) for _ in range(2)]
    U_dev = [torch.empty_like(inp.U) for _ in range(2)]
    bset = [bufs, dataclasses.replace(bufs, out=torch.empty_like(bufs.out), aux=torch.empty_like(bufs.aux))]
    s_in, s_comp, s_out = (torch.cuda.Stream(device) for _ in range(3))
    ev_in = [torch.cuda.Event() for _ in range(2)]
    ev_comp = [torch.cuda.Event() for _ in range(2)]
    ev_out = [torch.cuda.Event() for _ in range(2)]
    for e in ev_comp + ev_out:
        e.record(torch.cuda.current_stream(device))

    def e2e_step(j):
        b = j % 2
        with torch.cuda.stream(s_in):
            s_in.wait_event(ev_comp[b])            # the layer two steps back has read U_dev[b]
            U_dev[b].copy_(U_host[b], non_blocking=True)
            ev_in[b].record(s_in)
        with torch.cuda.stream(s_comp):
            s_comp.wait_event(ev_in[b])
            s_comp.wait_event(ev_out[b])           # out[b] of two steps back has been read
            if fp8:
                L.moe_layer_forward_fp8(cfg, U_dev[b], inp.W_r, inp.b_r, inp.W_noise, inp.eps, run.w8, inp.W_down,
                                        bset[b], run.rows8, stream=s_comp, sel_bias=inp.sel_bias, shared=inp.shared,
                                        W_r_packed=run.W_r_packed)
            else:
                L.moe_layer_forward(cfg, U_dev[b], inp.W_r, inp.b_r, inp.W_noise, inp.eps, inp.W_gate, inp.W_up,
                                    inp.W_down, bset[b], stream=s_comp, sel_bias=inp.sel_bias, shared=inp.shared,
                                    W_r_packed=run.W_r_packed)
            ev_comp[b].record(s_comp)
        with torch.cuda.stream(s_out):
            s_out.wait_event(ev_comp[b])
            out_host[b].copy_(bset[b].out, non_blocking=True)
            aux_host[b].copy_(bset[b].aux, non_blocking=True)
            ev_out[b].record(s_out)

    for j in range(3):
        e2e_step(j)
    torch.cuda.synchronize(device)
    barrier(device)
    t0 = time.perf_counter()
    for j in range(K):
        e2e_step(j)
    torch.cuda.synchronize(device)
    e2e_s = time.perf_counter() - t0
    barrier(device)
    clk = clocks.stop() if clocks else None
    code = L.moe_get_device_status(bufs.ws)
    if code != 0:
        raise SystemExit(f"bench.py: device status {code} after the timed region")

    # the layer backward (bf16): L = <dO, out> + 0.01 E sum f P + 0.001 L_z, on the forward of
    # the first batch; timed over min(K, 50) steps after 3 warm-up steps (not part of `value`)
    train = None
    if w.dtype == W.BF16 and not args.no_backward and not fp8:
        fb = L.LayerBuffers.allocate(cfg, device=device, with_logits=True)
        fwd_args = (cfg, pool[0], inp.W_r, inp.b_r, inp.W_noise, inp.eps, inp.W_gate, inp.W_up, inp.W_down, fb)
        L.moe_layer_forward(*fwd_args, sel_bias=inp.sel_bias, shared=inp.shared)
        grads = L.GradBuffers.allocate(cfg, device=device)
        dO = synth.normal((w.T, w.h), 1.0, 7, "Y", device, w.torch_dtype)

        def bwd():
            L.moe_layer_backward(*fwd_args, dO, grads, w_aux=0.01, w_z=0.001, sel_bias=inp.sel_bias,
                                 shared=inp.shared)

        for _ in range(3):
            bwd()
        KB = min(K, 50)
        b0, b1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        b0.record()
        for _ in range(KB):
            bwd()
        b1.record()
        torch.cuda.synchronize(device)
        bwd_ms = b0.elapsed_time(b1) / KB
        code = L.moe_get_device_status(fb.ws)
        if code != 0:
            raise SystemExit(f"bench.py: device status {code} after the backward")
        A0 = run.A_of[0]
        bwd_flops = 12 * A0 * w.h * w.d_e + 2 * 6 * w.T * w.h * w.E  # experts (2x the forward) + router
        if w.n_shared:
            bwd_flops += 12 * w.T * w.h * w.d_shared * w.n_shared
        step_ms = statistics.median(regions) / K
        train = {"backward_ms": round(bwd_ms, 4), "steps": KB,
                 "forward_plus_backward_tokens_per_s": round(w.T / ((step_ms + bwd_ms) * 1e-3), 1),
                 "backward_TFLOP/s": round(bwd_flops / (bwd_ms * 1e-3) / 1e12, 2),
                 "what": "moe_layer_backward: combine, gate/aux/z, grouped expert backward (recomputed gate|up), "
                         "router linear, permute; float32 weight gradients"}
        del fb, grads

    total_ms = statistics.median(regions)
    max_ms = max_over_ranks(total_ms, device)
    max_e2e = max_over_ranks(e2e_s, device)
    if rank != 0:
        return 0

    A_mean, act_mean, work = run.work(K)
    stages = stage_report(stage_ms, work, peaks)
    roof = roofline(w, work, stage_ms["ffn"], A_mean, peaks, peak_src, fp8)
    value = weak_scaling_value(w.T, K, ws_n, max_ms * 1e-3)
    e2e_value = weak_scaling_value(w.T, K, ws_n, max_e2e)
    line = {"metric": METRIC, "value": round(value, 1), "unit": "tokens/s", "n_gpus": ws_n, "steps": K,
            "warmup": args.warmup, "ms_per_step": round(max_ms / K, 5), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None,
            "dtype": ("e4m3 dispatch and gate|up, bf16 elsewhere" if fp8 else "bf16") if w.dtype == W.BF16 else "f32",
            "data": "synthetic (seeded N(0,1) tokens, N(0,0.02) weights, device-resident)",
            "config": dict(workload_config(w, n_rot), **({"fp8": "E4M3 token rows and gate/up weight rows, "
                                                                  "one power-of-two scale per row"} if fp8 else {}),
                           **({"x": "not materialised: the first GEMM gathers U rows"} if run.gather else {})),
            "repeats": args.repeats,
            "value_range": [round(weak_scaling_value(w.T, K, ws_n, max(regions) * 1e-3), 1),
                            round(weak_scaling_value(w.T, K, ws_n, min(regions) * 1e-3), 1)],
            "roofline": roof, "stages": stages,
            "stage_timing": run.stage_timing_desc(),
            "stage_sum_ms": round(sum(stage_ms.values()), 5),
            "kept_pairs_A": A_mean, "active_experts": act_mean,
            "router_pack_ms": None if run.pack_ms is None else round(run.pack_ms, 5),
            "e2e": {"value": round(e2e_value, 1), "unit": "tokens/s",
                    "h2d_bytes_per_step": w.T * w.h * w.elem_bytes,
                    "d2h_bytes_per_step": w.T * w.h * w.elem_bytes + 4,
                    "how": f"moe_layer_forward{'_fp8' if fp8 else ''} per step with its U copied in from pinned host memory and out + aux "
                           "copied back; copy-in, layer and copy-out of consecutive steps overlap on three streams"},
            "gpu_launches": launches_per_step(w, run.gather, run.fp8) * K,
            "launch": "one CUDA graph replay per step (the whole layer)" if run.graphs else
                      ("eager stage calls" + (f" (graph capture failed: {run.graph_error})" if run.graph_error else "")),
            "clocks": clk}
    if train:
        line["train_step"] = train
    del run, bset, U_dev
    torch.cuda.empty_cache()
    if ws_n == 1 and not args.no_per_config and not fp8 and not args.gather:
        line["per_config"] = [per_config_entry(x, device, K, args.warmup, args.repeats, peaks, peak_src)
                              for x in W.FULL if x.name != w.name]
    if ws_n == 1 and not args.no_cpu_baseline and not fp8:
        line["cpu_baseline"] = cpu_baseline(w, inp, args.cpu_sample_tokens)
    print(json.dumps(line), flush=True)
    return 0


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--repeats", type=int, default=5, help="timed regions of exactly --steps steps; value = median")
    ap.add_argument("--workload", default=W.STRESS.name, choices=sorted(W.BY_NAME))
    ap.add_argument("--impl", default="b300", choices=["b300", "reference"])
    ap.add_argument("--cpu-sample-tokens", type=int, default=0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-per-config", action="store_true", help="time the named workload only")
    ap.add_argument("--no-graph", action="store_true", help="time eager launches instead of CUDA-graph replays")
    ap.add_argument("--no-backward", action="store_true", help="skip timing the layer backward")
    ap.add_argument("--gather", action="store_true",
                    help="bf16: no X; the first expert GEMM gathers the token rows (moe_layer_forward with X = NULL)")
    ap.add_argument("--fp8", action="store_true",
                    help="time moe_layer_forward_fp8 (E4M3 dispatch and gate|up GEMM) instead of the bf16 layer")
    ap.add_argument("--reference-budget-s", type=float, default=120.0)
    args = ap.parse_args(argv)
    if args.warmup < 3:
        raise SystemExit("bench.py: --warmup must be >= 3")
    if args.repeats < 1:
        raise SystemExit("bench.py: --repeats must be >= 1")
    w = W.BY_NAME[args.workload]
    if args.impl == "reference":
        return run_reference(args, w)
    return run_b300(args, w)


if __name__ == "__main__":
    sys.exit(main())
