#!/usr/bin/env python3
"""Benchmark of the GB300 W8A16 block-scaled GEMM.

One JSON line on stdout (rank 0). A step is one full W8A16 GEMM call on the
workload (default: decode GEMV M=1, N=K=4096, the configuration the headline
metric is quoted on), through w8a16_gemm_ws with a workspace: up to 16 tokens
that is one launch of the kernel that splits its own activation tiles; above,
the split pre-pass and the FP8 x FP8 kernel.

Timing. Steps rotate over B distinct input/output buffer sets totalling at least
3x the L2 size, so every step streams its weights from HBM. The steps are
replayed from CUDA graphs; every graph is replayed once, and then W warm-up
steps are run, before anything is timed. A timed region is exactly K steps
between two CUDA events on the launching stream, preceded by a short spin kernel
so that the host has queued the whole region before the GPU reaches its first
event (no host gap inside a region). Regions are repeated (at least 5 times, and
until the GPU has spent `--min-seconds` in them, so the clock sampler sees the
GPU under load), the whole set bracketed by a barrier and
torch.cuda.synchronize(); ms_per_step is the MEDIAN region / K. The job time
of N ranks is the slowest rank's.

  value    = algorithmic bytes of K steps / median region time (GB/s, whole job)
  configs  = every workload of the metric measured the same way (the headline
             one included), with GB/s, TFLOP/s, % of the HBM roofline, and for
             the multi-tile workload the BF16 tensor bound as well
  roofline = the dominant kernel alone: its own launches replayed back to back
             from a graph and timed with events (for the pre-split path, the
             FP8 x FP8 GEMM without its split pre-pass, which is timed apart)
  e2e      = the same metric through the host-buffer entry point: per step the
             pinned host->device copies of A, W and block_scale, the GEMM, and the
             device->host copy of C
  cpu_baseline = the CPU oracle on the host cores, on a bounded sample

--path w8a8 times the W8A8 variant instead: a step is the per-token 128-group
activation quantiser followed by the FP8 x FP8 block-scaled GEMM (two launches);
`value` still counts the BF16-activation problem's bytes, and the roofline entry
is the GEMM kernel alone (its own algorithmic bytes: FP8 activation codes and
group scales instead of BF16 activations).

--tokens M runs a workload at another token count, e.g. the multi-tile workload at
M=256 (two 128-token tiles: one weight pass from HBM, the second token tile of each
weight tile reading it from L2); the JSON line then names it multitile_m256_...

--impl reference times the CPU oracle (the reference arm: there is no runnable
reference implementation) on the same workload and metric.
"""
from __future__ import annotations

import argparse
import ctypes
import dataclasses
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
from pathlib import Path

ROOT = Path(__file__).resolve().parent
sys.path.insert(0, str(ROOT))

import workloads  # noqa: E402

METRIC = "W8A16 GEMM achieved HBM GB/s and TFLOP/s at M=1..32; % of GB300 HBM roofline"
METRIC_W8A8 = ("W8A8 variant (activation quantiser + FP8xFP8 GEMM) achieved HBM GB/s of the W8A16 "
               "problem; % of GB300 HBM roofline")
DEFAULT_WORKLOAD = "decode_gemv_m1_n4096_k4096"
FALLBACK_HBM_GBS = 6800.0
FALLBACK_BF16_TFLOPS = 1900.0
# GPU cycles of the spin kernel queued before each timed region (~30 us at 2 GHz):
# long enough for the host to queue the region's events and graph replays.
PREROLL_CYCLES = 60000
# Longest timed region of a workload that is not the headline (its K is capped so).
CONFIG_REGION_SECONDS = 0.02

ARITHMETIC = {
    "two_term": "BF16 activations as two E4M3 terms (hi + lo/32 per 128-K block, exact for |a| >= "
                "2^-14 of the block maximum) x E4M3 weights on the tensor cores, FP32 accumulate, "
                "one FP32 block-scale fold per 128-K step, BF16 output",
    "w8a8": "E4M3 activations (per-token 128-K group scales) x E4M3 weights on the tensor cores, "
            "FP32 accumulate, BF16 output",
    "oracle": "FP64 products and plain k-order FP64 sum, one BF16 rounding (the CPU oracle)",
}


def w8a8_gemm_bytes(wl, terms: int = 1) -> int:
    """Algorithmic bytes of one FP8 x FP8 GEMM launch: E4M3 weights, block scales,
    `terms` E4M3 activation codes per value, FP32 factors per token and 128-K
    group, BF16 output, each once."""
    kb = wl.K // 128
    return (wl.N * wl.K + 4 * ((wl.N + 127) // 128) * kb + terms * wl.M * wl.K + 4 * wl.M * kb
            + 2 * wl.M * wl.N)


def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def max_over_ranks(value: float, ws: int, device=None) -> float:
    """The largest of every rank's value (the job's time is its slowest rank's);
    the value itself with one rank."""
    if ws <= 1:
        return value
    import torch
    import torch.distributed as dist
    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def peaks():
    p = ROOT / "MEASURED_PEAKS.json"
    if p.exists():
        d = json.loads(p.read_text())
        return (float(d["hbm_gbs"]), float(d["bf16_tflops"]), float(d.get("bf16_tflops_sustained",
                d["bf16_tflops"])), "measured")
    return FALLBACK_HBM_GBS, FALLBACK_BF16_TFLOPS, 1700.0, "fallback"


def kernel_source_hash(files=None) -> str:
    """Hash of the listed kernel sources (names under the package's csrc/; all
    of them when None)."""
    csrc = ROOT / "fp8_weight_only_gemm_gb300" / "csrc"
    paths = sorted(csrc.glob("*")) if files is None else [csrc / f for f in sorted(files)]
    h = hashlib.sha256()
    for f in paths:
        h.update(f.name.encode())
        h.update(f.read_bytes())
    return h.hexdigest()[:16]


def recorded_traffic(workload: str):
    """DRAM bytes per launch from the committed ncu summary, if it was taken on
    the current kernel sources; None otherwise."""
    p = ROOT / "profiles" / "traffic.json"
    if not p.exists():
        return None
    try:
        d = json.loads(p.read_text())
        e = d.get(workload)
        if e and e.get("kernel_source_hash") == kernel_source_hash(e.get("kernel_sources")):
            return float(e["dram_bytes_per_launch"])
    except Exception:
        return None
    return None


def config_dict(name: str, wl, path: str) -> dict:
    """The workload's description, identical in both arms."""
    return {"workload": name, "path": path, "M": wl.M, "N": wl.N, "K": wl.K, "a_row_stride": wl.lda,
            "c_row_stride": wl.ldc, "seed": wl.seed}


class ClockSampler:
    """nvidia-smi clocks and throttle reasons, sampled every 100 ms."""

    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.samples = []
        self._stop = threading.Event()
        self._t = None

    def _run(self):
        while not self._stop.is_set():
            try:
                out = subprocess.run(["nvidia-smi", f"--id={self.index}", f"--query-gpu={self.QUERY}",
                                      "--format=csv,noheader,nounits"], capture_output=True,
                                     text=True, timeout=5).stdout.strip()
                if out:
                    self.samples.append([x.strip() for x in out.split(",")])
            except Exception:
                pass
            self._stop.wait(0.1)

    def __enter__(self):
        self._t = threading.Thread(target=self._run, daemon=True)
        self._t.start()
        return self

    def __exit__(self, *a):
        self._stop.set()
        if self._t:
            self._t.join(timeout=10)

    def summary(self):
        if not self.samples:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no nvidia-smi samples"], "samples": 0}
        sm = [float(s[1]) for s in self.samples if s[1].replace(".", "").isdigit()]
        mx = [float(s[2]) for s in self.samples if s[2].replace(".", "").isdigit()]
        pw = [float(s[3]) for s in self.samples if s[3].replace(".", "").isdigit()]
        reasons = set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for s in self.samples:
            for i, n in enumerate(names):
                if len(s) > 5 + i and s[5 + i].lower() == "active":
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(mx) if mx else None, "reasons": sorted(reasons),
                "samples": len(self.samples),
                "power_w_median": statistics.median(pw) if pw else None,
                "note": "every sample was taken while timed regions were running"}


# --------------------------------------------------------------- our arm --
def resolve_workload(args):
    """The named workload, or with --tokens the same workload at another token
    count M; its name then carries the new count (multitile_m128_... at 256
    tokens is multitile_m256_...), and so do its traffic record and JSON line."""
    wl = workloads.CONFIGS[args.workload]
    if args.tokens is None or args.tokens == wl.M:
        return args.workload, wl
    name = re.sub(r"_m\d+_", f"_m{args.tokens}_", args.workload, count=1)
    return name, dataclasses.replace(wl, name=name, M=args.tokens)


def graph_split(K: int, nsets: int, cap: int = 512):
    """A graph of G steps replayed q times plus a graph of the r = K - q*G rest:
    G = K up to `cap` steps, else the largest multiple of the buffer-set count
    that fits, so every replay of the full graph walks whole rotations."""
    if K <= cap:
        return K, 1, 0
    G = max(nsets, cap // nsets * nsets)
    q, r = divmod(K, G)
    return G, q, r


class Runner:
    """Graph capture and event timing on one stream."""

    def __init__(self, torch, dev, stream, ws):
        self.torch, self.dev, self.stream, self.ws = torch, dev, stream, ws

    def capture(self, fn, count: int):
        torch = self.torch
        g = torch.cuda.CUDAGraph()
        with torch.cuda.stream(self.stream):
            with torch.cuda.graph(g, stream=self.stream):
                for i in range(count):
                    fn(i)
        return g

    def barrier(self):
        if self.ws > 1:
            import torch.distributed as dist
            dist.barrier()

    def regions(self, replays, min_seconds: float, min_reps: int = 5, max_reps: int = 50000,
                batch: int = 32):
        """Time repeated regions; each region is `replays` (a list of graphs, replayed
        in order) between two events, after a pre-roll spin. Returns the region times
        in ms (at least min_reps of them, and at least min_seconds of GPU time in
        all, unless max_reps is reached)."""
        torch = self.torch
        times = []
        self.barrier()
        torch.cuda.synchronize(self.dev)
        with torch.cuda.stream(self.stream):
            while True:
                evs = []
                for _ in range(batch):
                    torch.cuda._sleep(PREROLL_CYCLES)
                    s = torch.cuda.Event(enable_timing=True)
                    e = torch.cuda.Event(enable_timing=True)
                    s.record(self.stream)
                    for g in replays:
                        g.replay()
                    e.record(self.stream)
                    evs.append((s, e))
                torch.cuda.synchronize(self.dev)
                times += [s.elapsed_time(e) for s, e in evs]
                if len(times) >= max_reps or (len(times) >= min_reps and sum(times) / 1e3 >= min_seconds):
                    break
                # grow the batch once the region length is known (fewer host syncs)
                per = max(statistics.median(times), 1e-3)
                batch = int(min(512, max(batch, 0.05 / (per / 1e3 + 30e-6))))
        self.barrier()
        return times


def measure_workload(name, wl, args, ctx, K: int, headline: bool):
    """Time one workload through the product entry point; returns its entry of
    the JSON line (and, for the headline, the clock record and e2e)."""
    torch, w8, lib = ctx["torch"], ctx["w8"], ctx["lib"]
    dev, stream, sh, flags, l2, sms = (ctx["dev"], ctx["stream"], ctx["sh"], ctx["flags"], ctx["l2"],
                                       ctx["sms"])
    runner = ctx["runner"]
    hbm, bf16, bf16_sus, src = peaks()
    case = workloads.make_case(wl)
    set_bytes = wl.N * wl.K + case.A.numel() * 2 + case.C0.numel() * 2 + case.scale.numel() * 4
    nsets = max(2, -(-3 * l2 // set_bytes))
    A0, W0, S0, C0 = (case.A.to(dev), case.W.to(dev), case.scale.to(dev), case.C0.to(dev))
    sets = [(A0.clone(), W0.clone(), S0.clone(), C0.clone()) for _ in range(nsets)]
    del A0, W0, S0, C0
    w8a8 = args.path == "w8a8"
    qsets = [w8.quantize_activations(A[:, :wl.K]) for (A, _, _, _) in sets] if w8a8 else None
    # a workspace every plan fits in; the workspace path's own choice for it, or
    # (--stream-k, 3..32 tokens) the forced persistent stream-K plan
    wsb = max(16, w8.workspace_bytes_for(wl.M, wl.N, wl.K), w8.workspace_bytes(wl.M, wl.K))
    wss = [torch.zeros(wsb, dtype=torch.uint8, device=dev) for _ in range(nsets)] if not w8a8 else None
    stream_k = not w8a8 and args.stream_k and 3 <= wl.M <= 32
    forced = w8.plan_variant(wl.M, wl.N, wl.K, w8.VARIANT_STREAM, 0, 0, sms) if stream_k else None
    if w8a8:   # w8a16_gemm_w8a8's own choice: the decode kernel where its rule admits the shape
        auto = w8.plan_current(wl.M, wl.N, wl.K)
        plan = (auto if auto["variant"] == w8.VARIANT_GEMV else
                w8.plan_variant(wl.M, wl.N, wl.K, w8.VARIANT_W8A8, 0, 0, sms).as_dict())
    else:
        plan = forced.as_dict() if stream_k else w8.plan_ws(wl.M, wl.N, wl.K, wsb)
    presplit = not w8a8 and plan["variant"] in (w8.VARIANT_PRESPLIT, w8.VARIANT_STREAM)
    gemm_launches = 2 if plan.get("tail_tiles") else 1
    launches_per_step = (1 if (w8a8 or presplit) else 0) + gemm_launches

    def ck(rc):
        if rc != 0:
            raise RuntimeError(w8.last_error())

    def gemm8(i, fl=None):
        A, W, S, C = sets[i % nsets]
        q, qs = qsets[i % nsets]
        ck(lib.w8a16_gemm_w8a8(q.data_ptr(), q.stride(0), qs.data_ptr(), qs.stride(0), W.data_ptr(),
                               S.data_ptr(), C.data_ptr(), C.stride(0), wl.M, wl.N, wl.K,
                               flags if fl is None else fl, sh))

    def split_only(i):
        A, _, _, _ = sets[i % nsets]
        ws_ = wss[i % nsets]
        ck(lib.w8a16_split_activations(A.data_ptr(), A.stride(0), wl.M, wl.K, ws_.data_ptr(), ws_.numel(), sh))

    def terms_only(i):
        _, W, S, C = sets[i % nsets]
        ws_ = wss[i % nsets]
        ck(lib.w8a16_gemm_split_terms(ws_.data_ptr(), ws_.numel(), W.data_ptr(), S.data_ptr(), C.data_ptr(),
                                      C.stride(0), wl.M, wl.N, wl.K, flags, sh))

    def call(i, fl=None):
        A, W, S, C = sets[i % nsets]
        fl = flags if fl is None else fl
        if w8a8:
            q, qs = qsets[i % nsets]
            ck(lib.w8a16_quantize_activations(A.data_ptr(), A.stride(0), wl.M, wl.K, q.data_ptr(),
                                              qs.data_ptr(), qs.stride(0), sh))
            gemm8(i, fl)
            return
        ws_ = wss[i % nsets]
        ck(lib.w8a16_gemm_ws(A.data_ptr(), A.stride(0), W.data_ptr(), S.data_ptr(), C.data_ptr(),
                             C.stride(0), wl.M, wl.N, wl.K, ctypes.byref(forced) if forced is not None else None,
                             ws_.data_ptr(), ws_.numel(), fl, sh))

    # ---- graphs: a region of exactly K steps = q replays of G steps + r steps
    G, q, r = graph_split(K, nsets)
    with torch.cuda.stream(stream):
        for i in range(min(G, 2 * nsets)):   # the launch path and the planner's caches, outside capture
            call(i)
        if presplit and not stream_k:         # the kernel-only entry points too (set 0 holds a split)
            split_only(0)
            terms_only(0)
        elif w8a8:
            gemm8(0)
    torch.cuda.synchronize(dev)
    full = runner.capture(call, G)
    rest = runner.capture(call, r) if r else None
    region = [full] * q + ([rest] if rest else [])
    # kernel-only graphs of the dominant kernel (and of the pre-pass)
    kgraphs = {}
    if presplit and not stream_k:   # (the stream-K kernel has no kernel-only entry point)
        kgraphs["gemm"] = runner.capture(terms_only, G)
        kgraphs["split"] = runner.capture(split_only, G)
    elif w8a8:
        kgraphs["gemm"] = runner.capture(gemm8, G)
    torch.cuda.synchronize(dev)

    # ---- warm-up: every graph once, then at least W steps in whole replays
    with torch.cuda.stream(stream):
        for g in [full] + ([rest] if rest else []) + list(kgraphs.values()):
            g.replay()
        for _ in range(max(1, -(-args.warmup // G))):
            full.replay()
    torch.cuda.synchronize(dev)

    # ---- timed regions
    min_seconds = args.min_seconds if headline else args.config_seconds
    clk = ClockSampler(ctx["local"]) if headline else None
    if clk:
        clk.__enter__()
    try:
        times = runner.regions(region, min_seconds)
    finally:
        if clk:
            clk.__exit__()
    med_ms = max_over_ranks(statistics.median(times), runner.ws, dev)
    step_s = med_ms / 1e3 / K
    bytes_step = wl.roofline_bytes()
    out = {
        "M": wl.M, "N": wl.N, "K": wl.K,
        "steps_per_region": K, "regions": len(times),
        "us_per_step": step_s * 1e6,
        "region_ms": {"min": min(times), "median": statistics.median(times), "max": max(times)},
        "gbs": bytes_step / step_s / 1e9,
        "tflops": wl.flops() / step_s / 1e12,
        "frac_hbm": bytes_step / step_s / 1e9 / hbm,
        "roofline_bytes": bytes_step,
        "path": ("activation quantiser + W8A8 GEMM" if w8a8 else
                 "w8a16_gemm_ws: split pre-pass + FP8 x FP8 GEMM on two terms, persistent stream-K grid"
                 if stream_k else
                 "w8a16_gemm_ws: split pre-pass + FP8 x FP8 GEMM on two terms" if presplit else
                 "w8a16_gemm_ws: one launch of the two-term FP8 kernel" if plan["variant"] == 3 else
                 "w8a16_gemm_ws: one launch of the decode kernel" if plan["variant"] == 6 else
                 "w8a16_gemm_ws: one launch of the BF16 kernel"),
        "launches_per_step": launches_per_step,
        "plan": plan,
    }
    # both bounds where the tensor work is not negligible
    t_hbm = bytes_step / (hbm * 1e9)
    t_tensor = wl.flops() / (bf16 * 1e12)
    out["bound_us"] = {"hbm": t_hbm * 1e6, "bf16_tensor": t_tensor * 1e6}
    out["bound"] = "hbm" if t_hbm >= t_tensor else "tensor"
    out["frac_of_binding_bound"] = max(t_hbm, t_tensor) / step_s

    # ---- the dominant kernel alone
    if kgraphs:
        kt = {k: statistics.median(runner.regions([g], 0.1 if not headline else 0.5)) / G * 1e3
              for k, g in kgraphs.items()}
        kbytes = w8a8_gemm_bytes(wl, 2 if presplit else 1)
        out["kernel"] = {"name": ("w8a16_w8a8_kernel (terms 2)" if presplit else
                                  "w8a16_gemv_kernel (E4M3 activations)" if plan["variant"] == w8.VARIANT_GEMV else
                                  "w8a16_w8a8_kernel (terms 1)"),
                         "us": kt["gemm"], "bytes": kbytes, "gbs": kbytes / kt["gemm"] / 1e3,
                         "frac_hbm": kbytes / kt["gemm"] / 1e3 / hbm,
                         "timing": f"{G} launches of the GEMM alone replayed back to back from a graph"
                                   f"{' (programmatic dependent launches)' if flags else ''}"}
        if presplit:
            out["kernel"]["split_prepass_us"] = kt["split"]
            out["kernel"]["split_timing"] = f"{G} launches of split_act_kernel alone from a graph"
    elif stream_k:
        out["kernel"] = {"name": "split_act_kernel + w8a16_w8a8_kernel (terms 2, stream-K)",
                         "us": step_s * 1e6, "bytes": bytes_step, "gbs": bytes_step / step_s / 1e9,
                         "frac_hbm": bytes_step / step_s / 1e9 / hbm,
                         "timing": "the step: the split pre-pass and the stream-K kernel"}
    else:
        out["kernel"] = {"name": {3: "w8a16_tc8_kernel", 6: "w8a16_gemv_kernel"}.get(plan["variant"],
                                                                                       "w8a16_tc_kernel"),
                         "us": step_s * 1e6,
                         "bytes": bytes_step, "gbs": bytes_step / step_s / 1e9,
                         "frac_hbm": bytes_step / step_s / 1e9 / hbm,
                         "timing": "the step is this kernel's launch" +
                                   ("es (whole tiles + split-K tail)" if gemm_launches > 1 else " alone")}
    traffic_key = name + ("/w8a8" if w8a8 else "/stream" if stream_k else "/presplit" if presplit else "")
    out["kernel"]["traffic"] = recorded_traffic(traffic_key)
    out["gpu_launches_timed"] = len(times) * K * launches_per_step

    extra = {"case": case, "sets": sets, "clocks": clk.summary() if clk else None, "nsets": nsets,
             "set_bytes": set_bytes, "G": G, "call": call, "presplit": presplit, "w8a8": w8a8}
    return out, extra


def e2e_host(wl, case, sets, ctx, steps: int, w8a8: bool, call) -> dict:
    """The same metric end to end through the host-buffer entry point."""
    torch, w8 = ctx["torch"], ctx["w8"]
    dev, stream = ctx["dev"], ctx["stream"]
    A_h = case.A.pin_memory()
    W_h = case.W.pin_memory()
    S_h = case.scale.pin_memory()
    C_h = case.C0.clone().pin_memory()
    dA, dW, dS, dC = sets[0]
    e_steps = max(3, min(steps, 200))

    if w8a8:
        def host_step():
            dA.copy_(A_h, non_blocking=True)
            dW.copy_(W_h, non_blocking=True)
            dS.copy_(S_h, non_blocking=True)
            call(0, 0)
            C_h.copy_(dC, non_blocking=True)
    else:
        def host_step():
            w8.gemm_host(A_h[:, :wl.K], W_h, S_h, C_h[:, :wl.N], dA, dW, dS, dC, stream=stream)

    with torch.cuda.stream(stream):
        for _ in range(3):
            host_step()
        torch.cuda.synchronize(dev)
        s2, e2 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        s2.record(stream)
        for _ in range(e_steps):
            host_step()
        e2.record(stream)
    torch.cuda.synchronize(dev)
    e_sec = s2.elapsed_time(e2) / 1e3
    h2d = case.A.numel() * 2 + wl.N * wl.K + case.scale.numel() * 4
    d2h = case.C0.numel() * 2
    return {"value": wl.roofline_bytes() * e_steps / e_sec / 1e9, "unit": "GB/s",
            "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "steps": e_steps,
            "ms_per_step": e_sec * 1e3 / e_steps,
            "path": ("pinned host copies + quantiser + W8A8 GEMM + copy of C, one stream" if w8a8 else
                     "w8a16_gemm_host: pinned host copies of A (full pitch), W and block_scale, the GEMM, "
                     "the copy of C (full pitch), one stream")}


def bench_gpu(args, ws, rank, local):
    import torch
    import fp8_weight_only_gemm_gb300 as w8
    from fp8_weight_only_gemm_gb300.build import build_library

    build_library()
    lib = w8.load()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    props = torch.cuda.get_device_properties(dev)
    stream = torch.cuda.Stream(dev)
    ctx = {"torch": torch, "w8": w8, "lib": lib, "dev": dev, "stream": stream, "sh": int(stream.cuda_stream),
           "flags": w8.FLAG_PDL if args.pdl == "on" else 0, "local": local,
           "l2": int(getattr(props, "L2_cache_size", 126 * 2 ** 20)), "sms": props.multi_processor_count,
           "runner": Runner(torch, dev, stream, ws)}
    hbm, bf16, bf16_sus, src = peaks()
    name, wl = resolve_workload(args)

    head, extra = measure_workload(name, wl, args, ctx, args.steps, headline=True)
    e2e = None if args.no_e2e else e2e_host(wl, extra["case"], extra["sets"], ctx, args.steps, extra["w8a8"],
                                            extra["call"])
    del extra["sets"]
    configs = {name: head}
    if args.configs == "all":
        for other in workloads.CONFIG_ORDER:
            if other == name:
                continue
            owl = workloads.CONFIGS[other]
            est = owl.roofline_bytes() / (0.5 * hbm * 1e9)   # a generous guess of a step's time
            k = max(5, min(args.steps, int(CONFIG_REGION_SECONDS / est)))
            torch.cuda.empty_cache()
            configs[other], _ = measure_workload(other, owl, args, ctx, k, headline=False)
            torch.cuda.empty_cache()

    st = w8.device_status(stream=stream)
    if st[0] != 0:
        raise RuntimeError(f"device status {st}: a bounded wait ran out during the benchmark")

    step_s = head["us_per_step"] / 1e6
    kern = head["kernel"]
    w8a8, presplit = extra["w8a8"], extra["presplit"]
    line = {
        "metric": METRIC_W8A8 if w8a8 else METRIC, "value": head["gbs"] * ws, "unit": "GB/s", "n_gpus": ws,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": step_s * 1e3, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "arithmetic": ARITHMETIC["w8a8" if w8a8 else "two_term"],
        "data": "synthetic",
        "config": config_dict(name, wl, args.path),
        "parallelism": f"replicas x{ws} (no collective)" if ws > 1 else "single GPU",
        "method": {
            "l2": f"inputs rotate over {extra['nsets']} buffer sets ({extra['nsets'] * extra['set_bytes'] / 1e6:.0f} "
                  f"MB, >= 3x the {ctx['l2'] / 1e6:.0f} MB L2): weights stream from HBM every step",
            "graphs": f"steps replayed from CUDA graphs of {extra['G']} launches; every graph replayed once "
                      f"and >= {args.warmup} warm-up steps run before timing",
            "timing": f"median of {head['regions']} timed regions of exactly {args.steps} steps, each between "
                      "two CUDA events on the launching stream after a pre-roll spin kernel; all regions "
                      "bracketed by a barrier and torch.cuda.synchronize(); max over ranks",
            "launch": ("programmatic dependent launch (W8A16_FLAG_PDL): each call's weight prefetch overlaps "
                       "the previous call's tail" if ctx["flags"] else "plain stream order"),
            "plan": head["plan"],
        },
        "tflops": head["tflops"] * ws,
        "roofline": {"bound": "hbm", "achieved": kern["gbs"], "peak": hbm, "unit": "GB/s",
                     "frac": kern["gbs"] / hbm, "traffic": kern["traffic"],
                     "peak_source": f"{src}: HBM copy bandwidth (MEASURED_PEAKS.json hbm_gbs)" if src == "measured"
                                    else "fallback HBM figure",
                     "kernel": kern["name"], "kernel_us": kern["us"], "kernel_timing": kern["timing"],
                     "bytes_per_launch": kern["bytes"],
                     "tensor_frac_of_bf16_peak": head["tflops"] / bf16},
        "configs": configs,
        "gpu_launches": head["gpu_launches_timed"],
        "clocks": extra["clocks"],
        "e2e": e2e,
    }
    if presplit:
        line["roofline"]["split_prepass_us"] = kern.get("split_prepass_us")
    return line


# ----------------------------------------------------------- CPU oracle --
def oracle_step(wl, path: str, threads: int):
    """One full call of the workload on the CPU oracle (for w8a8: its activation
    quantiser, then its W8A8 product)."""
    import oracle
    case = workloads.make_case(wl)
    o = oracle.get()
    A, W, S, C0 = case.A_np(), case.W_np(), case.scale_np(), case.C0_np()
    if path == "w8a8":
        def step():
            q, qs = o.quantize_activations(A, wl.M, wl.K, a_row_stride=wl.lda)
            o.w8a8_gemm(q, qs, W, S, wl.M, wl.N, wl.K, C=C0, c_row_stride=wl.ldc, threads=threads)
    else:
        def step():
            o.gemm(A, W, S, wl.M, wl.N, wl.K, a_row_stride=wl.lda, C=C0, c_row_stride=wl.ldc,
                   threads=threads)
    return step


def oracle_rate(wl, seconds: float, threads: int | None = None, path: str = "w8a16"):
    """Time the CPU oracle on a bounded sample of the workload: as many full calls
    as fit in about `seconds` (at least one)."""
    threads = threads or os.cpu_count() or 1
    step = oracle_step(wl, path, threads)
    t0 = time.perf_counter()
    step()
    t1 = time.perf_counter() - t0
    reps = max(1, int(seconds / max(t1, 1e-6)))
    t0 = time.perf_counter()
    for _ in range(reps):
        step()
    dt = (time.perf_counter() - t0) / reps
    return wl.roofline_bytes() / dt / 1e9, dt, reps, threads


def cpu_baseline(wl, name: str, path: str, seconds: float) -> dict:
    """The oracle as it stands on this host: as many full calls as fit in about
    `seconds` on all cores, then again on one core where a single full call on one
    core fits in the same budget (otherwise that part is left out)."""
    v, dt, reps, thr = oracle_rate(wl, seconds, path=path)
    out = {"value": v, "unit": "GB/s", "cores": thr, "kind": "oracle",
           "sample": f"{reps} full calls of {name} "
                     f"{'(quantiser + W8A8 product) ' if path == 'w8a8' else ''}"
                     f"({dt * 1e3:.1f} ms each) on the CPU oracle"}
    if thr > 1 and dt * thr <= seconds:
        v1, dt1, reps1, _ = oracle_rate(wl, seconds, threads=1, path=path)
        out["single_core"] = {"value": v1, "unit": "GB/s", "cores": 1,
                              "sample": f"{reps1} full calls ({dt1 * 1e3:.1f} ms each) on one core"}
    return out


def bench_reference(args):
    name, wl = resolve_workload(args)
    threads = os.cpu_count() or 1
    step = oracle_step(wl, args.path, threads)

    for _ in range(args.warmup):
        step()
    t0 = time.perf_counter()
    for _ in range(args.steps):
        step()
    sec = time.perf_counter() - t0
    v = wl.roofline_bytes() * args.steps / sec / 1e9
    return {"impl": "reference", "metric": METRIC_W8A8 if args.path == "w8a8" else METRIC, "value": v,
            "unit": "GB/s", "n_gpus": 1, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": sec * 1e3 / args.steps, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f64", "arithmetic": ARITHMETIC["oracle"], "data": "synthetic",
            "config": config_dict(name, wl, args.path),
            "cpu_baseline": {"value": v, "unit": "GB/s", "cores": threads, "kind": "oracle",
                             "sample": f"{args.steps} full calls of {name} on the CPU oracle "
                                       f"({'quantiser + W8A8 product, ' if args.path == 'w8a8' else ''}"
                                       "FP64, plain k-order loops)"},
            "e2e": {"value": v, "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
            "note": "no runnable reference implementation exists (the pages ship host code only); "
                    "the reference arm is the CPU oracle"}


def main():
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=None)
    ap.add_argument("--warmup", type=int, default=None)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD, choices=workloads.CONFIG_ORDER)
    ap.add_argument("--tokens", type=int, default=None,
                    help="run the workload at this token count M instead of its own")
    ap.add_argument("--configs", choices=["all", "none"], default="all",
                    help="also measure every other workload of the metric (entries under 'configs')")
    ap.add_argument("--min-seconds", type=float, default=2.0,
                    help="GPU time spent in the headline workload's timed regions (at least 5 regions)")
    ap.add_argument("--config-seconds", type=float, default=0.5,
                    help="GPU time spent in each other workload's timed regions")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--stream-k", action="store_true",
                    help="force the persistent stream-K plan on the 3..32-token workloads (never the "
                         "planner's choice: slower on GB300)")
    ap.add_argument("--path", choices=["w8a16", "w8a8"], default="w8a16",
                    help="w8a8: activation quantiser + W8A8 GEMM per step")
    ap.add_argument("--pdl", choices=["on", "off"], default="on",
                    help="queue the timed calls with W8A16_FLAG_PDL (weights are read-only)")
    ap.add_argument("--cpu-seconds", type=float, default=10.0,
                    help="bounded CPU-oracle sample for cpu_baseline")
    args = ap.parse_args()
    if args.tokens is not None and not 1 <= args.tokens <= 4096:
        ap.error("--tokens must be in 1..4096")
    ws, rank, local = dist_env()
    if args.impl == "reference":
        if args.steps is None:
            args.steps = 20
        if args.warmup is None:
            args.warmup = 3
        if rank != 0:
            return
        print(json.dumps(bench_reference(args)), flush=True)
        return
    if args.steps is None:
        args.steps = 20000
    if args.warmup is None:
        args.warmup = 2000
    args.warmup = max(3, args.warmup)
    if args.steps < 1:
        ap.error("--steps must be at least 1")
    if ws > 1:
        import torch
        import torch.distributed as dist
        dist.init_process_group("nccl" if torch.cuda.is_available() else "gloo")
    line = bench_gpu(args, ws, rank, local)
    if rank == 0:
        if args.cpu_seconds > 0:
            name, wl = resolve_workload(args)
            line["cpu_baseline"] = cpu_baseline(wl, name, args.path, args.cpu_seconds)
        print(json.dumps(line), flush=True)
    if ws > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
