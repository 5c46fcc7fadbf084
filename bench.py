#!/usr/bin/env python3
"""Benchmark of the GB300 W8A16 block-scaled GEMM.

One JSON line on stdout (rank 0). A step is one full W8A16 GEMM call on the
workload (default: decode GEMV M=1, N=K=4096, the configuration the headline
metric is quoted on), through w8a16_gemm_ws with a workspace: up to 16 tokens
that is one launch of the kernel that splits its own activation tiles; above,
the split pre-pass and the FP8 x FP8 kernel (two launches). Timing: W untimed warm-up steps, then exactly K steps,
bracketed by a barrier and torch.cuda.synchronize(), timed with CUDA events on
the launching stream. Steps rotate over B distinct input/output buffer sets
totalling at least 3x the L2 size, so every step streams its weights from HBM.
The K steps are replayed from CUDA graphs.

  value    = algorithmic bytes of all steps / timed seconds  (GB/s, whole job)
  e2e      = the same metric through the host-buffer entry point: per step the
             pinned host->device copies of A, W and block_scale, the GEMM, and the
             device->host copy of C
  roofline = the dominant (only) kernel against the measured HBM copy bandwidth
  cpu_baseline = the CPU oracle on the host cores, on a bounded sample

--path w8a8 times the W8A8 variant instead: a step is the per-token 128-group
activation quantiser followed by the FP8 x FP8 block-scaled GEMM (two launches);
`value` still counts the BF16-activation problem's bytes, and the roofline entry
is the GEMM kernel alone (its own algorithmic bytes: FP8 activation codes and
group scales instead of BF16 activations), timed from a graph of GEMM launches.

--tokens M runs a workload at another token count, e.g. the multi-tile workload at
M=256 (two 128-token tiles: one weight pass from HBM, the second token tile of each
weight tile reading it from L2); the JSON line then names it multitile_m256_...

--impl reference times the CPU oracle (the reference arm: there is no runnable
reference implementation) on the same workload and metric.
"""
from __future__ import annotations

import argparse
import dataclasses
import hashlib
import json
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


def w8a8_gemm_bytes(wl) -> int:
    """Algorithmic bytes of one W8A8 GEMM launch: E4M3 weights, block scales,
    E4M3 activation codes, FP32 group scales, BF16 output, each once."""
    kb = wl.K // 128
    return wl.N * wl.K + 4 * ((wl.N + 127) // 128) * kb + wl.M * wl.K + 4 * wl.M * kb + 2 * wl.M * wl.N
DEFAULT_WORKLOAD = "decode_gemv_m1_n4096_k4096"
FALLBACK_HBM_GBS = 6800.0
FALLBACK_BF16_TFLOPS = 1900.0


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
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no nvidia-smi samples"]}
        sm = [float(s[1]) for s in self.samples if s[1].replace(".", "").isdigit()]
        mx = [float(s[2]) for s in self.samples if s[2].replace(".", "").isdigit()]
        reasons = set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for s in self.samples:
            for i, n in enumerate(names):
                if len(s) > 5 + i and s[5 + i].lower() == "active":
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(mx) if mx else None, "reasons": sorted(reasons),
                "samples": len(self.samples)}


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


def bench_gpu(args, ws, rank, local):
    import torch
    import fp8_weight_only_gemm_gb300 as w8
    from fp8_weight_only_gemm_gb300.build import build_library

    build_library()
    w8.load()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    props = torch.cuda.get_device_properties(dev)
    name, wl = resolve_workload(args)
    case = workloads.make_case(wl)
    l2 = int(getattr(props, "L2_cache_size", 126 * 2 ** 20))
    set_bytes = wl.N * wl.K + case.A.numel() * 2 + case.C0.numel() * 2 + case.scale.numel() * 4
    nsets = max(2, -(-3 * l2 // set_bytes))
    A0, W0, S0, C0 = (case.A.to(dev), case.W.to(dev), case.scale.to(dev), case.C0.to(dev))
    sets = [(A0.clone(), W0.clone(), S0.clone(), C0.clone()) for _ in range(nsets)]
    del A0, W0, S0, C0
    w8a8 = args.path == "w8a8"
    qsets = [w8.quantize_activations(A[:, :wl.K]) for (A, _, _, _) in sets] if w8a8 else None
    presplit = not w8a8 and wl.M > 16
    wss = [torch.empty(max(16, w8.workspace_bytes(wl.M, wl.K)), dtype=torch.uint8, device=dev)
           for _ in range(nsets)] if not w8a8 else None
    sms = props.multi_processor_count
    plan = (w8.plan_variant(wl.M, wl.N, wl.K, w8.VARIANT_W8A8, 0, 0, sms).as_dict() if w8a8 else
            w8.plan_variant(wl.M, wl.N, wl.K, w8.VARIANT_PRESPLIT, 0, 0, sms).as_dict() if presplit else
            w8.plan_current(wl.M, wl.N, wl.K))
    # kernel launches per step: the quantiser or split pre-pass (W8A8, pre-split), then
    # the GEMM, which is two launches when the plan has a split-K tail
    launches_per_step = (1 if (w8a8 or presplit) else 0) + (2 if plan.get("tail_tiles") else 1)
    stream = torch.cuda.Stream(dev)
    lib = w8.load()
    sh = int(stream.cuda_stream)
    flags = w8.FLAG_PDL if args.pdl == "on" else 0

    def gemm8(i, fl):
        A, W, S, C = sets[i % nsets]
        q, qs = qsets[i % nsets]
        rc = lib.w8a16_gemm_w8a8(q.data_ptr(), q.stride(0), qs.data_ptr(), qs.stride(0), W.data_ptr(),
                                 S.data_ptr(), C.data_ptr(), C.stride(0), wl.M, wl.N, wl.K, fl, sh)
        if rc != 0:
            raise RuntimeError(w8.last_error())

    def call(i, fl=None):
        A, W, S, C = sets[i % nsets]
        fl = flags if fl is None else fl
        if w8a8:
            q, qs = qsets[i % nsets]
            rc = lib.w8a16_quantize_activations(A.data_ptr(), A.stride(0), wl.M, wl.K, q.data_ptr(),
                                                qs.data_ptr(), qs.stride(0), sh)
            if rc != 0:
                raise RuntimeError(w8.last_error())
            gemm8(i, fl)
            return
        ws = wss[i % nsets]
        rc = lib.w8a16_gemm_ws(A.data_ptr(), A.stride(0), W.data_ptr(), S.data_ptr(), C.data_ptr(),
                               C.stride(0), wl.M, wl.N, wl.K, None, ws.data_ptr(), ws.numel(), fl, sh)
        if rc != 0:
            raise RuntimeError(w8.last_error())

    # graphs of G steps (one kernel each); K = q*G + r
    G = min(args.steps, max(nsets, 64) // nsets * nsets) if args.steps >= nsets else args.steps
    G = max(1, G)
    q, r = divmod(args.steps, G)
    graphs = {}
    with torch.cuda.stream(stream):
        for (n, cnt) in [("full", G), ("rest", r)]:
            if cnt == 0:
                continue
            for i in range(cnt):        # warm the launch path outside capture
                call(i)
            torch.cuda.synchronize(dev)
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=stream):
                for i in range(cnt):
                    call(i)
            graphs[n] = g
        if w8a8:   # the GEMM kernel alone, for its roofline entry
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=stream):
                for i in range(G):
                    gemm8(i, flags)
            graphs["gemm"] = g
    torch.cuda.synchronize(dev)

    def run_steps(k):
        full, rest = divmod(k, G)
        for _ in range(full):
            graphs["full"].replay()
        for i in range(rest):
            call(i)

    with torch.cuda.stream(stream):
        run_steps(args.warmup)
    torch.cuda.synchronize(dev)
    if ws > 1:
        import torch.distributed as dist
        dist.barrier()
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with ClockSampler(local) as clk:
        with torch.cuda.stream(stream):
            # make the timed region long enough for the clock sampler when K is tiny
            torch.cuda.synchronize(dev)
            start.record(stream)
            for _ in range(q):
                graphs["full"].replay()
            if r:
                graphs["rest"].replay()
            end.record(stream)
        torch.cuda.synchronize(dev)
        if clk.samples == [] and args.steps > 0:
            time.sleep(0.25)
    ms = max_over_ranks(start.elapsed_time(end), ws, dev)
    if ws > 1:
        import torch.distributed as dist
        dist.barrier()
    kernel_bytes, kernel_us = wl.roofline_bytes(), ms * 1e3 / args.steps
    if w8a8:
        with torch.cuda.stream(stream):
            for _ in range(3):
                graphs["gemm"].replay()
            s1, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            reps = max(1, args.steps // G)
            s1.record(stream)
            for _ in range(reps):
                graphs["gemm"].replay()
            e1.record(stream)
        torch.cuda.synchronize(dev)
        kernel_bytes, kernel_us = w8a8_gemm_bytes(wl), s1.elapsed_time(e1) * 1e3 / (reps * G)
    sec = ms / 1e3
    bytes_step = wl.roofline_bytes()
    gbs = bytes_step * args.steps / sec / 1e9
    tflops = wl.flops() * args.steps / sec / 1e12
    hbm, bf16, bf16_sus, src = peaks()
    traffic = recorded_traffic(name + ("/w8a8" if w8a8 else "/presplit" if presplit else ""))
    kernel_gbs = kernel_bytes / kernel_us / 1e3

    # end to end through the host-buffer entry point
    e2e = None
    if not args.no_e2e and w8a8:
        A_h = case.A.pin_memory()
        W_h = case.W.pin_memory()
        S_h = case.scale.pin_memory()
        C_h = case.C0.clone().pin_memory()
        dA, dW, dS, dC = sets[0]
        e_steps = max(3, min(args.steps, 200))

        def host_step():
            dA.copy_(A_h, non_blocking=True)
            dW.copy_(W_h, non_blocking=True)
            dS.copy_(S_h, non_blocking=True)
            call(0, 0)
            C_h.copy_(dC, non_blocking=True)

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
        e2e = {"value": bytes_step * e_steps / e_sec / 1e9, "unit": "GB/s",
               "h2d_bytes_per_step": case.A.numel() * 2 + wl.N * wl.K + case.scale.numel() * 4,
               "d2h_bytes_per_step": case.C0.numel() * 2, "steps": e_steps,
               "ms_per_step": e_sec * 1e3 / e_steps,
               "path": "pinned host copies + quantiser + W8A8 GEMM + copy of C, one stream"}
    elif not args.no_e2e:
        A_h = case.A.pin_memory()
        W_h = case.W.pin_memory()
        S_h = case.scale.pin_memory()
        C_h = case.C0.clone().pin_memory()
        dA, dW, dS, dC = sets[0]
        e_steps = max(3, min(args.steps, 200))
        with torch.cuda.stream(stream):
            for _ in range(3):
                w8.gemm_host(A_h[:, :wl.K], W_h, S_h, C_h[:, :wl.N], dA, dW, dS, dC, stream=stream)
            torch.cuda.synchronize(dev)
            s2, e2 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            s2.record(stream)
            for _ in range(e_steps):
                w8.gemm_host(A_h[:, :wl.K], W_h, S_h, C_h[:, :wl.N], dA, dW, dS, dC, stream=stream)
            e2.record(stream)
        torch.cuda.synchronize(dev)
        e_sec = s2.elapsed_time(e2) / 1e3
        h2d = wl.M * wl.K * 2 + wl.N * wl.K + case.scale.numel() * 4
        d2h = wl.M * wl.N * 2
        e2e = {"value": bytes_step * e_steps / e_sec / 1e9, "unit": "GB/s",
               "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "steps": e_steps,
               "ms_per_step": e_sec * 1e3 / e_steps}

    st = w8.device_status(stream=stream)
    if st[0] != 0:
        raise RuntimeError(f"device status {st}: a bounded wait ran out during the benchmark")

    line = {
        "metric": METRIC_W8A8 if w8a8 else METRIC, "value": gbs, "unit": "GB/s", "n_gpus": ws, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms / args.steps, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "fp8" if w8a8 else "bf16",
        "data": "synthetic",
        "config": {"workload": name, "path": args.path, "M": wl.M, "N": wl.N, "K": wl.K,
                   "a_row_stride": wl.lda, "c_row_stride": wl.ldc, "seed": wl.seed,
                   "l2": f"inputs rotate over {nsets} buffer sets ({nsets * set_bytes / 1e6:.0f} MB, "
                         f">= 3x the {l2 / 1e6:.0f} MB L2): weights stream from HBM every step",
                   "graphs": f"steps replayed from CUDA graphs of {G} launches",
                   "launch": ("programmatic dependent launch (W8A16_FLAG_PDL): each call's weight "
                              "prefetch overlaps the previous call's tail" if flags else
                              "plain stream order"),
                   "plan": plan, "parallelism": f"replicas x{ws}" if ws > 1 else "single GPU"},
        "tflops": tflops,
        "roofline": {"bound": "hbm", "achieved": kernel_gbs, "peak": hbm, "unit": "GB/s",
                     "frac": kernel_gbs / hbm, "traffic": traffic,
                     "peak_source": f"{src}: hbm copy bandwidth",
                     "kernel": ("w8a16_w8a8_kernel (terms 1), timed alone" if w8a8 else
                                "split pre-pass + w8a16_w8a8_kernel (terms 2): the whole step" if presplit
                                else "w8a16_tc8_kernel, one launch per step"),
                     "kernel_us": kernel_us,
                     "bytes_per_launch": kernel_bytes,
                     "tensor_frac_of_bf16_peak": tflops / bf16},
        "gpu_launches": args.steps * launches_per_step,
        "clocks": clk.summary(),
        "e2e": e2e,
    }
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
    return {"impl": "reference", "metric": METRIC_W8A8 if args.path == "w8a8" else METRIC, "value": v, "unit": "GB/s", "n_gpus": 1,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": sec * 1e3 / args.steps,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic",
            "config": {"workload": name, "path": args.path, "M": wl.M, "N": wl.N, "K": wl.K},
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
    ap.add_argument("--no-e2e", action="store_true")
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
