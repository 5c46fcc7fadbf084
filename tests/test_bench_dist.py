"""The multi-process parts of bench.py on CPU with the gloo backend (world size 2):
the job time is the slowest rank's, and under torchrun the reference arm prints one
JSON line from rank 0 while the other rank exits without work. Also the host side of
--tokens (a workload at another token count keeps its recipe and carries the new
count in its name)."""
from __future__ import annotations

import json
import os
import socket
import subprocess
import sys
from pathlib import Path

import pytest

ROOT = Path(__file__).resolve().parents[1]


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank: int, ws: int, port: int, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    import torch.distributed as dist
    sys.path.insert(0, str(ROOT))
    import bench
    dist.init_process_group("gloo", rank=rank, world_size=ws)
    try:
        out.put((rank, bench.max_over_ranks(1.5 + rank, ws)))
    finally:
        dist.destroy_process_group()


def test_max_over_ranks_gloo():
    import torch.multiprocessing as mp
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    got = dict(q.get(timeout=10) for _ in range(2))
    assert got == {0: 2.5, 1: 2.5}


def test_max_over_ranks_single_process():
    sys.path.insert(0, str(ROOT))
    import bench
    assert bench.max_over_ranks(3.25, 1) == 3.25


def test_reference_arm_under_torchrun_prints_one_line():
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node=2",
           "--master-addr", "127.0.0.1", "--master-port", str(_free_port()), "bench.py", "--impl",
           "reference", "--gpus", "2", "--steps", "1", "--warmup", "0", "--workload", "tiny_m1_n256_k256"]
    r = subprocess.run(cmd, cwd=ROOT, capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1, r.stdout
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["config"]["workload"] == "tiny_m1_n256_k256"
    assert d["cpu_baseline"]["kind"] == "oracle" and d["value"] > 0


def test_tokens_override_names_the_workload():
    sys.path.insert(0, str(ROOT))
    import argparse
    import bench
    name, wl = bench.resolve_workload(argparse.Namespace(workload="multitile_m128_n28672_k8192", tokens=256))
    assert name == "multitile_m256_n28672_k8192" and wl.M == 256 and (wl.N, wl.K) == (28672, 8192)
    assert wl.outlier_frac == 0.01 and wl.seed == 4                 # the rest of the recipe is kept
    name, wl = bench.resolve_workload(argparse.Namespace(workload="decode_gemv_m1_n4096_k4096", tokens=None))
    assert name == "decode_gemv_m1_n4096_k4096" and wl.M == 1


def test_reference_arm_with_tokens():
    cmd = [sys.executable, "bench.py", "--impl", "reference", "--steps", "1", "--warmup", "0",
           "--workload", "tiny_m1_n256_k256", "--tokens", "3"]
    r = subprocess.run(cmd, cwd=ROOT, capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stderr[-2000:]
    d = json.loads([l for l in r.stdout.splitlines() if l.startswith("{")][0])
    assert d["config"]["workload"] == "tiny_m3_n256_k256" and d["config"]["M"] == 3
    bad = subprocess.run([sys.executable, "bench.py", "--impl", "reference", "--tokens", "0"], cwd=ROOT,
                         capture_output=True, text=True, timeout=300)
    assert bad.returncode != 0 and "--tokens" in bad.stderr


def test_cpu_baseline_all_cores_and_one():
    sys.path.insert(0, str(ROOT))
    import bench
    import workloads
    d = bench.cpu_baseline(workloads.CONFIGS["tiny_m1_n256_k256"], "tiny_m1_n256_k256", "w8a16", 0.3)
    assert d["kind"] == "oracle" and d["value"] > 0 and d["cores"] >= 1
    if d["cores"] > 1:
        assert d["single_core"]["cores"] == 1 and d["single_core"]["value"] > 0


def test_graph_split_covers_exactly_k_steps():
    sys.path.insert(0, str(ROOT))
    import bench
    for K, nsets in [(1, 25), (20, 25), (512, 3), (513, 25), (20000, 25), (20000, 2), (777, 600)]:
        G, q, r = bench.graph_split(K, nsets)
        assert q * G + r == K and G >= 1 and q >= 1 and 0 <= r < G
        if K > 512:
            assert G % nsets == 0 or G == nsets


def test_both_arms_print_the_same_config():
    sys.path.insert(0, str(ROOT))
    import argparse
    import bench
    import workloads
    args = argparse.Namespace(workload="strided_m32_n14336_k5120", tokens=None, path="w8a16", steps=1,
                              warmup=0)
    name, wl = bench.resolve_workload(args)
    ours = bench.config_dict(name, wl, args.path)
    small = workloads.CONFIGS["tiny_m1_n256_k256"]
    ref = bench.bench_reference(argparse.Namespace(workload="tiny_m1_n256_k256", tokens=None, path="w8a16",
                                                   steps=1, warmup=0))
    assert set(ref["config"]) == set(ours)
    assert ref["config"] == bench.config_dict("tiny_m1_n256_k256", small, "w8a16")
    assert ours["a_row_stride"] == 5184 and ours["c_row_stride"] == 14400
