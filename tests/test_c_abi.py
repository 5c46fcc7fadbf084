"""The boundary as a C program sees it: include/w8a16.h compiles as strict C11 and
C++17 with every warning an error, and a plain C client linked against
libw8a16.so (no Python, no torch) gets the page's argument checks, error strings,
the planner and the workspace size through the C ABI. Only host-side calls run:
the one entry point that would launch work must report that no usable device is
present, not fall back to anything (asked for only where torch sees no GPU)."""
from __future__ import annotations

import shutil
import subprocess
from pathlib import Path

import pytest

from fp8_weight_only_gemm_gb300.build import build_library

ROOT = Path(__file__).resolve().parent.parent
INCLUDE = ROOT / "include"

CLIENT = r"""
#include <stdio.h>
#include <string.h>
#include "w8a16.h"

int main(int argc, char **argv) {
    w8a16_plan_t p;
    int rc;
    printf("version %s\n", w8a16_version());
    /* the page's checks, in its order, each with its own code */
    printf("m0 %d\n", w8a16_check_args(NULL, 4096, NULL, NULL, NULL, 4096, 0, 4096, 4096));
    printf("k100 %d\n", w8a16_check_args(NULL, 4096, NULL, NULL, NULL, 4096, 1, 4096, 100));
    printf("pitch %d\n", w8a16_check_args(NULL, 4000, NULL, NULL, NULL, 4096, 1, 4096, 4096));
    printf("align %d\n", w8a16_check_args(NULL, 4100, NULL, NULL, NULL, 4096, 1, 4096, 4096));
    printf("n0 %d\n", w8a16_check_args(NULL, 4096, NULL, NULL, NULL, 4096, 1, 0, 4096));
    printf("good %d\n", w8a16_check_args(NULL, 4096, NULL, NULL, NULL, 4096, 1, 4096, 4096));
    rc = w8a16_check_args(NULL, 4096, NULL, NULL, NULL, 4096, 1, 4096, 100);
    printf("msg %d %s\n", rc, w8a16_last_error());
    printf("str %s\n", w8a16_strerror(W8A16_ERR_K_BLOCK));
    /* the planner: pure host code */
    memset(&p, 0, sizeof p);
    rc = w8a16_plan_for(1, 4096, 4096, 152, NULL, &p);
    printf("plan %d %d %u %u %u %u %u %u\n", rc, p.variant, p.token_tile, p.split_k, p.stages,
           p.grid[0], p.grid[1], p.cluster[0]);
    printf("ws %llu %llu\n", (unsigned long long)w8a16_workspace_bytes(32, 5120),
           (unsigned long long)w8a16_workspace_bytes(32, 100));
    printf("scratch %llu\n", (unsigned long long)w8a16_noalloc_scratch_bytes());
    /* a well-formed call with nothing to run it on: a device error, never a fallback.
     * Only on request: the pointers are placeholders that no GPU may be given. */
    if (argc > 1 && strcmp(argv[1], "--no-gpu-call") == 0) {
        rc = w8a16_gemm((const void *)0x1000, 4096, (const void *)0x2000, (const float *)0x3000,
                        (void *)0x4000, 4096, 1, 4096, 4096, NULL);
        printf("gemm %d\n", rc);
    }
    return 0;
}
"""


def _compilers():
    cc, cxx = shutil.which("gcc"), shutil.which("g++")
    if not cc or not cxx:
        pytest.skip("gcc/g++ not available")
    return cc, cxx


def test_header_is_strict_c_and_cxx(tmp_path):
    cc, cxx = _compilers()
    src_c = tmp_path / "h.c"
    src_c.write_text('#include "w8a16.h"\nint w8a16_header_probe(void) { return W8A16_OK; }\n')
    src_cpp = tmp_path / "h.cpp"
    src_cpp.write_text('#include "w8a16.h"\nint w8a16_header_probe() { return W8A16_OK; }\n')
    for comp, src, std in [(cc, src_c, "-std=c11"), (cc, src_c, "-std=c99"), (cxx, src_cpp, "-std=c++17")]:
        r = subprocess.run([comp, std, "-Wall", "-Wextra", "-Wpedantic", "-Werror", "-I", str(INCLUDE),
                            "-c", str(src), "-o", str(tmp_path / "h.o")], capture_output=True, text=True)
        assert r.returncode == 0, f"{comp} {std}:\n{r.stderr}"


def test_c_client_through_the_abi(tmp_path):
    cc, _ = _compilers()
    lib = build_library()
    src = tmp_path / "client.c"
    src.write_text(CLIENT)
    exe = tmp_path / "client"
    r = subprocess.run([cc, "-std=c11", "-Wall", "-Wextra", "-Werror", "-I", str(INCLUDE), str(src),
                        "-L", str(lib.parent), "-lw8a16", f"-Wl,-rpath,{lib.parent}", "-o", str(exe)],
                       capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
    import torch
    no_gpu = not torch.cuda.is_available()
    run = subprocess.run([str(exe)] + (["--no-gpu-call"] if no_gpu else []), capture_output=True,
                         text=True, timeout=60)
    assert run.returncode == 0, run.stderr
    out = dict(line.split(" ", 1) for line in run.stdout.strip().splitlines())
    assert out["version"].startswith("w8a16")
    assert out["m0"] == "-1" and out["k100"] == "-2" and out["pitch"] == "-3"
    assert out["align"] == "-4" and out["n0"] == "-5" and out["good"] == "0"
    assert out["msg"].startswith("-2 ") and "K=100" in out["msg"] and "128" in out["msg"]
    assert "multiple of 128" in out["str"]
    rc, variant, tn, split, stages, g0, g1, cl = map(int, out["plan"].split())
    assert rc == 0 and variant == 6 and tn == 2 and g1 == 1        # the decode kernel, one token tile
    assert g0 == 32 * split and cl == split and split == 4 and stages == 5   # 8 K steps per CTA
    ws_32, ws_bad = map(int, out["ws"].split())
    assert ws_32 == 2 * 32 * 5120 + 4 * 40 * 32 and ws_bad == 0
    assert int(out["scratch"]) == 32 << 20
    if no_gpu:
        assert out["gemm"] == "-9"                                 # W8A16_ERR_DEVICE
