"""A call queued with W8A16_FLAG_PDL behind a long kernel that lets dependents start
early must not charge that kernel's run time to its own bounded waits: each role
starts its time limit after the grid-dependency wait. The predecessor is the
library's wait self-test (one CTA whose wait runs out after 300 ms and records
W8A16_STATUS_WAIT_TIMEOUT with detail 0xFF); the calls behind it run with a 40 ms
limit in a child process (the limit is read once per process). Every call must
give the right result, and the only recorded failure must be the self-test's."""
from __future__ import annotations

import json
import os
import subprocess
import sys
from pathlib import Path

import pytest

pytestmark = pytest.mark.gpu
ROOT = Path(__file__).resolve().parents[1]

CHILD = r"""
import json, sys
import numpy as np
import torch
sys.path.insert(0, sys.argv[1])
sys.path.insert(0, sys.argv[1] + "/tests")
import workloads
from fp8_weight_only_gemm_gb300 import binding
from parity import compare, oracle_full

binding.load()
binding.device_status(clear=True)
out = []
# (M, variant): the two-term kernel, the pre-split path (FP8 x FP8 kernel), the BF16 kernel
for M, path in ((1, "gemm"), (8, "gemm"), (40, "ws"), (40, "gemm")):
    case = workloads.make_case("strided_m32_n14336_k5120", M=M, N=640, K=2048, a_row_stride=2056,
                               c_row_stride=650, seed=91 + M)
    wl = case.wl
    A, W, S, C = case.A.cuda(), case.W.cuda(), case.scale.cuda(), case.C0.cuda()
    ws = torch.empty(binding.workspace_bytes(M, wl.K), dtype=torch.uint8, device="cuda")
    torch.cuda.synchronize()
    binding.selftest_wait_timeout(300000)          # 300 ms, lets dependents start at once
    if path == "ws":
        binding.gemm_ws(A[:, :wl.K], W, S, C[:, :wl.N], workspace=ws, flags=binding.FLAG_PDL)
    else:
        binding.gemm(A[:, :wl.K], W, S, C[:, :wl.N], flags=binding.FLAG_PDL)
    torch.cuda.synchronize()
    st, where, detail = binding.device_status(clear=True)
    got = C.cpu().view(torch.int16).numpy().view(np.uint16)
    ref, exact, absum = oracle_full(case)
    compare(case, got, ref, exact, absum, split_k=16, label=f"after a long predecessor M={M} {path}",
            variant=3 if (M <= 16 or path == "ws") else 2)
    out.append({"M": M, "path": path, "status": st, "detail": detail})
print(json.dumps(out))
"""


def test_pdl_call_behind_a_long_kernel_keeps_its_own_time_limit():
    env = dict(os.environ, W8A16_WAIT_TIMEOUT_MS="40")
    r = subprocess.run([sys.executable, "-c", CHILD, str(ROOT)], cwd=ROOT, env=env, capture_output=True,
                       text=True, timeout=600)
    assert r.returncode == 0, r.stdout[-3000:] + r.stderr[-3000:]
    rows = json.loads(r.stdout.strip().splitlines()[-1])
    assert len(rows) == 4
    for row in rows:
        # the self-test's own time-out (detail 0xFF) is the only failure recorded
        assert row["status"] == 1 and row["detail"] == 0xFF, row
