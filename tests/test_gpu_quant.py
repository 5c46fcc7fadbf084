"""GPU parity of the weight block quantiser: codes and scales from the CUDA kernel,
through the C ABI, against the CPU oracle, bit for bit (a quantised code is an
integer decision taken in FP32 on both sides), and the quantised weights driving
the GEMM."""
from __future__ import annotations

import numpy as np
import pytest
import torch

import workloads
from parity import compare, oracle_full, run_gpu

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def o():
    import oracle
    return oracle.get()


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from fp8_weight_only_gemm_gb300.build import build_library
    from fp8_weight_only_gemm_gb300 import binding
    build_library()
    binding.load()
    yield


def _weights(N, K, ld, seed, dtype=torch.float32):
    g = torch.Generator().manual_seed(seed)
    w = torch.randn(N, ld, generator=g) * 0.02
    if N > 128 and K > 128:
        w[128:min(N, 256), 128:256] = 0.0                      # one zero block
    idx = torch.randperm(N * K, generator=g)[: max(1, N * K // 100)]
    w[:, :K].reshape(-1)[idx] *= 50.0                           # 1 % outliers
    return w.to(dtype)


@pytest.mark.parametrize("N,K,ld,dtype", [
    (256, 256, 256, torch.float32), (300, 384, 400, torch.float32), (130, 128, 132, torch.bfloat16),
    (1, 128, 128, torch.float32), (129, 1024, 1024, torch.bfloat16), (4096, 4096, 4096, torch.float32),
])
def test_quantizer_matches_oracle(o, N, K, ld, dtype):
    from fp8_weight_only_gemm_gb300 import binding
    w = _weights(N, K, ld, seed=N * 7 + K, dtype=dtype)
    wd = w.cuda()[:, :K]                                        # row pitch ld, first K used
    codes, scale = binding.quantize_weights(wd)
    torch.cuda.synchronize()
    rc, rs = o.quantize_weights(w.float().numpy(), N, K, w_row_stride=ld)
    got_c, got_s = codes.cpu().numpy(), scale.cpu().numpy()
    assert np.array_equal(got_s.view(np.uint32), rs.view(np.uint32)), "scales differ"
    bad = np.argwhere(got_c != rc)
    assert bad.size == 0, f"{len(bad)} codes differ, first at {bad[:3].tolist()}"


def test_quantizer_nan_weight(o):
    from fp8_weight_only_gemm_gb300 import binding
    w = _weights(128, 256, 256, seed=5)
    w[3, 200] = float("nan")
    codes, scale = binding.quantize_weights(w.cuda())
    rc, rs = o.quantize_weights(w.numpy(), 128, 256)
    assert np.array_equal(scale.cpu().numpy(), rs) and np.isfinite(rs).all()
    assert np.array_equal(codes.cpu().numpy(), rc)
    assert codes[3, 200].item() & 0x7F == 0x7F


def test_quantized_weights_drive_the_gemm():
    """Weights quantised on the GPU equal the input recipe's, so the GEMM on them
    meets the oracle like every workload does."""
    from fp8_weight_only_gemm_gb300 import binding
    g = torch.Generator().manual_seed(77)
    N, K, M = 1000, 1024, 8
    w = torch.randn(N, K, generator=g) * 0.02
    codes, scale = binding.quantize_weights(w.cuda())
    rc, rs = workloads.block_quantize_e4m3(w)
    assert torch.equal(codes.cpu(), rc) and torch.equal(scale.cpu(), rs)
    case = workloads.make_case("decode_gemv_m1_n4096_k4096", M=M, N=N, K=K, seed=78)
    case.W.copy_(codes.cpu())
    case.scale.copy_(scale.cpu())
    plan = binding.plan_current(M, N, K)
    got = run_gpu(case)
    ref, exact, absum = oracle_full(case)
    compare(case, got, ref, exact, absum, split_k=plan["split_k"], label="gpu-quantised W",
            variant=plan["variant"])


def test_quantizer_bandwidth_report():
    """Times the quantiser on a 16 Ki x 8 Ki FP32 matrix (informational: prints
    the achieved HBM GB/s; reads 4 B and writes 1 B per weight)."""
    from fp8_weight_only_gemm_gb300 import binding
    N, K = 16384, 8192
    w = torch.randn(N, K, device="cuda", dtype=torch.float32)
    for _ in range(3):
        binding.quantize_weights(w)
    torch.cuda.synchronize()
    s, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    s.record()
    reps = 10
    for _ in range(reps):
        binding.quantize_weights(w)
    e.record()
    torch.cuda.synchronize()
    us = s.elapsed_time(e) * 1e3 / reps
    gbs = N * K * 5 / us / 1e3
    print(f"\nquantiser {N}x{K} fp32: {us:.1f} us, {gbs:.0f} GB/s")
    assert gbs > 100
