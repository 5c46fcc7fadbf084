"""The allocation-free entry point (w8a16_gemm_noalloc): the pre-split W8A16 path on
the library's fixed device scratch buffer. Two calls in a row reuse the buffer; each
matches the oracle, and the same bits as the workspace entry point with its own
buffer. Sizes past the buffer are refused before any device work."""
from __future__ import annotations

import numpy as np
import pytest
import torch

import workloads
from parity import compare, oracle_full

ERR_RANGE, ERR_NULL = -8, -6


@pytest.fixture(scope="module")
def lib():
    from fp8_weight_only_gemm_gb300.build import build_library
    from fp8_weight_only_gemm_gb300 import binding
    build_library()
    return binding.load()


def test_declared_and_sized(lib):
    from fp8_weight_only_gemm_gb300 import binding
    assert "w8a16_gemm_noalloc" in binding.header_functions()
    assert binding.noalloc_scratch_bytes() == 32 << 20


def test_refuses_sizes_past_the_buffer(lib):
    from fp8_weight_only_gemm_gb300 import binding
    M, K = 2048, 8192                          # 2*M*K + factors > 32 MiB
    assert binding.workspace_bytes(M, K) > binding.noalloc_scratch_bytes()
    rc = binding.gemm_noalloc_ptr(0x1000, K, 0x2000, 0x3000, 0x4000, 256, M, 256, K)
    assert rc == ERR_RANGE and "scratch" in binding.last_error()
    # the page's checks and the pointer checks still come first
    assert binding.gemm_noalloc_ptr(0x1000, 260, 0x2000, 0x3000, 0x4000, 256, 32, 256, 256) == -4
    assert binding.gemm_noalloc_ptr(0, 256, 0x2000, 0x3000, 0x4000, 256, 32, 256, 256) == ERR_NULL


@pytest.mark.gpu
def test_two_calls_in_a_row(lib):
    """Back-to-back calls on one stream (the second's split overwrites the buffer the
    first read), a token count without scratch in between."""
    from fp8_weight_only_gemm_gb300 import binding
    cases = [workloads.make_case("strided_m32_n14336_k5120", N=1024, K=2048, seed=901),
             workloads.make_case("skinny_qkv_m8_n12288_k4096", N=512, K=1024, seed=902),
             workloads.make_case("multitile_m128_n28672_k8192", M=100, N=768, K=1536, seed=903)]
    outs = []
    for case in cases:
        wl = case.wl
        A, W, S, C = case.A.cuda(), case.W.cuda(), case.scale.cuda(), case.C0.cuda()
        binding.gemm_noalloc(A[:, :wl.K], W, S, C[:, :wl.N])
        outs.append((case, C))
    torch.cuda.synchronize()
    for case, C in outs:
        wl = case.wl
        got = C.cpu().view(torch.int16).numpy().view(np.uint16)
        ref, exact, absum = oracle_full(case)
        compare(case, got, ref, exact, absum, split_k=16, label=f"noalloc M{wl.M}", variant=3)
        C2 = case.C0.cuda()
        binding.gemm_ws(case.A.cuda()[:, :wl.K], case.W.cuda(), case.scale.cuda(), C2[:, :wl.N])
        torch.cuda.synchronize()
        assert torch.equal(C2.view(torch.int16), C.view(torch.int16)), "differs from the workspace path"
    assert binding.device_status() == (0, 0, 0)
