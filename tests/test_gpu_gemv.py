"""GPU parity of the decode kernel (W8A16_VARIANT_GEMV, one or two tokens) against the
CPU oracle, element by element: every K-steps-per-CTA count 1..8 (so 0..3 steps
read from TMEM), splits 1..8, ragged N, row pitches, both token counts, every E4M3
code under log-uniform scales, NaN and zero blocks, run-to-run determinism and
chains of programmatic dependent launches (each call's A the previous call's C).
The two-term error bound of tests/parity.py applies (the same split as the
two-term kernel)."""
from __future__ import annotations

import numpy as np
import pytest
import torch

import workloads
from parity import bf16_to_f64 as bf, compare, oracle_full, run_gpu

pytestmark = pytest.mark.gpu
GEMV = 6


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from fp8_weight_only_gemm_gb300.build import build_library
    from fp8_weight_only_gemm_gb300 import binding
    build_library()
    binding.load()
    binding.device_status(clear=True)
    yield
    st, where, detail = binding.device_status()
    assert st == 0, f"a kernel recorded device status {st} (cta {where:#x}, wait {detail})"


def _plan(M, N, K, split):
    from fp8_weight_only_gemm_gb300 import binding
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    p = binding.plan_variant(M, N, K, GEMV, split, 0, sms)
    assert p.variant == GEMV and p.split_k == split
    return p


@pytest.mark.parametrize("M", [1, 2])
@pytest.mark.parametrize("K,split", [(128, 1), (256, 1), (640, 1), (1024, 1), (768, 1), (896, 1),
                                     (1024, 2), (2048, 4), (4096, 4), (4096, 8), (1280, 2), (1152, 3),
                                     (5120, 5), (8192, 8), (6016, 8)])
def test_steps_per_cta_and_splits(M, K, split):
    N = 300
    case = workloads.make_case("strided_m32_n14336_k5120", M=M, N=N, K=K, a_row_stride=K + 8,
                               c_row_stride=N + 5, seed=11 * K + split + M)
    got = run_gpu(case, plan=_plan(M, N, K, split))
    ref, exact, absum = oracle_full(case)
    compare(case, got, ref, exact, absum, split_k=split, label=f"gemv M{M} K{K} split{split}", variant=3)
    assert np.array_equal(got, run_gpu(case, plan=_plan(M, N, K, split))), "same plan, different bits"


@pytest.mark.parametrize("name", ["tiny_m1_n256_k256", "decode_gemv_m1_n4096_k4096"])
@pytest.mark.parametrize("M", [1, 2])
def test_workloads_on_the_decode_kernel(name, M):
    from fp8_weight_only_gemm_gb300 import binding
    case = workloads.make_case(name, M=M)
    wl = case.wl
    p = binding.plan_current(wl.M, wl.N, wl.K)
    assert p["variant"] == GEMV, p
    got = run_gpu(case)
    ref, exact, absum = oracle_full(case)
    compare(case, got, ref, exact, absum, split_k=p["split_k"], label=f"{name} M{M}", variant=3)
    assert not np.any(got.reshape(wl.M, wl.ldc)[:, :wl.N] == workloads.C_USED_SENTINEL)


@pytest.mark.parametrize("M,N,K,lda,ldc", [(1, 1, 128, 128, 1), (2, 7, 128, 136, 9), (1, 129, 256, 264, 130),
                                           (2, 255, 384, 392, 300), (1, 1000, 1024, 1024, 1000)])
def test_edge_shapes(M, N, K, lda, ldc):
    from fp8_weight_only_gemm_gb300 import binding
    case = workloads.make_case("tiny_m1_n256_k256", M=M, N=N, K=K, a_row_stride=lda, c_row_stride=ldc,
                               seed=M * 1000 + N + 7)
    p = binding.plan_current(M, N, K)
    assert p["variant"] == GEMV
    got = run_gpu(case)
    ref, exact, absum = oracle_full(case)
    compare(case, got, ref, exact, absum, split_k=16, label=f"gemv edge M{M} N{N} K{K}", variant=3)


@pytest.mark.parametrize("M", [1, 2])
def test_every_code_and_scale_range(M):
    case = workloads.random_codes_case(M, 384, 1024, seed=500 + M)
    got = run_gpu(case, plan=_plan(M, 384, 1024, 2))
    ref, exact, absum = oracle_full(case)
    compare(case, got, ref, exact, absum, split_k=2, label=f"gemv all-codes M{M}", variant=3)


def test_nan_weight_and_activation():
    case = workloads.make_case("tiny_m1_n256_k256", M=2, N=256, K=1024, seed=81)
    case.W[3, 200] = 0x7F          # step 1 of rank 0
    case.W[130, 1000] = 0xFF       # step 7 (read from a shared-memory slot)
    A = case.A.clone()
    A[1, 300] = float("inf")       # token 1, step 2
    case.A = A
    got = run_gpu(case, plan=_plan(2, 256, 1024, 1))
    ref, exact, absum = oracle_full(case)
    g = got.reshape(2, 256)
    isnan = ((g & 0x7F80) == 0x7F80) & ((g & 0x7F) != 0)
    # token 0: the two NaN weight rows; token 1: every output (an infinite activation)
    assert isnan[0, 3] and isnan[0, 130] and isnan[0].sum() == 2 and isnan[1].all()
    # the oracle agrees on token 0's pattern (token 1's exact sums are mostly +-Inf: on the
    # FP8 datapath a non-finite activation makes every output of its token NaN)
    assert np.array_equal(np.isnan(bf(ref.reshape(2, 256)[0])), isnan[0])
    # the other outputs within the bounds: the same case without the NaN codes
    sub = workloads.make_case("tiny_m1_n256_k256", M=1, N=256, K=1024, seed=81)
    sub.W[3, 200] = 0
    sub.W[130, 1000] = 0
    gs = run_gpu(sub, plan=_plan(1, 256, 1024, 1))
    rs, es, ab = oracle_full(sub)
    compare(sub, gs, rs, es, ab, split_k=1, label="gemv nan-free twin", variant=3)


def test_zero_block_and_zero_scale():
    case = workloads.make_case("skinny_qkv_m8_n12288_k4096", M=1, N=512, K=1024, zero_blocks=((2, 3),))
    assert float(case.scale[2, 3]) == 0.0
    got = run_gpu(case, plan=_plan(1, 512, 1024, 2))
    ref, exact, absum = oracle_full(case)
    compare(case, got, ref, exact, absum, split_k=2, label="gemv zero-block", variant=3)


@pytest.mark.parametrize("M", [1, 2])
def test_programmatic_launch_chain(M):
    """Six dependent decode calls (each call's A is the previous call's C, N = K =
    2048, split 4: 8 steps per CTA) with the programmatic-launch flag give the bits
    of the same chain without it, and each link matches the oracle on its input."""
    import fp8_weight_only_gemm_gb300 as w8
    K = 2048
    cases = [workloads.make_case("decode_gemv_m1_n4096_k4096", M=M, N=K, K=K, seed=400 + i) for i in range(6)]
    Ws = [c.W.cuda() for c in cases]
    Ss = [c.scale.cuda() for c in cases]
    x0 = cases[0].A.cuda()
    assert w8.plan_current(M, K, K)["variant"] == GEMV

    def chain(flags):
        xs = [x0]
        for W, S in zip(Ws, Ss):
            xs.append(w8.gemm(xs[-1], W, S, flags=flags))
        torch.cuda.synchronize()
        return [x.view(torch.int16).cpu().numpy().view(np.uint16) for x in xs]

    ref_bits = chain(0)
    for _ in range(3):
        got = chain(w8.FLAG_PDL)
        for a, b in zip(got, ref_bits):
            assert np.array_equal(a, b)
    for i, c in enumerate(cases[:3]):   # each link against the oracle on the GPU's own input
        c.A = torch.from_numpy(ref_bits[i].view(np.int16)).view(torch.bfloat16)
        ref, exact, absum = oracle_full(c)
        out = ref_bits[i + 1].reshape(M, K)
        compare(c, out, ref, exact, absum, split_k=4, label=f"gemv chain link {i}", variant=3)
