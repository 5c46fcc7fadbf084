"""GPU parity: the CUDA path through the C ABI against the CPU oracle, element by
element, on seeded synthetic inputs (full outputs for every workload; the
tolerances are described in tests/parity.py)."""
from __future__ import annotations

import numpy as np
import pytest
import torch

import workloads
from parity import compare, oracle_full, run_gpu

pytestmark = pytest.mark.gpu


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


def _plan(M, N, K, variant, split_k=0, stages=0):
    from fp8_weight_only_gemm_gb300 import binding
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    return binding.plan_variant(M, N, K, variant, split_k, stages, sms)


TC_VARIANTS = [2, 3]   # BF16 datapath, FP8 datapath


@pytest.mark.parametrize("name", workloads.CONFIG_ORDER)
def test_workload_auto_plan(name):
    case = workloads.make_case(name)
    got = run_gpu(case)
    ref, exact, absum = oracle_full(case)
    from fp8_weight_only_gemm_gb300 import binding
    wl = case.wl
    p = binding.plan_current(wl.M, wl.N, wl.K)
    compare(case, got, ref, exact, absum, split_k=p["split_k"], label=name, variant=p["variant"])
    # every output of the used region was written (no sentinel left)
    assert not np.any(got.reshape(wl.M, wl.ldc)[:, :wl.N] == workloads.C_USED_SENTINEL)


@pytest.mark.parametrize("variant", TC_VARIANTS)
@pytest.mark.parametrize("name", workloads.CONFIG_ORDER[:4])
def test_workload_each_tc_variant(name, variant):
    case = workloads.make_case(name)
    wl = case.wl
    got = run_gpu(case, plan=_plan(wl.M, wl.N, wl.K, variant))
    ref, exact, absum = oracle_full(case)
    compare(case, got, ref, exact, absum, split_k=16, label=f"{name}/v{variant}", variant=variant)


@pytest.mark.parametrize("name", workloads.CONFIG_ORDER[:4])
def test_workload_simt_variant(name):
    from fp8_weight_only_gemm_gb300 import binding
    case = workloads.make_case(name)
    wl = case.wl
    got = run_gpu(case, plan=_plan(wl.M, wl.N, wl.K, binding.VARIANT_SIMT))
    ref, exact, absum = oracle_full(case)
    compare(case, got, ref, exact, absum, label=name + "/simt")


@pytest.mark.parametrize("variant", TC_VARIANTS)
@pytest.mark.parametrize("split_k", [1, 2, 3, 5, 8, 13, 16])
@pytest.mark.parametrize("M", [1, 8, 32])
def test_forced_splits(split_k, M, variant):
    case = workloads.make_case("decode_gemv_m1_n4096_k4096", M=M, N=640, K=2048, seed=100 + M)
    wl = case.wl
    p = _plan(wl.M, wl.N, wl.K, variant, split_k=split_k)
    got = run_gpu(case, plan=p)
    ref, exact, absum = oracle_full(case)
    compare(case, got, ref, exact, absum, split_k=split_k, label=f"split{split_k}/M{M}/v{variant}",
            variant=variant)
    again = run_gpu(case, plan=p)
    assert np.array_equal(got, again), "same plan, different bits: not deterministic"


@pytest.mark.parametrize("variant,M,stages,split", [
    (2, 4, 4, 2), (2, 4, 6, 2), (2, 4, 8, 2), (2, 4, 10, 3), (2, 24, 3, 2), (2, 24, 4, 2),
    (2, 24, 6, 2), (2, 24, 8, 3), (2, 48, 4, 2), (2, 48, 6, 2), (2, 48, 8, 3), (2, 100, 4, 2),
    (2, 100, 6, 1), (2, 100, 4, 3),
    (3, 4, 4, 2), (3, 4, 6, 2), (3, 4, 8, 3), (3, 24, 4, 2), (3, 24, 6, 2), (3, 24, 8, 3),
    (3, 48, 4, 2), (3, 48, 6, 3)])
def test_stage_instances(variant, M, stages, split):
    case = workloads.make_case("decode_gemv_m1_n4096_k4096", M=M, N=384, K=1536, seed=200 + M)
    wl = case.wl
    p = _plan(wl.M, wl.N, wl.K, variant, split_k=split, stages=stages)
    got = run_gpu(case, plan=p)
    ref, exact, absum = oracle_full(case)
    compare(case, got, ref, exact, absum, split_k=split, label=f"v{variant}/stages{stages}/M{M}",
            variant=variant)


@pytest.mark.parametrize("M,N,K,lda,ldc", [
    (1, 1, 128, 128, 1), (2, 7, 128, 136, 9), (15, 129, 256, 256, 130), (16, 128, 384, 392, 128),
    (17, 255, 256, 264, 300), (31, 300, 640, 640, 301), (33, 200, 512, 520, 200),
    (64, 130, 256, 256, 131), (65, 257, 384, 384, 257), (127, 64, 256, 264, 64),
    (129, 300, 256, 256, 300), (200, 129, 128, 136, 133), (257, 128, 256, 256, 128),
])
@pytest.mark.parametrize("variant", [0, 2, 3])
def test_edge_shapes(M, N, K, lda, ldc, variant):
    case = workloads.make_case("tiny_m1_n256_k256", M=M, N=N, K=K, a_row_stride=lda,
                               c_row_stride=ldc, seed=M * 1000 + N)
    plan = None if variant == 0 else _plan(M, N, K, variant)
    got = run_gpu(case, plan=plan)
    ref, exact, absum = oracle_full(case)
    v = variant or __import__("fp8_weight_only_gemm_gb300").plan_current(M, N, K)["variant"]
    compare(case, got, ref, exact, absum, split_k=16, label=f"edge M{M} N{N} K{K} v{variant}",
            variant=v)


@pytest.mark.parametrize("variant", TC_VARIANTS)
@pytest.mark.parametrize("M,N,K", [(3, 256, 512), (20, 384, 1024)])
def test_every_code_and_scale_range(M, N, K, variant):
    """Uniform codes (subnormals, +-448, -0 included) under log-uniform scales."""
    case = workloads.random_codes_case(M, N, K, seed=M + N + K)
    got = run_gpu(case, plan=_plan(M, N, K, variant))
    ref, exact, absum = oracle_full(case)
    compare(case, got, ref, exact, absum, split_k=16, label=f"all-codes/v{variant}", variant=variant)


@pytest.mark.parametrize("variant", TC_VARIANTS)
def test_nan_weight_code_propagates(variant):
    case = workloads.make_case("tiny_m1_n256_k256", M=5, N=256, K=384, seed=77)
    case.W[3, 200] = 0x7F
    case.W[130, 5] = 0xFF
    got = run_gpu(case, plan=_plan(5, 256, 384, variant))
    ref, exact, absum = oracle_full(case)
    compare(case, got, ref, exact, absum, split_k=16, label=f"nan/v{variant}", variant=variant)
    g = got.reshape(5, 256)
    isnan = ((g & 0x7F80) == 0x7F80) & ((g & 0x7F) != 0)
    assert isnan[:, 3].all() and isnan[:, 130].all() and isnan.sum() == 10


@pytest.mark.parametrize("variant", TC_VARIANTS)
def test_nan_activation_propagates(variant):
    case = workloads.make_case("tiny_m1_n256_k256", M=6, N=256, K=384, seed=78)
    A = case.A.clone()
    A[2, 300] = float("nan")
    case.A = A
    got = run_gpu(case, plan=_plan(6, 256, 384, variant))
    ref, exact, absum = oracle_full(case)
    compare(case, got, ref, exact, absum, split_k=16, label=f"nan-a/v{variant}", variant=variant)
    g = got.reshape(6, 256)
    isnan = ((g & 0x7F80) == 0x7F80) & ((g & 0x7F) != 0)
    assert isnan[2].all() and isnan.sum() == 256


@pytest.mark.parametrize("variant", TC_VARIANTS)
def test_activation_dynamic_range(variant):
    """Activations spread over 2^+-40 within each 128-K block (tiny values next to
    large ones): exact on the BF16 datapath, within the two-term bound on TC8."""
    case = workloads.make_case("tiny_m1_n256_k256", M=7, N=384, K=768, seed=79)
    g = torch.Generator().manual_seed(80)
    e = torch.randint(-40, 40, case.A.shape, generator=g).to(torch.float32)
    case.A = (case.A.float() * torch.pow(2.0, e)).to(torch.bfloat16)
    got = run_gpu(case, plan=_plan(7, 384, 768, variant))
    ref, exact, absum = oracle_full(case)
    compare(case, got, ref, exact, absum, split_k=16, label=f"range/v{variant}", variant=variant)


@pytest.mark.parametrize("variant", TC_VARIANTS)
def test_zero_block_and_zero_scale(variant):
    case = workloads.make_case("skinny_qkv_m8_n12288_k4096", N=512, K=1024, zero_blocks=((2, 3),))
    assert float(case.scale[2, 3]) == 0.0
    got = run_gpu(case, plan=_plan(8, 512, 1024, variant))
    ref, exact, absum = oracle_full(case)
    compare(case, got, ref, exact, absum, split_k=16, label=f"zero-block/v{variant}", variant=variant)


def test_host_buffer_entry_point_matches_device_path():
    import fp8_weight_only_gemm_gb300 as w8
    case = workloads.make_case("strided_m32_n14336_k5120", N=1024, K=1024, a_row_stride=1088,
                               c_row_stride=1100)
    wl = case.wl
    dev = run_gpu(case)
    A_h = case.A.pin_memory()
    W_h = case.W.pin_memory()
    S_h = case.scale.pin_memory()
    C_h = case.C0.clone().pin_memory()
    dA = torch.empty_like(case.A, device="cuda")
    dW = torch.empty_like(case.W, device="cuda")
    dS = torch.empty_like(case.scale, device="cuda")
    dC = torch.empty_like(case.C0, device="cuda")
    w8.gemm_host(A_h[:, :wl.K], W_h, S_h, C_h[:, :wl.N], dA, dW, dS, dC)
    torch.cuda.synchronize()
    host = C_h.view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(host, dev.reshape(host.shape))


def test_determinism_across_calls():
    case = workloads.make_case("skinny_qkv_m8_n12288_k4096")
    a = run_gpu(case)
    b = run_gpu(case)
    assert np.array_equal(a, b)


def test_bounded_wait_times_out_and_context_survives():
    from fp8_weight_only_gemm_gb300 import binding
    binding.device_status(clear=True)
    binding.selftest_wait_timeout(2000)      # 2 ms: nothing ever arrives
    st, where, detail = binding.device_status(clear=True)
    assert st == binding.STATUS_WAIT_TIMEOUT and detail == 0xFF
    # the context is still usable: a normal call afterwards is correct
    case = workloads.make_case("tiny_m1_n256_k256")
    got = run_gpu(case)
    ref, exact, absum = oracle_full(case)
    compare(case, got, ref, exact, absum, label="after-timeout")
    assert binding.device_status()[0] == 0


def test_programmatic_launch_chain_is_ordered():
    """Four dependent calls (each call's A is the previous call's C, N = K) queued
    with the programmatic-launch flag give the same bits as without it, and the
    first link matches the oracle."""
    import fp8_weight_only_gemm_gb300 as w8
    K = 1024
    cases = [workloads.make_case("decode_gemv_m1_n4096_k4096", M=8, N=K, K=K, seed=300 + i)
             for i in range(4)]
    Ws = [c.W.cuda() for c in cases]
    Ss = [c.scale.cuda() for c in cases]
    x0 = cases[0].A.cuda()

    def chain(flags):
        x = x0
        for W, S in zip(Ws, Ss):
            x = w8.gemm(x, W, S, flags=flags)
        torch.cuda.synchronize()
        return x.view(torch.int16).cpu().numpy()

    ref_bits = chain(0)
    for _ in range(3):
        assert np.array_equal(chain(w8.FLAG_PDL), ref_bits)
    first = run_gpu(cases[0])
    ref, exact, absum = oracle_full(cases[0])
    compare(cases[0], first, ref, exact, absum, split_k=16, label="pdl-chain-first")


def test_live_plan_and_capacity():
    import fp8_weight_only_gemm_gb300 as w8
    cap = w8.cluster_capacity(16, 4)
    assert cap[0] == 0 and cap[1] >= torch.cuda.get_device_properties(0).multi_processor_count
    p = w8.plan_current(1, 4096, 4096)
    cap = w8.cluster_capacity(p["token_tile"], p["stages"], p["variant"])
    # the chosen cluster size can run, and the plan fits the SMs' CTA slots (the
    # occupancy query counts one CTA per SM; two of this plan's CTAs share one)
    assert cap[p["split_k"]] > 0, (p, cap)
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    assert p["grid"][0] * p["grid"][1] <= sms * p["ctas_per_sm"], p


@pytest.mark.parametrize("M,N,K,stages,tail,tsplit", [
    (100, 1000, 1280, 4, 3, 2), (40, 640, 2048, 4, 2, 4), (20, 900, 1024, 4, 4, 3)])
def test_bf16_kernel_split_k_tail(M, N, K, stages, tail, tsplit):
    """BF16 kernel: whole weight tiles in a first launch, the last ones split over
    clusters in a second (programmatic dependent) launch; twice, bit for bit."""
    from fp8_weight_only_gemm_gb300 import binding
    case = workloads.make_case("strided_m32_n14336_k5120", M=M, N=N, K=K, a_row_stride=K + 64,
                               c_row_stride=N + 3, seed=M + N + tail)
    p = _plan(M, N, K, binding.VARIANT_TC, split_k=1, stages=stages)
    p.tail_tiles, p.tail_split = tail, tsplit
    p.grid[0] = -(-N // 128) - tail
    got = run_gpu(case, plan=p)
    ref, exact, absum = oracle_full(case)
    compare(case, got, ref, exact, absum, split_k=tsplit, label=f"bf16 tail M{M} {tail}x{tsplit}")
    assert np.array_equal(got, run_gpu(case, plan=p))
