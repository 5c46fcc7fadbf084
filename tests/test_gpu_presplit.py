"""GPU parity of the pre-split W8A16 path (w8a16_gemm_ws): the two-term split
pre-pass into the caller's workspace, then the FP8 x FP8 kernel on both terms,
element by element against the CPU oracle of the W8A16 product (the two-term
error bound of tests/parity.py applies, as for the kernel that splits its own
tiles), over token tiles, splits, stage counts, ragged and strided shapes, the
workspace contents, NaN propagation and the fall-backs of the entry point."""
from __future__ import annotations

import numpy as np
import pytest
import torch

import workloads
from parity import compare, oracle_full

pytestmark = pytest.mark.gpu

PRESPLIT = 5


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


def _plan(M, N, K, token_tile, split_k, stages):
    """A pre-split plan with the given token tile (the planner's choice depends on M)."""
    from fp8_weight_only_gemm_gb300 import binding
    p = binding.plan_variant(token_tile, N, K, PRESPLIT, split_k, stages)
    assert (p.token_tile, p.split_k, p.stages) == (token_tile, split_k, stages)
    p.grid[1] = (M + token_tile - 1) // token_tile
    return p


def run_ws(case, plan=None, workspace=None, flags=0):
    """The case through w8a16_gemm_ws; C [M, ldc] as uint16 codes."""
    from fp8_weight_only_gemm_gb300 import binding
    wl = case.wl
    A, W, S, C = case.A.cuda(), case.W.cuda(), case.scale.cuda(), case.C0.cuda()
    binding.gemm_ws(A[:, :wl.K], W, S, C[:, :wl.N], workspace=workspace, plan=plan, flags=flags)
    torch.cuda.synchronize()
    return C.cpu().view(torch.int16).numpy().view(np.uint16)


@pytest.mark.parametrize("name", workloads.CONFIG_ORDER)
def test_workloads_through_the_workspace_entry(name):
    case = workloads.make_case(name)
    got = run_ws(case)
    ref, exact, absum = oracle_full(case)
    compare(case, got, ref, exact, absum, split_k=16, label=f"ws/{name}", variant=3)
    assert not np.any(got.reshape(case.wl.M, case.wl.ldc)[:, :case.wl.N] == workloads.C_USED_SENTINEL)


@pytest.mark.parametrize("M,N,K,lda,tile,split,stages", [
    (1, 256, 512, 512, 16, 2, 4), (16, 640, 2048, 2048, 16, 8, 4), (17, 300, 1280, 1344, 16, 3, 4),
    (32, 640, 2048, 2048, 32, 4, 4), (20, 384, 1536, 1536, 32, 1, 6), (33, 256, 1280, 1280, 32, 3, 4),
    (64, 384, 1024, 1032, 64, 2, 4), (50, 130, 1280, 1280, 64, 3, 6), (64, 256, 512, 512, 64, 1, 6),
    (128, 260, 512, 512, 128, 1, 4), (100, 384, 1024, 1024, 128, 1, 4), (130, 256, 768, 776, 128, 1, 4),
    (96, 256, 768, 768, 64, 3, 4), (16, 384, 2048, 2048, 16, 16, 4),
    # split 2 (the owner's straight-line sum) with a partial last token group and ragged N
    (29, 520, 1536, 1544, 32, 2, 4), (13, 300, 1024, 1024, 16, 2, 4), (61, 200, 1024, 1024, 64, 2, 4),
])
def test_forced_plans(M, N, K, lda, tile, split, stages):
    case = workloads.make_case("strided_m32_n14336_k5120", M=M, N=N, K=K, a_row_stride=lda,
                               c_row_stride=N + 3, seed=M * 31 + N + K, outlier_frac=0.01)
    p = _plan(M, N, K, tile, split, stages)
    got = run_ws(case, plan=p)
    ref, exact, absum = oracle_full(case)
    compare(case, got, ref, exact, absum, split_k=split, label=f"presplit M{M} tn{tile} s{split} st{stages}",
            variant=3)
    assert np.array_equal(got, run_ws(case, plan=p)), "same plan, different bits"


def _tail_plan(M, N, K, token_tile, stages, tail_tiles, tail_split, variant=PRESPLIT):
    """Whole tiles in a first launch, the last `tail_tiles` split over `tail_split` CTAs."""
    from fp8_weight_only_gemm_gb300 import binding
    p = binding.plan_variant(token_tile, N, K, variant, 1, stages)
    p.tail_tiles, p.tail_split = tail_tiles, tail_split
    p.grid[0] = (N + 127) // 128 - tail_tiles
    return p


@pytest.mark.parametrize("M,N,K,tile,stages,tail,tsplit", [
    (20, 640, 1024, 32, 4, 2, 3), (100, 1000, 1280, 128, 4, 3, 2), (64, 384, 2048, 64, 6, 1, 16),
    (9, 300, 512, 16, 4, 2, 4),
])
def test_split_k_tail(M, N, K, tile, stages, tail, tsplit):
    case = workloads.make_case("strided_m32_n14336_k5120", M=M, N=N, K=K, a_row_stride=K + 64,
                               c_row_stride=N + 5, seed=M + N + K + tail, outlier_frac=0.01)
    p = _tail_plan(M, N, K, tile, stages, tail, tsplit)
    got = run_ws(case, plan=p)
    ref, exact, absum = oracle_full(case)
    compare(case, got, ref, exact, absum, split_k=tsplit, label=f"tail M{M} N{N} tail{tail}x{tsplit}",
            variant=3)
    assert np.array_equal(got, run_ws(case, plan=p)), "same plan, different bits"


@pytest.mark.parametrize("tile,split,stages", [(32, 2, 4), (32, 4, 4), (64, 2, 4)])
def test_split_k_at_scale_repeated(tile, split, stages):
    """Many clusters at once (two CTAs per SM where the plan allows), five runs,
    each checked against the oracle and bit-identical to the first."""
    case = workloads.make_case("strided_m32_n14336_k5120", M=32 if tile == 32 else 64)
    wl = case.wl
    p = _plan(wl.M, wl.N, wl.K, tile, split, stages)
    ref, exact, absum = oracle_full(case)
    first = None
    for rep in range(5):
        got = run_ws(case, plan=p)
        if first is None:
            compare(case, got, ref, exact, absum, split_k=split, label=f"scale tn{tile} s{split}", variant=3)
            first = got
        else:
            assert np.array_equal(got, first), f"run {rep} differs from run 0"


def test_planner_uses_a_tail_when_tiles_overflow_one_wave():
    from fp8_weight_only_gemm_gb300 import binding
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    p = binding.plan_variant(128, 128 * (sms + sms // 2), 1024, PRESPLIT, 0, 0, sms)
    assert p.split_k == 1 and p.tail_tiles == sms // 2 and p.tail_split == 2 and p.grid[0] == sms
    case = workloads.make_case("tiny_m1_n256_k256", M=128, N=128 * (sms + sms // 2), K=1024, seed=88)
    got = run_ws(case, plan=p)
    ref, exact, absum = oracle_full(case)
    compare(case, got, ref, exact, absum, split_k=2, label="planned tail", variant=3)


@pytest.mark.parametrize("M,N,K", [(3, 256, 512), (40, 384, 1024)])
def test_every_code_and_scale_range(M, N, K):
    case = workloads.random_codes_case(M, N, K, seed=M + N + K + 5)
    got = run_ws(case, plan=_plan(M, N, K, 16 if M <= 16 else 64, 2, 4))
    ref, exact, absum = oracle_full(case)
    compare(case, got, ref, exact, absum, split_k=2, label="presplit all-codes", variant=3)


def test_activation_dynamic_range():
    case = workloads.make_case("tiny_m1_n256_k256", M=40, N=384, K=768, seed=81)
    g = torch.Generator().manual_seed(82)
    e = torch.randint(-40, 40, case.A.shape, generator=g).to(torch.float32)
    case.A = (case.A.float() * torch.pow(2.0, e)).to(torch.bfloat16)
    got = run_ws(case, plan=_plan(40, 384, 768, 64, 2, 4))
    ref, exact, absum = oracle_full(case)
    compare(case, got, ref, exact, absum, split_k=2, label="presplit range", variant=3)


def test_nan_activation_propagates():
    case = workloads.make_case("tiny_m1_n256_k256", M=24, N=256, K=384, seed=83)
    A = case.A.clone()
    A[5, 300] = float("nan")
    case.A = A
    got = run_ws(case, plan=_plan(24, 256, 384, 32, 1, 4))
    ref, exact, absum = oracle_full(case)
    compare(case, got, ref, exact, absum, split_k=1, label="presplit nan", variant=3)
    g = got.reshape(24, 256)
    isnan = ((g & 0x7F80) == 0x7F80) & ((g & 0x7F) != 0)
    assert isnan[5].all() and isnan.sum() == 256


def test_infinite_activation_gives_nan_row():
    """E4M3 has no infinity: an infinite activation makes its token's outputs NaN
    (where the exact sum would be +-Inf), as on the kernel that splits its own
    tiles; the other tokens are unaffected."""
    case = workloads.make_case("tiny_m1_n256_k256", M=24, N=256, K=384, seed=87)
    A = case.A.clone()
    A[9, 7] = float("inf")
    case_ok = workloads.make_case("tiny_m1_n256_k256", M=24, N=256, K=384, seed=87)
    case.A = A
    got = run_ws(case, plan=_plan(24, 256, 384, 32, 1, 4)).reshape(24, 256)
    isnan = ((got & 0x7F80) == 0x7F80) & ((got & 0x7F) != 0)
    assert isnan[9].all() and isnan.sum() == 256
    clean = run_ws(case_ok, plan=_plan(24, 256, 384, 32, 1, 4)).reshape(24, 256)
    rows = [m for m in range(24) if m != 9]
    assert np.array_equal(got[rows], clean[rows])


def test_workspace_holds_the_two_term_split():
    """Per token and 128-K group: factor = 2^(E-7) with E the exponent of the group's
    largest |a|, and factor * (hi + lo / 32) = a, exactly where |a| >= 2^-14 of that
    maximum and within 2^-22 of it below."""
    from fp8_weight_only_gemm_gb300 import binding
    M, N, K = 37, 256, 640
    case = workloads.make_case("tiny_m1_n256_k256", M=M, N=N, K=K, a_row_stride=648, seed=84)
    g = torch.Generator().manual_seed(85)
    e = torch.randint(-30, 30, (M, 648), generator=g).to(torch.float32)
    case.A = (case.A.float() * torch.pow(2.0, e)).to(torch.bfloat16)
    case.A[3, 128:256] = 0.0
    ws = torch.zeros(binding.workspace_bytes(M, K), dtype=torch.uint8, device="cuda")
    run_ws(case, plan=_plan(M, N, K, 64, 1, 4), workspace=ws)
    w = ws.cpu()
    codes = w[: 2 * M * K].view(2, M, K)
    S = (M + 3) // 4 * 4
    fac = w[2 * M * K:].view(torch.float32).view(K // 128, S)[:, :M].double()
    dec = lambda c: c.contiguous().view(torch.float8_e4m3fn).double()
    x = dec(codes[0]) + dec(codes[1]) / 32.0
    a = case.A[:, :K].double()
    amax = a.abs().view(M, K // 128, 128).amax(dim=2)
    expect_fac = torch.where(amax > 0, torch.pow(2.0, torch.floor(torch.log2(amax.clamp_min(1e-300))) - 7), 0.0)
    assert torch.equal(fac.T, expect_fac), "factors are not 2^(E-7)"
    rec = x * fac.T.repeat_interleave(128, dim=1)
    big = a.abs() >= amax.repeat_interleave(128, dim=1) * 2.0 ** -14
    assert torch.equal(rec[big], a[big]), "split not exact above 2^-14 of the group maximum"
    assert ((rec - a).abs() <= amax.repeat_interleave(128, dim=1) * 2.0 ** -22).all()


def test_entry_point_fallbacks():
    """No workspace, or one too small for the split: the call runs what w8a16_gemm
    runs (same bits), as does M <= 16 with a workspace too small for the stream-K
    layout; a pre-split plan without a workspace is refused."""
    import fp8_weight_only_gemm_gb300 as w8
    from fp8_weight_only_gemm_gb300 import binding
    for M in (8, 32):
        case = workloads.make_case("skinny_qkv_m8_n12288_k4096", M=M, N=512, K=1024, seed=86 + M)
        wl = case.wl
        A, W, S = case.A.cuda(), case.W.cuda(), case.scale.cuda()
        base = w8.gemm(A[:, :wl.K], W, S)
        for ws in (False, torch.empty(binding.workspace_bytes(M, wl.K) - 16, dtype=torch.uint8, device="cuda")):
            got = binding.gemm_ws(A[:, :wl.K], W, S, workspace=ws)
            assert torch.equal(got.view(torch.int16), base.view(torch.int16))
        if M == 8:
            ws = torch.empty(binding.workspace_bytes_for(M, wl.N, wl.K) - 1, dtype=torch.uint8, device="cuda")
            assert binding.plan_ws(M, wl.N, wl.K, ws.numel())["variant"] == w8.plan_current(M, wl.N, wl.K)["variant"]
            got = binding.gemm_ws(A[:, :wl.K], W, S, workspace=ws)
            assert torch.equal(got.view(torch.int16), base.view(torch.int16))
    p = _plan(32, 512, 1024, 32, 2, 4)
    with pytest.raises(binding.W8A16Error, match="workspace"):
        binding.gemm_ws(A[:, :1024], W, S, workspace=False, plan=p)


def test_programmatic_chain_through_the_workspace():
    """Dependent calls (each A the previous C) through one workspace with the
    programmatic-launch flag give the bits of the same chain without it."""
    from fp8_weight_only_gemm_gb300 import binding
    K = 1024
    cases = [workloads.make_case("strided_m32_n14336_k5120", M=32, N=K, K=K, seed=400 + i) for i in range(4)]
    Ws = [c.W.cuda() for c in cases]
    Ss = [c.scale.cuda() for c in cases]
    ws = torch.empty(binding.workspace_bytes(32, K), dtype=torch.uint8, device="cuda")
    x0 = cases[0].A.cuda()[:, :K]

    def chain(flags):
        x = x0
        for W, S in zip(Ws, Ss):
            x = binding.gemm_ws(x, W, S, workspace=ws, flags=flags)
        torch.cuda.synchronize()
        return x.view(torch.int16).cpu().numpy()

    ref_bits = chain(0)
    for _ in range(3):
        assert np.array_equal(chain(binding.FLAG_PDL), ref_bits)


def test_split_k_tail_with_shared_receive_buffer_repeated():
    """The 128-token two-term tile's split-K tail reuses the rings' shared memory for
    the partials (the end-of-loop cluster barrier orders it): at full size, five runs
    bit-identical, the first against the oracle."""
    from fp8_weight_only_gemm_gb300 import binding
    case = workloads.make_case("multitile_m128_n28672_k8192")
    wl = case.wl
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    p = binding.plan_variant(wl.M, wl.N, wl.K, PRESPLIT, 0, 0, sms)
    assert p.tail_tiles > 0 and p.tail_split >= 2
    first = None
    for rep in range(5):
        got = run_ws(case, plan=p)
        if first is None:
            ref, exact, absum = oracle_full(case)
            compare(case, got, ref, exact, absum, split_k=p.tail_split, label="tail alias", variant=3)
            first = got
        else:
            assert np.array_equal(got, first), f"run {rep} differs from run 0"


@pytest.mark.parametrize("M,N,K,lda", [(40, 300, 1280, 1344), (32, 14336, 5120, 5184), (5, 256, 512, 512),
                                       (129, 640, 1024, 1024)])
def test_split_then_terms_matches_the_one_call_path(M, N, K, lda):
    """w8a16_split_activations + w8a16_gemm_split_terms give the bits of
    w8a16_gemm_ws's pre-split path (same split, same kernel, same plan), and each
    of three weights multiplied from one split matches the oracle."""
    from fp8_weight_only_gemm_gb300 import binding
    cases = [workloads.make_case("strided_m32_n14336_k5120", M=M, N=N, K=K, a_row_stride=lda,
                                 c_row_stride=N + 5, seed=7 * M + N + s) for s in range(3)]
    A = cases[0].A.cuda()   # one activation matrix, three weights (the seeds differ only in W)
    ws = binding.split_activations(A[:, :K])
    for i, case in enumerate(cases):
        case = workloads.Case(case.wl, cases[0].A, case.W, case.scale, case.C0)
        W, S, C = case.W.cuda(), case.scale.cuda(), case.C0.cuda()
        binding.gemm_split_terms(ws, M, W, S, C[:, :N])
        torch.cuda.synchronize()
        got = C.cpu().view(torch.int16).numpy().view(np.uint16)
        ref, exact, absum = oracle_full(case)
        compare(case, got, ref, exact, absum, split_k=16, label=f"split+terms M{M} w{i}", variant=3)
        if M > 16:   # w8a16_gemm_ws with the split's workspace: the same pre-split plan
            ws1 = torch.empty(binding.workspace_bytes(M, K), dtype=torch.uint8, device="cuda")
            assert binding.plan_ws(M, N, K, ws1.numel())["variant"] == PRESPLIT
            assert np.array_equal(got, run_ws(case, workspace=ws1)), "two calls differ from w8a16_gemm_ws"


def test_split_terms_checks():
    from fp8_weight_only_gemm_gb300 import binding
    lib = binding.load()
    A = torch.zeros((4, 256), dtype=torch.bfloat16, device="cuda")
    small = torch.zeros(16, dtype=torch.uint8, device="cuda")
    assert lib.w8a16_split_activations(A.data_ptr(), 256, 4, 256, small.data_ptr(), small.numel(), None) == -13
    assert lib.w8a16_split_activations(A.data_ptr(), 256, 0, 256, small.data_ptr(), small.numel(), None) == -1
    assert lib.w8a16_split_activations(A.data_ptr(), 256, 4, 200, small.data_ptr(), small.numel(), None) == -2
    ws = binding.split_activations(A)
    W = torch.zeros((256, 256), dtype=torch.uint8, device="cuda")
    S = torch.zeros((2, 2), dtype=torch.float32, device="cuda")
    C = torch.zeros((4, 256), dtype=torch.bfloat16, device="cuda")
    assert lib.w8a16_gemm_split_terms(ws.data_ptr(), 15, W.data_ptr(), S.data_ptr(), C.data_ptr(), 256,
                                      4, 256, 256, 0, None) == -13
    assert lib.w8a16_gemm_split_terms(ws.data_ptr(), ws.numel(), W.data_ptr(), S.data_ptr(), C.data_ptr(), 255,
                                      4, 256, 256, 0, None) == -3
    assert lib.w8a16_gemm_split_terms(ws.data_ptr(), ws.numel(), W.data_ptr(), S.data_ptr(), C.data_ptr(), 256,
                                      4, 256, 256, 2, None) == -13
    binding.gemm_split_terms(ws, 4, W, S, C)
    torch.cuda.synchronize()
    assert float(C.float().abs().max()) == 0.0
