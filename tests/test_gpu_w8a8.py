"""GPU parity of the W8A8 variant: the per-token 128-group activation quantiser
bit for bit against the oracle (a code is an integer decision taken in FP32 on
both sides), and the FP8 x FP8 block-scaled GEMM element by element against the
oracle's W8A8 product, through the C ABI, over token tiles, forced K splits,
stage counts, ragged M and N, padded pitches and every finite E4M3 code; one and
two tokens also on the decode kernel (the codes copied in as its hi term)."""
from __future__ import annotations

import math

import numpy as np
import pytest
import torch

import workloads
from parity import bf16_to_f64, ulp_bf16

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


def _acts(M, K, lda, seed, zero_group=True, outliers=True):
    g = torch.Generator().manual_seed(seed)
    a = torch.randn(M, lda, generator=g)
    if outliers:
        idx = torch.randperm(M * lda, generator=g)[: max(1, M * lda // 100)]
        a.view(-1)[idx] *= 50.0
    if zero_group and K >= 256:
        a[M // 2, 128:256] = 0.0                                # one all-zero group
    return a.to(torch.bfloat16)


def _codes_u16(t):
    return t.contiguous().view(torch.int16).numpy().view(np.uint16)


def _device_w8a8_inputs(codes, scales, M, K, lda, scale_stride):
    """Activation codes at row pitch `lda` bytes and scales [K/128, scale_stride]
    on the GPU, pad bytes random so that reading them would show."""
    g = torch.Generator().manual_seed(M * 31 + K)
    Ad = torch.randint(0, 256, (M, lda), generator=g, dtype=torch.int32).to(torch.uint8)
    Ad[:, :K] = torch.from_numpy(codes)
    Sd = torch.full((K // 128, scale_stride), float("nan"), dtype=torch.float32)
    Sd[:, :M] = torch.from_numpy(scales)
    return Ad.cuda()[:, :K], Sd.cuda()


def _w8a8_check(o, Aq, a_scale, W, scale, M, N, K, got, C0, ldc, split_k, label):
    """GPU result vs the oracle's W8A8 product: pad columns bit for bit, the
    stated tolerance (dequantised activations standing for A), and the FP32
    arithmetic bound of a step-wise FP32 accumulation."""
    ref, exact, absum = o.w8a8_gemm(Aq, a_scale, W, scale, M, N, K, C=C0, c_row_stride=ldc,
                                    want_exact=True)
    got = got.reshape(M, ldc)
    assert np.array_equal(got[:, N:], ref[:, N:]), f"{label}: pad columns of C were written"
    g = bf16_to_f64(got[:, :N])
    r = bf16_to_f64(ref[:, :N])
    assert np.array_equal(np.isnan(g), np.isnan(r)), f"{label}: NaN pattern differs"
    fin = ~np.isnan(r)
    e4 = lambda c: torch.from_numpy(np.ascontiguousarray(c)).view(torch.float8_e4m3fn).to(torch.float64)
    adq = e4(Aq).reshape(M, K) * torch.from_numpy(a_scale).to(torch.float64).T.repeat_interleave(128, 1)
    wdq = (e4(W).reshape(N, K) *
           torch.from_numpy(scale).to(torch.float64).repeat_interleave(128, 0)[:N].repeat_interleave(128, 1))
    amax = float(adq.abs().nan_to_num(0.0).max())
    wmax = float(wdq.abs().nan_to_num(0.0).max())
    tol = 2.0 ** -7 * np.abs(r) + 1e-3 * math.sqrt(K) * amax * wmax
    err = np.abs(g - r)
    bad = fin & ~(err <= tol)
    assert not bad.any(), (f"{label}: {bad.sum()} outputs outside the stated tolerance; first at "
                           f"{np.argwhere(bad)[0]}: gpu={g[bad][0]} ref={r[bad][0]}")
    gamma = (K / 128 + 256 + split_k) * 2.0 ** -23
    tight = gamma * absum + 0.5 * ulp_bf16(np.abs(exact) + gamma * absum) + 2.0 ** -133
    err2 = np.abs(g - exact)
    bad2 = fin & ~(err2 <= tight)
    assert not bad2.any(), (f"{label}: {bad2.sum()} outputs outside the arithmetic bound; first at "
                            f"{np.argwhere(bad2)[0]}: gpu={g[bad2][0]} exact={exact[bad2][0]} "
                            f"bound={tight[bad2][0]}")


def _forced_plan(M, N, K, token_tile, split_k, stages):
    """A W8A8 plan with the given token tile (the library's own choice depends on M)."""
    from fp8_weight_only_gemm_gb300 import binding
    p = binding.plan_variant(token_tile, N, K, binding.VARIANT_W8A8, split_k, stages)
    assert p.token_tile == token_tile and p.split_k == split_k and p.stages == stages
    p.grid[1] = (M + token_tile - 1) // token_tile
    return p


# ------------------------------------------------------ activation quantiser --

@pytest.mark.parametrize("M,K,lda", [
    (1, 128, 128), (5, 4096, 4104), (33, 384, 392), (130, 1024, 1024), (16, 5120, 5184),
])
def test_act_quantizer_matches_oracle(o, M, K, lda):
    from fp8_weight_only_gemm_gb300 import binding
    a = _acts(M, K, lda, seed=M * 13 + K)
    codes, scales = binding.quantize_activations(a.cuda()[:, :K])
    torch.cuda.synchronize()
    rc, rs = o.quantize_activations(_codes_u16(a), M, K, a_row_stride=lda)
    got_s = scales.cpu().numpy()
    assert np.array_equal(got_s[:, :M].view(np.uint32), rs.view(np.uint32)), "scales differ"
    assert not got_s[:, M:].any(), "scale pad columns were written"
    bad = np.argwhere(codes.cpu().numpy() != rc)
    assert bad.size == 0, f"{len(bad)} codes differ, first at {bad[:3].tolist()}"


def test_act_quantizer_nan_and_tiny(o):
    """A NaN does not enter its group's maximum and encodes as NaN; a group of
    subnormal BF16 values still gets a nonzero scale."""
    from fp8_weight_only_gemm_gb300 import binding
    a = _acts(4, 256, 256, seed=9, zero_group=False, outliers=False)
    a[1, 7] = float("nan")
    a[2, 128:] = torch.linspace(-1e-38, 1e-38, 128).to(torch.bfloat16)
    codes, scales = binding.quantize_activations(a.cuda())
    rc, rs = o.quantize_activations(_codes_u16(a), 4, 256)
    assert np.array_equal(scales.cpu().numpy()[:, :4].view(np.uint32), rs.view(np.uint32))
    assert np.array_equal(codes.cpu().numpy(), rc)
    assert codes[1, 7].item() & 0x7F == 0x7F and np.isfinite(rs).all() and rs[1, 2] > 0


# -------------------------------------------------------------- W8A8 GEMM --

# (M, N, K, lda pad bytes, ldc pad, plan: None = the library's, else (token_tile, split_k, stages))
W8A8_CASES = [
    (1, 4096, 4096, 0, 0, None),
    (5, 300, 384, 16, 10, None),
    (16, 1000, 1024, 0, 0, (16, 8, 6)),
    (17, 256, 2048, 32, 0, (16, 16, 4)),
    (32, 640, 2048, 0, 3, (32, 4, 4)),
    (32, 640, 1280, 0, 0, (32, 3, 6)),
    (64, 384, 1024, 16, 0, (64, 2, 6)),
    (64, 130, 1280, 0, 0, (64, 3, 4)),
    (100, 260, 512, 0, 0, (128, 1, 4)),
    (130, 260, 512, 0, 2, (128, 2, 4)),
    (200, 256, 1280, 0, 0, None),
    # split 2 (the owner's straight-line sum) with a partial last token group and ragged N
    (29, 520, 1536, 0, 5, (32, 2, 4)),
    (13, 300, 1024, 16, 0, (16, 2, 4)),
    (125, 390, 1024, 0, 0, (128, 2, 4)),
]


@pytest.mark.parametrize("M,N,K,apad,cpad,plan", W8A8_CASES)
def test_w8a8_matches_oracle(o, M, N, K, apad, cpad, plan):
    from fp8_weight_only_gemm_gb300 import binding
    case = workloads.make_case(workloads.Workload(
        f"w8a8_m{M}_n{N}_k{K}", M, N, K, seed=M * 7 + N + K, c_row_stride=(N + cpad) if cpad else None,
        outlier_frac=0.01, zero_blocks=((0, 1),) if K >= 256 else ()))
    Aq, a_scale = o.quantize_activations(case.A_np(), M, K)
    lda, ldc = K + apad, case.wl.ldc
    Ad, Sd = _device_w8a8_inputs(Aq, a_scale, M, K, lda, (M + 3) // 4 * 4 + 4)
    C = case.C0.cuda()
    p = None if plan is None else _forced_plan(M, N, K, *plan)
    binding.gemm_w8a8(Ad, Sd, case.W.cuda(), case.scale.cuda(), C[:, :N], plan=p)
    torch.cuda.synchronize()
    got = C.cpu().view(torch.int16).numpy().view(np.uint16)
    split = p.split_k if p is not None else 16
    _w8a8_check(o, Aq, a_scale, case.W_np(), case.scale_np(), M, N, K, got, case.C0_np(), ldc, split,
                f"w8a8 M={M} N={N} K={K} plan={plan}")
    assert binding.device_status() == (0, 0, 0)


@pytest.mark.parametrize("tile,split,stages", [(32, 2, 4), (32, 4, 4), (64, 2, 4), (16, 8, 4)])
def test_w8a8_split_k_at_scale_repeated(o, tile, split, stages):
    """Split-K over many clusters, two CTAs per SM where the plan allows, five runs:
    the owners' sums of the other ranks' pushed partials must see every push (a
    receive wait without cluster-scope acquire read stale partials now and then)."""
    from fp8_weight_only_gemm_gb300 import binding
    M, N, K = tile if tile < 64 else 64, 14336, 5120
    case = workloads.make_case(workloads.Workload(f"w8a8scale_{tile}", M, N, K, seed=tile + split))
    Aq, a_scale = o.quantize_activations(case.A_np(), M, K)
    Ad, Sd = _device_w8a8_inputs(Aq, a_scale, M, K, K, (M + 3) // 4 * 4)
    p = _forced_plan(M, N, K, tile, split, stages)
    Wd, Sw = case.W.cuda(), case.scale.cuda()
    first = None
    for rep in range(5):
        C = case.C0.cuda()
        binding.gemm_w8a8(Ad, Sd, Wd, Sw, C[:, :N], plan=p)
        torch.cuda.synchronize()
        got = C.cpu().view(torch.int16).numpy().view(np.uint16)
        if first is None:
            _w8a8_check(o, Aq, a_scale, case.W_np(), case.scale_np(), M, N, K, got, case.C0_np(), N, split,
                        f"w8a8 scale tn{tile} s{split}")
            first = got
        else:
            assert np.array_equal(got, first), f"run {rep} differs from run 0 (tn{tile} s{split})"
    assert binding.device_status() == (0, 0, 0)


@pytest.mark.parametrize("M,N,K,tile,tail,tsplit", [(30, 640, 1024, 32, 2, 4), (128, 900, 1536, 128, 3, 2)])
def test_w8a8_split_k_tail(o, M, N, K, tile, tail, tsplit):
    """Whole weight tiles in a first launch, the last ones split over clusters in a second."""
    from fp8_weight_only_gemm_gb300 import binding
    case = workloads.make_case(workloads.Workload(f"w8a8tail_m{M}", M, N, K, seed=M + N + tail,
                                                  outlier_frac=0.01))
    Aq, a_scale = o.quantize_activations(case.A_np(), M, K)
    Ad, Sd = _device_w8a8_inputs(Aq, a_scale, M, K, K, (M + 3) // 4 * 4)
    p = binding.plan_variant(tile, N, K, binding.VARIANT_W8A8, 1, 4)
    p.grid[1] = (M + tile - 1) // tile
    p.tail_tiles, p.tail_split = tail, tsplit
    p.grid[0] = (N + 127) // 128 - tail
    C = case.C0.cuda()
    binding.gemm_w8a8(Ad, Sd, case.W.cuda(), case.scale.cuda(), C[:, :N], plan=p)
    torch.cuda.synchronize()
    got = C.cpu().view(torch.int16).numpy().view(np.uint16)
    _w8a8_check(o, Aq, a_scale, case.W_np(), case.scale_np(), M, N, K, got, case.C0_np(), N, tsplit,
                f"w8a8 tail M={M} N={N}")
    assert binding.device_status() == (0, 0, 0)


def test_w8a8_every_code(o):
    """Every finite E4M3 code on both sides (subnormals, -0, +-448) with group and
    block scales spread over 2^-8..2^8."""
    from fp8_weight_only_gemm_gb300 import binding
    M, N, K = 20, 256, 512
    g = torch.Generator().manual_seed(1234)
    rnd = lambda *s: torch.randint(0, 256, s, generator=g, dtype=torch.int32).to(torch.uint8)
    Aq, W = rnd(M, K), rnd(N, K)
    for t in (Aq, W):
        t[(t == 0x7F) | (t == 0xFF)] = 0x7E
    a_scale = torch.pow(2.0, torch.rand((K // 128, M), generator=g) * 16 - 8).float()
    scale = torch.pow(2.0, torch.rand((N // 128, K // 128), generator=g) * 16 - 8).float()
    Ad, Sd = _device_w8a8_inputs(Aq.numpy(), a_scale.numpy(), M, K, K, 24)
    C0 = torch.full((M, N), workloads.C_USED_SENTINEL, dtype=torch.int32).to(torch.int16)
    C = C0.view(torch.bfloat16).cuda()
    for tile, split in ((32, 1), (16, 4)):
        p = _forced_plan(M, N, K, tile, split, 4)
        C.copy_(C0.view(torch.bfloat16))
        binding.gemm_w8a8(Ad, Sd, W.cuda(), scale.cuda(), C, plan=p)
        torch.cuda.synchronize()
        got = C.cpu().view(torch.int16).numpy().view(np.uint16)
        _w8a8_check(o, Aq.numpy(), a_scale.numpy(), W.numpy(), scale.numpy(), M, N, K, got,
                    C0.numpy().view(np.uint16), N, p.split_k, f"every code split={split}")


def test_w8a8_end_to_end_with_gpu_quantiser(o):
    """BF16 activations quantised on the GPU, then the W8A8 GEMM, twice in a row
    with programmatic dependent launch: the oracle's quantiser and product give
    the same result."""
    from fp8_weight_only_gemm_gb300 import binding
    case = workloads.make_case("skinny_qkv_m8_n12288_k4096")
    wl = case.wl
    Ad = case.A.cuda()
    Wd, Sd = case.W.cuda(), case.scale.cuda()
    codes, scales = binding.quantize_activations(Ad[:, :wl.K])
    C = case.C0.cuda()
    for _ in range(2):
        binding.gemm_w8a8(codes, scales, Wd, Sd, C[:, :wl.N], flags=binding.FLAG_PDL)
    torch.cuda.synchronize()
    Aq, a_scale = o.quantize_activations(case.A_np(), wl.M, wl.K, a_row_stride=wl.lda)
    assert np.array_equal(codes.cpu().numpy(), Aq)
    got = C.cpu().view(torch.int16).numpy().view(np.uint16)
    _w8a8_check(o, Aq, a_scale, case.W_np(), case.scale_np(), wl.M, wl.N, wl.K, got, case.C0_np(),
                wl.ldc, 16, "end to end")
    assert binding.device_status() == (0, 0, 0)


def test_w8a8_rejects_foreign_plan():
    from fp8_weight_only_gemm_gb300 import binding
    p = binding.plan_variant(8, 256, 256, binding.VARIANT_TC, 1, 0)
    Ad = torch.zeros((8, 256), dtype=torch.uint8, device="cuda")
    Sd = torch.zeros((2, 8), dtype=torch.float32, device="cuda")
    W = torch.zeros((256, 256), dtype=torch.uint8, device="cuda")
    s = torch.zeros((2, 2), dtype=torch.float32, device="cuda")
    with pytest.raises(binding.W8A16Error, match="neither a W8A8 nor a decode plan"):
        binding.gemm_w8a8(Ad, Sd, W, s, plan=p)


def _sms():
    return torch.cuda.get_device_properties(0).multi_processor_count


@pytest.mark.parametrize("M", [1, 2])
@pytest.mark.parametrize("N,K,split", [(4096, 4096, 4), (300, 1024, 1), (300, 1280, 2), (130, 640, 5),
                                       (256, 2048, 8), (1000, 128, 1)])
def test_w8a8_decode_kernel(o, M, N, K, split):
    """One or two tokens on the decode kernel: forced splits 1..8 (up to 8 K steps a
    CTA, some read from TMEM), ragged N, padded pitches; run to run bit-identical."""
    from fp8_weight_only_gemm_gb300 import binding
    case = workloads.make_case(workloads.Workload(f"w8a8dec_m{M}_n{N}_k{K}", M, N, K, seed=M * 13 + N + K + split,
                                                  c_row_stride=N + 3, outlier_frac=0.01,
                                                  zero_blocks=((0, 1),) if K >= 256 else ()))
    Aq, a_scale = o.quantize_activations(case.A_np(), M, K)
    Ad, Sd = _device_w8a8_inputs(Aq, a_scale, M, K, K + 32, 8)
    p = binding.plan_variant(M, N, K, binding.VARIANT_GEMV, split, 0, _sms())
    assert p.variant == binding.VARIANT_GEMV and p.split_k == split
    Wd, Sw = case.W.cuda(), case.scale.cuda()
    outs = []
    for _ in range(2):
        C = case.C0.cuda()
        binding.gemm_w8a8(Ad, Sd, Wd, Sw, C[:, :N], plan=p)
        torch.cuda.synchronize()
        outs.append(C.cpu().view(torch.int16).numpy().view(np.uint16))
    _w8a8_check(o, Aq, a_scale, case.W_np(), case.scale_np(), M, N, K, outs[0], case.C0_np(), N + 3, split,
                f"w8a8 decode M={M} N={N} K={K} split={split}")
    assert np.array_equal(outs[0], outs[1]), "same plan, different bits"
    assert binding.device_status() == (0, 0, 0)


def test_w8a8_decode_nan_codes(o):
    """A NaN weight code makes its row NaN for both tokens, a NaN activation code its
    token's outputs NaN, on the decode kernel as in the oracle."""
    from fp8_weight_only_gemm_gb300 import binding
    M, N, K = 2, 256, 1024
    case = workloads.make_case(workloads.Workload("w8a8dec_nan", M, N, K, seed=77))
    Aq, a_scale = o.quantize_activations(case.A_np(), M, K)
    Aq = Aq.copy()
    Aq[1, 700] = 0x7F
    W = case.W.clone()
    W[5, 300] = 0xFF
    Ad, Sd = _device_w8a8_inputs(Aq, a_scale, M, K, K, 4)
    p = binding.plan_variant(M, N, K, binding.VARIANT_GEMV, 2, 0, _sms())
    C = case.C0.cuda()
    binding.gemm_w8a8(Ad, Sd, W.cuda(), case.scale.cuda(), C[:, :N], plan=p)
    torch.cuda.synchronize()
    got = C.cpu().view(torch.int16).numpy().view(np.uint16)
    g = got.reshape(M, N)
    isnan = ((g & 0x7F80) == 0x7F80) & ((g & 0x7F) != 0)
    assert isnan[0, 5] and isnan[0].sum() == 1 and isnan[1].all()
    _w8a8_check(o, Aq, a_scale, W.numpy(), case.scale_np(), M, N, K, got, case.C0_np(), N, 2, "w8a8 decode NaN")


def test_w8a8_decode_chain_with_gpu_quantiser(o):
    """Quantiser then decode GEMM, five times in a row with programmatic dependent
    launch (each quantiser waits for the previous GEMM): the bits of the same calls
    without it, and the oracle's result."""
    from fp8_weight_only_gemm_gb300 import binding
    case = workloads.make_case("decode_gemv_m1_n4096_k4096")
    wl = case.wl
    Ad = case.A.cuda()
    Wd, Sd = case.W.cuda(), case.scale.cuda()

    def run(flags):
        C = case.C0.cuda()
        for _ in range(5):
            codes, scales = binding.quantize_activations(Ad[:, :wl.K])
            binding.gemm_w8a8(codes, scales, Wd, Sd, C[:, :wl.N], flags=flags)
        torch.cuda.synchronize()
        return C.cpu().view(torch.int16).numpy().view(np.uint16)

    base = run(0)
    assert np.array_equal(run(binding.FLAG_PDL), base)
    Aq, a_scale = o.quantize_activations(case.A_np(), wl.M, wl.K, a_row_stride=wl.lda)
    _w8a8_check(o, Aq, a_scale, case.W_np(), case.scale_np(), wl.M, wl.N, wl.K, base, case.C0_np(), wl.ldc, 4,
                "w8a8 decode chain")
    assert binding.device_status() == (0, 0, 0)
