"""Host-side tests of the C-ABI library (no GPU, no compute calls): it builds,
loads, exports every function include/w8a16.h declares, applies the page's checks
in the page's order with their own codes and messages, and plans launches."""
from __future__ import annotations

import ctypes
import re

import pytest

from fp8_weight_only_gemm_gb300 import binding
from fp8_weight_only_gemm_gb300.build import build_library


@pytest.fixture(scope="module")
def lib():
    build_library()
    return binding.load()


def test_exports_every_declared_function(lib):
    names = binding.header_functions()
    assert len(names) >= 12
    for n in names:
        assert hasattr(lib, n), f"{n} declared in include/w8a16.h but not exported"
    assert set(names) == set(binding._SIGS), "binding signatures out of sync with the header"


def test_header_constants_match_binding():
    text = binding.HEADER.read_text()
    def val(name):
        return int(re.search(rf"{name}\s*=\s*(-?\d+)", text).group(1))
    assert val("W8A16_VARIANT_SIMT") == binding.VARIANT_SIMT
    assert val("W8A16_VARIANT_TC") == binding.VARIANT_TC
    assert val("W8A16_VARIANT_TC8") == binding.VARIANT_TC8
    assert val("W8A16_STATUS_WAIT_TIMEOUT") == binding.STATUS_WAIT_TIMEOUT
    assert int(re.search(r"W8A16_FLAG_PDL\s*=\s*(\d+)u", text).group(1)) == binding.FLAG_PDL


ERR = dict(M_ZERO=-1, K_BLOCK=-2, PITCH=-3, A_PITCH_ALIGN=-4, N_ZERO=-5, NULL=-6, ALIGN=-7,
           RANGE=-8, DEVICE=-9, PLAN=-11)


@pytest.mark.parametrize("args,code,needle", [
    # (M, N, K, lda, ldc)
    ((0, 128, 128, 128, 128), ERR["M_ZERO"], "m=0"),
    ((1, 128, 0, 128, 128), ERR["K_BLOCK"], "K=0"),
    ((1, 128, 64, 128, 128), ERR["K_BLOCK"], "K=64"),
    ((1, 128, 200, 256, 128), ERR["K_BLOCK"], "multiple of 128"),
    ((1, 128, 256, 255, 128), ERR["PITCH"], "a=255"),
    ((1, 128, 256, 256, 100), ERR["PITCH"], "c=100"),
    ((1, 128, 256, 260, 128), ERR["A_PITCH_ALIGN"], "a_row_stride=260"),
    ((1, 0, 256, 256, 0), ERR["N_ZERO"], "n=0"),
    ((2 ** 31, 128, 128, 128, 128), ERR["RANGE"], "below 2^31"),
])
def test_checks_codes_and_messages(lib, args, code, needle):
    M, N, K, lda, ldc = args
    assert binding.check_args(M, N, K, lda, ldc) == code
    assert needle in binding.last_error()


def test_checks_run_in_the_pages_order(lib):
    # m=0 reported before the K rule, K before pitches, pitches before alignment
    assert binding.check_args(0, 128, 64, 3, 1) == ERR["M_ZERO"]
    assert binding.check_args(1, 128, 64, 3, 1) == ERR["K_BLOCK"]
    assert binding.check_args(1, 128, 128, 3, 1) == ERR["PITCH"]
    assert binding.check_args(1, 128, 128, 132, 128) == ERR["A_PITCH_ALIGN"]
    assert binding.check_args(1, 128, 128, 136, 128) == 0


def test_alignment_and_null_checks_before_any_device_work(lib):
    # the full entry point refuses before touching the device (there is none here)
    rc = binding.gemm_ptr(0, 128, 0, 0, 0, 128, 1, 128, 128)
    assert rc == ERR["NULL"] and "NULL A" in binding.last_error()
    rc = binding.gemm_ptr(0x1008, 128, 0x2000, 0x3000, 0x4000, 128, 1, 128, 128)
    assert rc == ERR["ALIGN"]
    rc = binding.gemm_ptr(0x1000, 128, 0x2000, 0x3002, 0x4000, 128, 1, 128, 128)
    assert rc == ERR["ALIGN"]
    rc = binding.gemm_ptr(0x1000, 128, 0x2000, 0x3000, 0x4001, 128, 1, 128, 128)
    assert rc == ERR["ALIGN"]
    assert binding.check_args(1, 128, 128, 128, 128, A=0x1008) == ERR["ALIGN"]


def test_valid_call_without_gpu_fails_loudly(lib):
    import torch
    if torch.cuda.is_available():
        pytest.skip("a GPU is present")
    rc = binding.gemm_ptr(0x1000, 128, 0x2000, 0x3000, 0x4000, 128, 1, 128, 128)
    assert rc == ERR["DEVICE"], binding.last_error()
    assert binding.last_error()


def test_strerror_covers_codes(lib):
    for c in list(ERR.values()) + [0, -10, -12, -13]:
        assert binding.strerror(c) and binding.strerror(c) != "unknown error code"
    assert binding.strerror(-999) == "unknown error code"


@pytest.mark.parametrize("M,N,K,tn", [(1, 256, 256, 2), (1, 4096, 4096, 2), (8, 12288, 4096, 16),
                                      (32, 14336, 5120, 32), (128, 28672, 8192, 128),
                                      (17, 1000, 1024, 32), (64, 512, 512, 64), (300, 512, 512, 128),
                                      (2, 4096, 4096, 2), (1, 14336, 4096, 16), (3, 4096, 4096, 16)])
def test_plans_for_the_workloads(lib, M, N, K, tn):
    p = binding.plan_for(M, N, K, sm_count=152)
    if tn == 2:
        assert p["variant"] == binding.VARIANT_GEMV
    else:
        assert p["variant"] == (binding.VARIANT_TC8 if M <= 16 else binding.VARIANT_TC)
    assert p["token_tile"] == tn
    ksteps = K // 128
    assert 1 <= p["split_k"] <= min(16, ksteps)
    # a split-K tail moves the last tail_tiles weight tiles to a second launch
    assert p["grid"][0] == (-(-N // 128) - p["tail_tiles"]) * p["split_k"]
    if p["tail_tiles"]:
        assert p["split_k"] == 1 and 2 <= p["tail_split"] <= min(16, ksteps)
        assert p["grid"][0] == 152 and p["tail_tiles"] * p["tail_split"] <= 152
    assert p["grid"][1] == -(-M // tn)
    assert p["cluster"][0] == p["split_k"]
    if p["variant"] == binding.VARIANT_TC8:
        assert p["block"][0] == 352
    elif p["variant"] == binding.VARIANT_GEMV:
        assert p["block"][0] == 256 and -(-ksteps // p["split_k"]) <= 8 and p["grid"][0] <= 152
    else:
        assert p["block"][0] == (768 if tn <= 32 else 640)
    assert p["tmem_cols"] * p["ctas_per_sm"] <= 512
    assert p["smem_bytes"] * p["ctas_per_sm"] <= 232448


def test_planner_fills_the_gpu_for_decode(lib):
    # a 32-tile decode GEMV must split K so that most SMs get work
    p = binding.plan_for(1, 4096, 4096, sm_count=152)
    ctas = p["grid"][0] * p["grid"][1]
    assert ctas >= 0.8 * 152                 # most SMs stream weights
    assert ctas <= 152 * p["ctas_per_sm"]    # in one wave


def test_planner_uses_cluster_capacity(lib):
    # A device where clusters of 8 only fit 15 at a time (120 CTAs) while 4-CTA
    # clusters fill 2 CTAs per SM: the 32-tile decode GEMV must not be split 8
    # ways (three waves of clusters); it picks a split whose clusters fit at once.
    cap = [0] + [304] * 4 + [300, 300, 294, 120] + [0] * 8
    p = binding.plan_for(3, 4096, 4096, sm_count=152, cluster_ctas=cap)   # 3 tokens: the two-term kernel
    s = p["split_k"]
    assert 32 * s <= cap[s], p
    assert s >= 4
    # a cluster size the device cannot run is never chosen
    cap2 = [0, 304, 0, 0, 0, 0, 0, 0, 0] + [0] * 8
    assert binding.plan_for(3, 4096, 4096, sm_count=152, cluster_ctas=cap2)["split_k"] == 1


def test_plan_variant_validation(lib):
    p = binding.plan_variant(8, 1024, 1024, binding.VARIANT_TC, split_k=4, stages=6)
    assert p.token_tile == 16 and p.variant == binding.VARIANT_TC
    p8 = binding.plan_variant(8, 1024, 1024, binding.VARIANT_TC8, split_k=2, stages=4)
    assert p8.variant == binding.VARIANT_TC8 and p8.block[0] == 352 and p8.tmem_cols == 128
    assert binding.plan_variant(100, 1024, 1024, binding.VARIANT_TC8).token_tile == 64
    assert p.split_k == 4 and p.stages == 6 and p.grid[0] == 8 * 4
    with pytest.raises(binding.W8A16Error) as e:
        binding.plan_variant(8, 1024, 1024, binding.VARIANT_TC, split_k=9)   # > K/128 = 8
    assert e.value.code == ERR["PLAN"]
    with pytest.raises(binding.W8A16Error):
        binding.plan_variant(8, 1024, 1024, binding.VARIANT_TC, stages=5)    # no instance
    # the widest token tile's 6-slot ring leaves room for small split-K receive
    # buffers only
    assert binding.plan_variant(100, 1024, 2048, binding.VARIANT_TC, split_k=2, stages=4).stages == 4
    assert binding.plan_variant(100, 1024, 2048, binding.VARIANT_TC, split_k=1, stages=6).stages == 6
    with pytest.raises(binding.W8A16Error) as e:
        binding.plan_variant(100, 1024, 2048, binding.VARIANT_TC, split_k=14, stages=6)
    assert "shared memory" in str(e.value)
    s = binding.plan_variant(8, 1024, 1024, binding.VARIANT_SIMT)
    assert s.variant == binding.VARIANT_SIMT and s.grid[0] == 128
    with pytest.raises(binding.W8A16Error):
        binding.plan_variant(8, 1024, 1024, 8)   # no such variant


def test_forced_plan_must_match_shape(lib):
    p = binding.plan_variant(8, 1024, 1024, binding.VARIANT_TC, split_k=2)
    rc = binding.gemm_ptr(0x1000, 1024, 0x2000, 0x3000, 0x4000, 2048, 8, 2048, 1024, plan=p)
    assert rc == ERR["PLAN"]


def test_version(lib):
    assert "sm_103a" in binding.version()


@pytest.mark.parametrize("args,code,needle", [
    # (dtype, ldw, N, K)
    ((0, 256, 0, 256), ERR["N_ZERO"], "n=0"),
    ((0, 256, 4, 200), ERR["K_BLOCK"], "K=200"),
    ((0, 200, 4, 256), ERR["PITCH"], "w_row_stride=200"),
    ((0, 258, 4, 256), ERR["A_PITCH_ALIGN"], "multiple of 4"),
    ((7, 256, 4, 256), -13, "unknown weight type"),
])
def test_quantizer_checks(lib, args, code, needle):
    dt, ldw, N, K = args
    rc = binding.quantize_weights_ptr(0x1000, dt, ldw, N, K, 0x2000, 0x3000)
    assert rc == code and needle in binding.last_error(), binding.last_error()


def test_quantizer_pointer_checks(lib):
    assert binding.quantize_weights_ptr(0, 0, 256, 4, 256, 0x2000, 0x3000) == ERR["NULL"]
    assert binding.quantize_weights_ptr(0x1008, 0, 256, 4, 256, 0x2000, 0x3000) == ERR["ALIGN"]
    assert binding.quantize_weights_ptr(0x1000, 0, 256, 4, 256, 0x2002, 0x3000) == ERR["ALIGN"]
    import torch
    if not torch.cuda.is_available():
        assert binding.quantize_weights_ptr(0x1000, 1, 256, 4, 256, 0x2000, 0x3000) == ERR["DEVICE"]


def test_quantizer_constants_match_header():
    text = binding.HEADER.read_text()
    assert int(re.search(r"W8A16_WEIGHTS_F32\s*=\s*(\d+)", text).group(1)) == binding.WEIGHTS_F32
    assert int(re.search(r"W8A16_WEIGHTS_BF16\s*=\s*(\d+)", text).group(1)) == binding.WEIGHTS_BF16


def test_workspace_bytes(lib):
    assert binding.workspace_bytes(32, 5120) == 2 * 32 * 5120 + 4 * 40 * 32
    assert binding.workspace_bytes(5, 256) == 2 * 5 * 256 + 4 * 2 * 8
    assert binding.workspace_bytes(0, 256) == 0 and binding.workspace_bytes(4, 200) == 0


def test_workspace_entry_checks(lib):
    args = (0x1000, 256, 0x2000, 0x3000, 0x4000, 256, 32, 256, 256)
    p = binding.plan_variant(32, 256, 256, binding.VARIANT_PRESPLIT, 1, 4)
    assert binding.gemm_ws_ptr(*args, 0, 0, plan=p) == -13
    assert "workspace" in binding.last_error()
    assert binding.gemm_ws_ptr(*args, 0x5008, 1 << 20) == ERR["ALIGN"]
    # the page's checks come first, as for w8a16_gemm
    assert binding.gemm_ws_ptr(0x1000, 256, 0x2000, 0x3000, 0x4000, 256, 0, 256, 256, 0x5000, 1 << 20) \
        == ERR["M_ZERO"]
    assert binding.gemm_ws_ptr(0x1000, 260, 0x2000, 0x3000, 0x4000, 256, 32, 256, 256, 0x5000, 1 << 20) \
        == ERR["A_PITCH_ALIGN"]
    assert binding.gemm_ws_ptr(*args, 0x5000, 1 << 20, flags=4) == -13


def test_presplit_plans(lib):
    for M, tn in ((1, 16), (17, 32), (33, 64), (100, 128)):
        p = binding.plan_variant(M, 4096, 4096, binding.VARIANT_PRESPLIT)
        assert p.variant == binding.VARIANT_PRESPLIT and p.token_tile == tn
        assert p.smem_bytes <= 232448 and p.tmem_cols in (128, 256, 512)
        assert p.grid[0] == 32 * p.split_k and p.block[0] in (256, 384, 640)


def test_split_k_tail_plans_are_validated(lib):
    """A tail needs the FP8 x FP8 kernel, one token tile, 1 <= tail_tiles < row tiles,
    2 <= tail_split <= min(16, K/128) and a first launch of the remaining tiles; the
    checks run before any device work."""
    p = binding.plan_variant(128, 1280, 1024, binding.VARIANT_PRESPLIT, 1, 4)
    args = (0x1000, 1024, 0x2000, 0x3000, 0x4000, 1280, 128, 1280, 1024)
    ws = (0x5000, 1 << 24)
    for tail, tsplit, grid0 in ((2, 1, 8), (10, 2, 0), (2, 9, 8), (2, 2, 10)):
        p.tail_tiles, p.tail_split, p.grid[0] = tail, tsplit, grid0
        rc = binding.gemm_ws_ptr(*args, *ws, plan=p)
        assert rc == ERR["PLAN"], (tail, tsplit, grid0, rc, binding.last_error())
    q = binding.plan_variant(8, 1280, 1024, binding.VARIANT_TC8, 1, 4)
    q.tail_tiles, q.tail_split, q.grid[0] = 2, 2, 8
    rc = binding.gemm_ws_ptr(0x1000, 1024, 0x2000, 0x3000, 0x4000, 1280, 8, 1280, 1024, *ws, plan=q)
    assert rc == ERR["PLAN"] and "tail" in binding.last_error()


def test_planner_adds_a_tail_only_past_one_wave(lib):
    sms = 152
    p = binding.plan_variant(128, 128 * 224, 8192, binding.VARIANT_PRESPLIT, 0, 0, sms)
    assert (p.split_k, p.tail_tiles, p.tail_split, p.grid[0]) == (1, 72, 2, 152)
    p = binding.plan_variant(128, 128 * 152, 8192, binding.VARIANT_PRESPLIT, 0, 0, sms)
    assert p.tail_tiles == 0 and p.grid[0] == 152
    p = binding.plan_variant(128, 128 * 224, 8192, binding.VARIANT_PRESPLIT, 1, 0, sms)
    assert p.tail_tiles == 0, "an explicit split has no tail"


@pytest.mark.parametrize("variant", [0, 2, 3, 4, 5])
def test_planner_invariants_over_shapes(lib, variant):
    """Every plan the pure planner emits fits one SM's resources, covers the shape
    exactly once (grid x split x tail) and keeps its split and tail in range."""
    Ms = [1, 2, 7, 16, 17, 31, 32, 33, 64, 65, 100, 128, 129, 200, 256, 1000]
    Ns = [1, 100, 128, 129, 1000, 4096, 12288, 28672, 38912]
    Ks = [128, 256, 1280, 4096, 8192]
    for M in Ms:
        for N in Ns:
            for K in Ks:
                try:
                    p = binding.plan_variant(M, N, K, variant, 0, 0, 152)
                except binding.W8A16Error as e:
                    pytest.fail(f"no plan for M={M} N={N} K={K} v={variant}: {e}")
                d = p.as_dict()
                if d["variant"] == binding.VARIANT_SIMT:
                    continue
                ksteps, row_tiles = K // 128, -(-N // 128)
                assert 1 <= d["split_k"] <= min(16, ksteps)
                assert d["smem_bytes"] <= 232448 and d["tmem_cols"] in (32, 64, 128, 256, 512)
                assert d["ctas_per_sm"] >= 1
                assert d["tmem_cols"] * d["ctas_per_sm"] <= 512
                assert (d["smem_bytes"] + 1024) * d["ctas_per_sm"] <= 233472
                assert d["block"][0] * d["ctas_per_sm"] <= 2048
                assert d["grid"][1] == -(-M // d["token_tile"]) and d["grid"][1] <= 65535
                tail = d["tail_tiles"]
                assert d["grid"][0] == (row_tiles - tail) * d["split_k"]
                if tail:
                    assert d["grid"][1] == 1 and d["split_k"] == 1
                    assert 2 <= d["tail_split"] <= min(16, ksteps)
                    assert 0 < tail < row_tiles
                    assert tail * d["tail_split"] <= 152 * d["ctas_per_sm"]


@pytest.mark.parametrize("args,code,needle", [
    # (lda, a_scale_stride, ldc, M, N, K)
    ((256, 8, 256, 0, 256, 256), ERR["M_ZERO"], "m=0"),
    ((256, 8, 256, 8, 256, 200), ERR["K_BLOCK"], "K=200"),
    ((200, 8, 256, 8, 256, 256), ERR["PITCH"], "a=200"),
    ((256, 4, 256, 8, 256, 256), ERR["PITCH"], "a_scale=4"),
    ((264, 8, 256, 8, 256, 256), ERR["A_PITCH_ALIGN"], "a_row_stride=264"),
    ((256, 10, 256, 8, 256, 256), ERR["A_PITCH_ALIGN"], "a_scale_stride=10"),
    ((256, 8, 256, 8, 0, 256), ERR["N_ZERO"], "n=0"),
])
def test_w8a8_checks(lib, args, code, needle):
    lda, sst, ldc, M, N, K = args
    rc = binding.gemm_w8a8_ptr(0x1000, lda, 0x2000, sst, 0x3000, 0x4000, 0x5000, ldc, M, N, K)
    assert rc == code and needle in binding.last_error(), (rc, binding.last_error())


def test_w8a8_pointer_and_flag_checks(lib):
    good = (0x1000, 256, 0x2000, 8, 0x3000, 0x4000, 0x5000, 256, 8, 256, 256)
    assert binding.gemm_w8a8_ptr(0, *good[1:]) == ERR["NULL"]
    assert binding.gemm_w8a8_ptr(0x1008, *good[1:]) == ERR["ALIGN"]
    assert binding.gemm_w8a8_ptr(*good[:2], 0x2008, *good[3:]) == ERR["ALIGN"]
    assert binding.gemm_w8a8_ptr(*good, flags=2) == -13


@pytest.mark.parametrize("args,code,needle", [
    # (a_row_stride, M, K, scale_stride)
    ((256, 0, 256, 4), ERR["M_ZERO"], "m=0"),
    ((256, 4, 200, 4), ERR["K_BLOCK"], "K=200"),
    ((200, 4, 256, 4), ERR["PITCH"], "a_row_stride=200"),
    ((256, 5, 256, 4), ERR["PITCH"], "scale_stride=4"),
    ((260, 4, 256, 4), ERR["A_PITCH_ALIGN"], "a_row_stride=260"),
    ((256, 4, 256, 6), ERR["A_PITCH_ALIGN"], "scale_stride=6"),
])
def test_activation_quantiser_checks(lib, args, code, needle):
    lda, M, K, sst = args
    rc = binding.load().w8a16_quantize_activations(0x1000, lda, M, K, 0x2000, 0x3000, sst, None)
    assert rc == code and needle in binding.last_error(), (rc, binding.last_error())


# ---- the binding's own checks: placement, dtypes and extents, before any call ----

def _cpu_operands(M=4, N=200, K=256):
    import torch
    A = torch.zeros((M, K), dtype=torch.bfloat16)
    W = torch.zeros((N, K), dtype=torch.uint8)
    S = torch.ones(((N + 127) // 128, K // 128), dtype=torch.float32)
    C = torch.zeros((M, N), dtype=torch.bfloat16)
    return A, W, S, C


def test_binding_refuses_host_tensors_for_device_calls(lib):
    A, W, S, C = _cpu_operands()
    for call in (lambda: binding.gemm(A, W, S, C), lambda: binding.gemm_ws(A, W, S, C, workspace=False),
                 lambda: binding.gemm_noalloc(A, W, S, C)):
        with pytest.raises(ValueError, match="CUDA device"):
            call()


def test_binding_checks_block_scale_extent(lib):
    import torch
    A, W, S, C = _cpu_operands(N=200, K=256)
    for bad in (torch.ones((1, 2)), torch.ones((2, 1)), torch.ones((2, 3))):
        with pytest.raises(ValueError, match=r"block_scale must be \[2, 2\]"):
            binding.gemm(A, W, bad, C)


def test_binding_checks_w8a8_operands(lib):
    import torch
    M, N, K = 4, 200, 256
    q = torch.zeros((M, K), dtype=torch.uint8)
    qs = torch.ones((K // 128, 4), dtype=torch.float32)
    W = torch.zeros((N, K), dtype=torch.uint8)
    S = torch.ones((2, 2), dtype=torch.float32)
    C = torch.zeros((M, N), dtype=torch.bfloat16)
    cases = [
        ((q.to(torch.bfloat16), qs, W, S, C), "A_codes"),
        ((q, torch.ones((1, 4)), W, S, C), "a_scale"),
        ((q, torch.ones((2, 3)), W, S, C), "a_scale"),
        ((q, qs, W[:, :128].contiguous(), S, C), "W must"),
        ((q, qs, W, torch.ones((2, 1)), C), "block_scale must be"),
        ((q, qs, W, S, C.float()), "C must"),
        ((q, qs, W, S, C), "CUDA device"),
    ]
    for args, needle in cases:
        with pytest.raises(ValueError, match=needle):
            binding.gemm_w8a8(*args)


def test_binding_checks_host_call_buffers(lib):
    import torch
    A, W, S, C = _cpu_operands()
    with pytest.raises(ValueError, match="C_host"):
        binding.gemm_host(A, W, S, C.float(), A, W, S, C)
    with pytest.raises(ValueError, match="CUDA device"):
        binding.gemm_host(A, W, S, C, A, W, S, C)


def test_binding_quantisers_refuse_host_tensors(lib):
    import torch
    with pytest.raises(ValueError, match="CUDA device"):
        binding.quantize_weights(torch.zeros((128, 256), dtype=torch.float32))
    with pytest.raises(TypeError, match="float32 or bfloat16"):
        binding.quantize_weights(torch.zeros((128, 256), dtype=torch.float16))
    with pytest.raises(ValueError, match="CUDA bfloat16"):
        binding.quantize_activations(torch.zeros((4, 256), dtype=torch.bfloat16))


def test_decode_kernel_plans(lib):
    """The decode kernel (M <= 2): at most 8 K steps per CTA, at most one CTA per SM
    in all, the largest portable split that satisfies both and leaves each CTA at
    least two K steps; otherwise the two-term kernel. Forced decode plans are
    validated against the shape."""
    for (M, N, K, split) in [(1, 4096, 4096, 4), (2, 4096, 4096, 4), (1, 256, 256, 1), (1, 2048, 4096, 8),
                             (1, 4096, 1024, 4), (2, 130, 640, 2), (1, 19 * 128, 8192, 8), (1, 1024, 1024, 4),
                             (1, 128, 128, 1), (1, 2048, 2048, 8)]:
        p = binding.plan_variant(M, N, K, 0, 0, 0, 152).as_dict()
        assert p["variant"] == binding.VARIANT_GEMV and p["split_k"] == split, (M, N, K, p)
        assert p["grid"][0] == -(-N // 128) * split <= 152 and p["cluster"][0] == split
        assert p["ctas_per_sm"] == 2 and p["tmem_cols"] == 128 and p["block"][0] == 256
    for (M, N, K) in [(1, 4096, 8192), (1, 14336, 4096), (3, 4096, 4096), (1, 20 * 128, 8192)]:
        assert binding.plan_variant(M, N, K, 0, 0, 0, 152).variant != binding.VARIANT_GEMV, (M, N, K)
    q = binding.plan_variant(1, 4096, 4096, binding.VARIANT_GEMV, 8, 0, 152)
    assert q.split_k == 8 and q.grid[0] == 256          # forced: more CTAs than SMs is allowed
    for bad in [dict(M=3), dict(split=2), dict(split=17), dict(stages=4)]:
        with pytest.raises(binding.W8A16Error):
            binding.plan_variant(bad.get("M", 1), 4096, 4096, binding.VARIANT_GEMV, bad.get("split", 4),
                                 bad.get("stages", 0), 152)


def _stream_cta_of(u, units, ctas):
    """The CTA whose contiguous range [c U / P, (c + 1) U / P) holds unit u (brute force)."""
    for c in range(ctas):
        if c * units // ctas <= u < (c + 1) * units // ctas:
            return c
    raise AssertionError(u)


def test_stream_plans(lib):
    """Stream-K plans (3..32 tokens): one token tile of 16 or 32, 4 stages, split 1,
    min(units, 2 x SMs) CTAs of at most the two-CTAs-per-SM resources; refused
    outside 3..32 tokens or with another split or stage count."""
    for (M, N, K) in [(3, 256, 256), (8, 12288, 4096), (16, 4096, 4096), (17, 14336, 5120), (32, 14336, 5120),
                      (24, 300, 1280), (32, 128, 128)]:
        p = binding.plan_variant(M, N, K, binding.VARIANT_STREAM, 0, 0, 152).as_dict()
        units = -(-N // 128) * (K // 128)
        assert p["variant"] == binding.VARIANT_STREAM and p["split_k"] == 1 and p["stages"] == 4
        assert p["token_tile"] == (16 if M <= 16 else 32)
        assert p["grid"] == [min(units, 304), 1, 1] and p["cluster"][0] == 1 and p["ctas_per_sm"] == 2
        assert p["tmem_cols"] * p["ctas_per_sm"] <= 512 and p["smem_bytes"] * p["ctas_per_sm"] <= 232448
        assert not p["tail_tiles"] and not p["tail_split"]
    for bad in [dict(M=2), dict(M=33), dict(split=2), dict(stages=6)]:
        with pytest.raises(binding.W8A16Error):
            binding.plan_variant(bad.get("M", 8), 4096, 4096, binding.VARIANT_STREAM, bad.get("split", 0),
                                 bad.get("stages", 0), 152)


def test_stream_cta_ranges_cover_every_unit_once():
    """The host's closed form for the CTA of a unit matches the brute-force range
    search, so every unit is in exactly one CTA's range and a tile's segments are
    the CTAs from the first unit's to the last unit's."""
    import itertools
    for units, ctas in itertools.product([1, 7, 64, 120, 257, 3072], [1, 3, 5, 64, 120, 304]):
        if ctas > units:
            continue
        owners = [_stream_cta_of(u, units, ctas) for u in range(units)]
        assert owners == sorted(owners) and owners[0] == 0 and owners[-1] == ctas - 1
        assert len(set(owners)) == ctas      # every CTA has at least one unit
        closed = [((u + 1) * ctas - 1) // units for u in range(units)]
        assert closed == owners


def test_stream_workspace_bytes(lib):
    """workspace_bytes_for: where the stream-K plan applies, the split's terms, a
    256-aligned counter per 128-row tile and, 256-aligned after them, 128 x token
    tile FP32 partials for each of the most segments any tile has; elsewhere the
    pre-split bytes above 16 tokens, else 0."""
    for (M, N, K) in [(3, 256, 256), (8, 12288, 4096), (32, 14336, 5120), (24, 300, 1280), (5, 129, 128)]:
        P = min(-(-N // 128) * (K // 128), 304)
        tiles, ksteps = -(-N // 128), K // 128
        units = tiles * ksteps
        maxseg = max(_stream_cta_of(t * ksteps + ksteps - 1, units, P) - _stream_cta_of(t * ksteps, units, P) + 1
                     for t in range(tiles))
        tn = 16 if M <= 16 else 32
        align = lambda x: -(-x // 256) * 256
        parts = align(align(binding.workspace_bytes(M, K)) + 4 * tiles)
        sms = 152
        # the library asks the current device for its SM count; without one it assumes 152
        got = binding.workspace_bytes_for(M, N, K)
        if got != parts + tiles * maxseg * 128 * tn * 4:
            pytest.skip(f"device with another SM count than {sms}")
    assert binding.workspace_bytes_for(1, 4096, 4096) == 0
    assert binding.workspace_bytes_for(64, 4096, 4096) == binding.workspace_bytes(64, 4096)
    assert binding.workspace_bytes_for(8, 4096, 100) == 0
