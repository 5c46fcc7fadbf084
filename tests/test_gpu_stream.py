"""GPU parity of the persistent stream-K plan of the pre-split path
(W8A16_VARIANT_STREAM, 3..32 tokens) against the CPU oracle, element by element:
CTA counts that put one unit per CTA (a tile summed from up to 40 segments), CTAs
that span several tiles, a single CTA (every tile whole), K = 128 (every segment
whole), ragged N and row pitches; run-to-run determinism (fixed segment order),
the tile counters back at zero after each call (and a workspace's prior contents
irrelevant), NaN propagation through a split tile and chains of programmatic
dependent launches. The plan runs only when forced (the planner does not choose it). The two-term error bound of tests/parity.py
applies, with one rounding per summed segment."""
from __future__ import annotations

import numpy as np
import pytest
import torch

import workloads
from parity import compare, oracle_full

pytestmark = pytest.mark.gpu
STREAM = 7


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


def _sms():
    return torch.cuda.get_device_properties(0).multi_processor_count


def _plan(M, N, K, ctas=0):
    from fp8_weight_only_gemm_gb300 import binding
    p = binding.plan_variant(M, N, K, STREAM, 0, 0, _sms())
    assert p.variant == STREAM and p.split_k == 1 and p.grid[1] == 1
    if ctas:
        p.grid[0] = ctas
    return p


def _ws_bound(M, N, K, tn):
    """Workspace bytes that cover any CTA count: the split, the counters and
    ceil(N/128) x min(K/128, CTAs) segments of 128 x tn FP32 partials."""
    from fp8_weight_only_gemm_gb300 import binding
    tiles, ksteps = -(-N // 128), K // 128
    return binding.workspace_bytes(M, K) + 512 + 4 * tiles + tiles * ksteps * 128 * tn * 4


def _counters(ws, M, N, K):
    """The tile counters: one uint32 per 128-row weight tile, 256-byte aligned after
    the split's terms and factors."""
    from fp8_weight_only_gemm_gb300 import binding
    off = -(-binding.workspace_bytes(M, K) // 256) * 256
    tiles = -(-N // 128)
    return ws[off:off + 4 * tiles].cpu().view(torch.int32)


def run_ws(case, plan=None, workspace=None, flags=0):
    from fp8_weight_only_gemm_gb300 import binding
    wl = case.wl
    A, W, S, C = case.A.cuda(), case.W.cuda(), case.scale.cuda(), case.C0.cuda()
    binding.gemm_ws(A[:, :wl.K], W, S, C[:, :wl.N], workspace=workspace, plan=plan, flags=flags)
    torch.cuda.synchronize()
    return C.cpu().view(torch.int16).numpy().view(np.uint16)


@pytest.mark.parametrize("M,N,K,lda,ldc,ctas", [
    (3, 1000, 1024, 1032, 1003, 0),     # 64 units on 64 CTAs: 8 segments per tile
    (8, 1000, 1024, 1024, 1000, 5),     # 12.8 units per CTA: CTAs across tile boundaries
    (16, 384, 5120, 5120, 390, 0),      # 120 CTAs, one unit each: 40 segments per tile
    (17, 640, 2048, 2056, 640, 7),
    (24, 300, 1280, 1280, 301, 3),
    (32, 640, 2048, 2048, 645, 1),      # one CTA: every tile whole, no partials
    (32, 2000, 1024, 1024, 2000, 0),
    (5, 129, 128, 128, 130, 0),         # K = 128: one step per tile, every segment whole
    (29, 1280, 3072, 3080, 1290, 37),
])
def test_forced_stream_plans(M, N, K, lda, ldc, ctas):
    case = workloads.make_case("strided_m32_n14336_k5120", M=M, N=N, K=K, a_row_stride=lda,
                               c_row_stride=ldc, seed=M * 131 + N + K + ctas, outlier_frac=0.01)
    p = _plan(M, N, K, ctas)
    ws = torch.empty(_ws_bound(M, N, K, p.token_tile), dtype=torch.uint8, device="cuda")
    got = run_ws(case, plan=p, workspace=ws)
    ref, exact, absum = oracle_full(case)
    compare(case, got, ref, exact, absum, split_k=K // 128, label=f"stream M{M} N{N} K{K} P{p.grid[0]}",
            variant=3)
    assert not np.any(got.reshape(M, ldc)[:, :N] == workloads.C_USED_SENTINEL)
    # columns past N untouched
    assert np.array_equal(got.reshape(M, ldc)[:, N:], case.C0.view(torch.int16).numpy().view(np.uint16)
                          .reshape(M, ldc)[:, N:])
    assert not _counters(ws, M, N, K).any(), "tile counters not back at zero"
    for _ in range(2):
        assert np.array_equal(got, run_ws(case, plan=p, workspace=ws)), "same plan, different bits"


@pytest.mark.parametrize("name", ["skinny_qkv_m8_n12288_k4096", "strided_m32_n14336_k5120"])
def test_workloads_on_the_stream_plan(name):
    """The full-size workloads on the forced stream-K plan, with a workspace of
    workspace_bytes_for (which the planner, left to itself, does not spend on it)."""
    from fp8_weight_only_gemm_gb300 import binding
    case = workloads.make_case(name)
    wl = case.wl
    need = binding.workspace_bytes_for(wl.M, wl.N, wl.K)
    assert need > binding.workspace_bytes(wl.M, wl.K)
    assert binding.plan_ws(wl.M, wl.N, wl.K, need)["variant"] == (
        5 if wl.M > 16 else binding.plan_current(wl.M, wl.N, wl.K)["variant"])
    ws = torch.empty(need, dtype=torch.uint8, device="cuda")
    p = _plan(wl.M, wl.N, wl.K)
    got = run_ws(case, plan=p, workspace=ws)
    ref, exact, absum = oracle_full(case)
    compare(case, got, ref, exact, absum, split_k=wl.K // 128, label=f"stream/{name}", variant=3)
    assert not np.any(got.reshape(wl.M, wl.ldc)[:, :wl.N] == workloads.C_USED_SENTINEL)
    assert np.array_equal(got, run_ws(case, plan=p, workspace=ws))


def test_workspace_contents_do_not_matter():
    """The split pre-pass clears the tile counters: a workspace full of garbage gives
    the bits of a zero-filled one, call after call, and each call leaves the
    counters at zero."""
    M, N, K = 12, 3000, 2048
    case = workloads.make_case("skinny_qkv_m8_n12288_k4096", M=M, N=N, K=K, seed=901)
    p = _plan(M, N, K)
    need = _ws_bound(M, N, K, p.token_tile)
    base = run_ws(case, plan=p, workspace=torch.zeros(need, dtype=torch.uint8, device="cuda"))
    ref, exact, absum = oracle_full(case)
    compare(case, base, ref, exact, absum, split_k=K // 128, label="stream base", variant=3)
    junk = torch.full((need,), 0xAB, dtype=torch.uint8, device="cuda")
    for _ in range(3):
        assert np.array_equal(run_ws(case, plan=p, workspace=junk), base)
        assert not _counters(junk, M, N, K).any()


def test_nan_weight_in_a_split_tile():
    """A NaN weight code makes exactly its output row NaN for every token, also when
    its tile is summed from several CTAs' partials."""
    from fp8_weight_only_gemm_gb300 import binding
    M, N, K = 6, 256, 2048
    case = workloads.make_case("skinny_qkv_m8_n12288_k4096", M=M, N=N, K=K, seed=902)
    case.W[70, 1500] = 0x7F
    p = _plan(M, N, K)            # 32 units on 32 CTAs: each tile from 16 segments
    assert p.grid[0] == 32
    ws = torch.empty(_ws_bound(M, N, K, p.token_tile), dtype=torch.uint8, device="cuda")
    got = run_ws(case, plan=p, workspace=ws).reshape(M, N)
    isnan = ((got & 0x7F80) == 0x7F80) & ((got & 0x7F) != 0)
    assert isnan[:, 70].all() and isnan.sum() == M
    case.W[70, 1500] = 0
    got = run_ws(case, plan=p, workspace=ws)
    ref, exact, absum = oracle_full(case)
    compare(case, got, ref, exact, absum, split_k=K // 128, label="stream nan-free twin", variant=3)


@pytest.mark.parametrize("M", [4, 16, 32])
def test_programmatic_chain(M):
    """Dependent calls through one workspace (each A the previous call's C, N = K =
    2048) with the programmatic-launch flag give the bits of the chain without it,
    and the first link matches the oracle."""
    from fp8_weight_only_gemm_gb300 import binding
    K = 2048
    cases = [workloads.make_case("strided_m32_n14336_k5120", M=M, N=K, K=K, a_row_stride=K, c_row_stride=K,
                                 seed=700 + i) for i in range(5)]
    Ws = [c.W.cuda() for c in cases]
    Ss = [c.scale.cuda() for c in cases]
    ws = torch.empty(binding.workspace_bytes_for(M, K, K), dtype=torch.uint8, device="cuda")
    p = _plan(M, K, K)
    x0 = cases[0].A.cuda()[:, :K]

    def chain(flags):
        xs = [x0]
        for W, S in zip(Ws, Ss):
            xs.append(binding.gemm_ws(xs[-1], W, S, workspace=ws, plan=p, flags=flags))
        torch.cuda.synchronize()
        return [x.view(torch.int16).cpu().numpy().view(np.uint16) for x in xs]

    ref_bits = chain(0)
    for _ in range(3):
        for a, b in zip(chain(binding.FLAG_PDL), ref_bits):
            assert np.array_equal(a, b)
    c = cases[0]
    ref, exact, absum = oracle_full(c)
    compare(c, ref_bits[1].reshape(M, K), ref, exact, absum, split_k=K // 128, label="stream chain", variant=3)


def test_forced_stream_plan_checks():
    """A forced stream-K plan is refused outside 3..32 tokens and without its
    workspace."""
    from fp8_weight_only_gemm_gb300 import binding
    with pytest.raises(binding.W8A16Error):
        binding.plan_variant(2, 256, 256, STREAM, 0, 0, _sms())
    with pytest.raises(binding.W8A16Error):
        binding.plan_variant(33, 256, 256, STREAM, 0, 0, _sms())
    case = workloads.make_case("skinny_qkv_m8_n12288_k4096", M=8, N=512, K=1024, seed=903)
    A, W, S = case.A.cuda()[:, :1024], case.W.cuda(), case.scale.cuda()
    p = _plan(8, 512, 1024)
    short = torch.empty(binding.workspace_bytes(8, 1024), dtype=torch.uint8, device="cuda")
    with pytest.raises(binding.W8A16Error, match="workspace"):
        binding.gemm_ws(A, W, S, workspace=short, plan=p)
