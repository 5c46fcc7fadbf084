"""Guard bands (the stand-in for a memory checker): every entry point writes C, the
workspace and the quantisers' outputs only inside their extents. Each output lives
in the middle of a larger device buffer whose bands before and after hold a fixed
pattern, checked byte for byte after the call, with C's pad columns."""
from __future__ import annotations

import numpy as np
import pytest
import torch

import workloads

pytestmark = pytest.mark.gpu
BAND = 4096   # bytes before and after


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from fp8_weight_only_gemm_gb300.build import build_library
    from fp8_weight_only_gemm_gb300 import binding
    build_library()
    binding.load()
    yield
    assert binding.device_status()[0] == 0


def _guarded(nbytes: int, fill=0x5A):
    """(whole buffer, view of nbytes in its middle) on the GPU, 256-byte aligned."""
    buf = torch.full((BAND + nbytes + BAND,), fill, dtype=torch.uint8, device="cuda")
    return buf, buf[BAND:BAND + nbytes]


def _bands_intact(buf, nbytes, fill=0x5A):
    h = buf.cpu().numpy()
    return bool((h[:BAND] == fill).all() and (h[BAND + nbytes:] == fill).all())


def _c_view(case):
    wl = case.wl
    nbytes = wl.M * wl.ldc * 2
    buf, v = _guarded(nbytes)
    C = v.view(torch.bfloat16).view(wl.M, wl.ldc)
    C.copy_(case.C0.cuda())
    return buf, nbytes, C


def _check_c(case, buf, nbytes, C, label):
    wl = case.wl
    assert _bands_intact(buf, nbytes), f"{label}: wrote outside C"
    got = C.view(torch.int16).cpu().numpy().view(np.uint16)
    assert (got[:, wl.N:] == workloads.C_PAD_FILL).all(), f"{label}: wrote C's pad columns"
    assert not (got[:, :wl.N] == workloads.C_USED_SENTINEL).any(), f"{label}: left outputs unwritten"


@pytest.mark.parametrize("M,N,K", [(1, 300, 512), (8, 1000, 1024), (33, 257, 640), (130, 384, 768)])
def test_every_entry_point_stays_inside_its_buffers(M, N, K):
    from fp8_weight_only_gemm_gb300 import binding
    case = workloads.make_case("strided_m32_n14336_k5120", M=M, N=N, K=K, a_row_stride=K + 64,
                               c_row_stride=N + 5, seed=M + N + K)
    wl = case.wl
    A, W, S = case.A.cuda()[:, :K], case.W.cuda(), case.scale.cuda()
    calls = {
        "gemm": lambda C: binding.gemm(A, W, S, C[:, :N]),
        "gemm_noalloc": lambda C: binding.gemm_noalloc(A, W, S, C[:, :N]),
    }
    for v in (binding.VARIANT_TC, binding.VARIANT_TC8, binding.VARIANT_SIMT):
        p = binding.plan_variant(M, N, K, v, 0, 0)
        calls[f"variant{v}"] = (lambda p: lambda C: binding.gemm(A, W, S, C[:, :N], plan=p))(p)
    for name, call in calls.items():
        buf, nbytes, C = _c_view(case)
        call(C)
        torch.cuda.synchronize()
        _check_c(case, buf, nbytes, C, name)
    # the workspace path, and the workspace itself
    need = binding.workspace_bytes(M, K)
    wbuf, ws = _guarded(need)
    buf, nbytes, C = _c_view(case)
    binding.gemm_ws(A, W, S, C[:, :N], workspace=ws)
    torch.cuda.synchronize()
    _check_c(case, buf, nbytes, C, "gemm_ws")
    assert _bands_intact(wbuf, need), "gemm_ws wrote outside its workspace"
    # the forced stream-K plan (3..32 tokens): counters and partials inside its layout
    need_sk = binding.workspace_bytes_for(M, N, K)
    if 3 <= M <= 32:
        p = binding.plan_variant(M, N, K, binding.VARIANT_STREAM, 0, 0)
        wbuf, ws = _guarded(need_sk)
        buf, nbytes, C = _c_view(case)
        binding.gemm_ws(A, W, S, C[:, :N], workspace=ws, plan=p)
        torch.cuda.synchronize()
        _check_c(case, buf, nbytes, C, "gemm_ws stream-K")
        assert _bands_intact(wbuf, need_sk), "gemm_ws (stream-K) wrote outside its workspace"


def test_quantisers_and_w8a8_stay_inside_their_buffers():
    from fp8_weight_only_gemm_gb300 import binding
    M, N, K = 37, 300, 640
    case = workloads.make_case("strided_m32_n14336_k5120", M=M, N=N, K=K, a_row_stride=K + 64,
                               c_row_stride=N + 5, seed=77)
    A = case.A.cuda()[:, :K]
    S_stride = (M + 3) // 4 * 4
    cbuf, cv = _guarded(M * K)
    sbuf, sv = _guarded((K // 128) * S_stride * 4)
    codes, scales = cv.view(M, K), sv.view(torch.float32).view(K // 128, S_stride)
    rc = binding.load().w8a16_quantize_activations(A.data_ptr(), A.stride(0), M, K, codes.data_ptr(),
                                                   scales.data_ptr(), S_stride, None)
    assert rc == 0
    torch.cuda.synchronize()
    assert _bands_intact(cbuf, M * K) and _bands_intact(sbuf, (K // 128) * S_stride * 4)
    buf, nbytes, C = _c_view(case)
    binding.gemm_w8a8(codes, scales, case.W.cuda(), case.scale.cuda(), C[:, :N])
    torch.cuda.synchronize()
    _check_c(case, buf, nbytes, C, "w8a8")
    wd = (torch.randn(300, 648) * 0.02).cuda()
    wbuf, wv = _guarded(300 * 640)
    sbuf2, sv2 = _guarded(3 * 5 * 4)
    rc = binding.quantize_weights_ptr(wd.data_ptr(), 0, 648, 300, 640, wv.data_ptr(), sv2.data_ptr())
    assert rc == 0
    torch.cuda.synchronize()
    assert _bands_intact(wbuf, 300 * 640) and _bands_intact(sbuf2, 3 * 5 * 4)
