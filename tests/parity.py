"""Shared helpers for the GPU parity tests: running a workload through the C-ABI
binding and comparing with the oracle element by element.

Tolerances:
  * the operation's stated bar, per element:
        |gpu - ref| <= 2^-7 * |ref| + 1e-3 * sqrt(K) * max|A| * max|W * scale|
    with ref the oracle's BF16 result;
  * a tighter bound derived from the arithmetic, used to catch bugs the stated
    bar is too loose for (a wrong but similar block scale, a dropped K step): the
    GPU's FP32 value differs from the exact sum by at most
        (K/128 + 256 + split_k) * 2^-23 * sum_k |A * W * scale|
    (tensor-core step sums, one fold per step, the cluster reduction), and
    rounding to BF16 adds half an ulp of the result. The FP8-datapath variant
    (TC8) represents each activation as two E4M3 terms, exact for values at
    least 2^-14 of their 128-K block maximum and within 2^-22 of it otherwise,
    which adds at most 2^-22 * max|A[m, :]| * sum_k |W[n, k] * scale| (the
    tests allow twice that).
"""
from __future__ import annotations

import math

import numpy as np
import torch

import oracle
import workloads


def bf16_to_f64(codes: np.ndarray) -> np.ndarray:
    return (codes.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def ulp_bf16(x: np.ndarray) -> np.ndarray:
    a = np.nan_to_num(np.abs(x), nan=1.0, posinf=1.0)
    e = np.floor(np.log2(np.maximum(a, 2.0 ** -126)))
    return np.ldexp(1.0, (e - 7).astype(np.int64))


def run_gpu(case: workloads.Case, plan=None, device="cuda:0"):
    """Upload the case, run the library, return the full C [M, ldc] as uint16 codes."""
    import fp8_weight_only_gemm_gb300 as w8
    wl = case.wl
    A = case.A.to(device)
    W = case.W.to(device)
    S = case.scale.to(device)
    C = case.C0.to(device)
    w8.gemm(A[:, :wl.K], W, S, C[:, :wl.N], plan=plan)
    torch.cuda.synchronize()
    return C.cpu().view(torch.int16).numpy().view(np.uint16)


def oracle_full(case: workloads.Case):
    wl = case.wl
    C, exact, absum = oracle.get().gemm(case.A_np(), case.W_np(), case.scale_np(), wl.M, wl.N, wl.K,
                                        a_row_stride=wl.lda, C=case.C0_np(), c_row_stride=wl.ldc,
                                        want_exact=True)
    return C, exact, absum


def stated_tolerance(case: workloads.Case, ref: np.ndarray) -> np.ndarray:
    wl = case.wl
    a = case.A[:, :wl.K].to(torch.float64).abs().nan_to_num(0.0, posinf=0.0).max().item()
    w = case.W.view(torch.float8_e4m3fn).to(torch.float64).abs().nan_to_num(0.0)
    s = case.scale.to(torch.float64)
    nb = s.shape[0]
    ws = 0.0
    for i in range(nb):
        blk = w[i * 128:(i + 1) * 128].reshape(-1, wl.K // 128, 128).amax(dim=(0, 2))
        ws = max(ws, float((blk * s[i]).max()))
    return 2.0 ** -7 * np.abs(ref) + 1e-3 * math.sqrt(wl.K) * a * ws


def split_term_bound(case: workloads.Case) -> np.ndarray:
    """2^-21 * max_k |A[m, k]| * sum_k |W[n, k] * scale|  ([M, N])."""
    wl = case.wl
    a = case.A[:, :wl.K].to(torch.float64).abs().nan_to_num(0.0, posinf=0.0).amax(dim=1).numpy()
    w = case.W.view(torch.float8_e4m3fn).to(torch.float64).abs().nan_to_num(0.0)
    s = case.scale.to(torch.float64).repeat_interleave(128, dim=0)[:wl.N]
    s = s.repeat_interleave(128, dim=1)
    wabs = (w * s).sum(dim=1).numpy()
    return 2.0 ** -21 * a[:, None] * wabs[None, :]


def compare(case: workloads.Case, got: np.ndarray, ref_C: np.ndarray, exact: np.ndarray,
            absum: np.ndarray, split_k: int = 1, label: str = "", variant: int = 2):
    """Element-by-element comparison of a GPU result with the oracle; asserts."""
    wl = case.wl
    M, N = wl.M, wl.N
    got = got.reshape(M, wl.ldc)
    ref_C = ref_C.reshape(M, wl.ldc)
    # pad columns untouched, bit for bit
    assert np.array_equal(got[:, N:], ref_C[:, N:]), f"{label}: pad columns of C were written"
    g = bf16_to_f64(got[:, :N])
    r = bf16_to_f64(ref_C[:, :N])
    nan_r = np.isnan(r)
    assert np.array_equal(np.isnan(g), nan_r), f"{label}: NaN pattern differs (unwritten outputs?)"
    fin = ~nan_r
    tol = stated_tolerance(case, r)
    err = np.abs(g - r)
    bad = fin & ~(err <= tol)
    assert not bad.any(), (f"{label}: {bad.sum()} outputs outside the stated tolerance; first at "
                           f"{np.argwhere(bad)[0]}: gpu={g[bad][0]} ref={r[bad][0]} tol={tol[bad][0]}")
    gamma = (wl.K / 128 + 256 + split_k) * 2.0 ** -23
    extra = split_term_bound(case) if variant == 3 else 0.0
    tight = gamma * absum + extra + 0.5 * ulp_bf16(np.abs(exact) + gamma * absum + extra) + 2.0 ** -133
    err2 = np.abs(g - exact)
    bad2 = fin & ~(err2 <= tight)
    assert not bad2.any(), (f"{label}: {bad2.sum()} outputs outside the arithmetic error bound; first "
                            f"at {np.argwhere(bad2)[0]}: gpu={g[bad2][0]} exact={exact[bad2][0]} "
                            f"bound={tight[bad2][0]}")
    return float(np.max(err[fin] / np.maximum(tol[fin], 1e-300))) if fin.any() else 0.0
