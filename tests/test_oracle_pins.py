"""Pins that tie the CPU oracle to facts other than itself.

Each ``pin_*`` function takes a loaded oracle build and raises AssertionError on a
mismatch; the ``test_*`` wrappers run them on the real oracle and
tests/test_oracle_mutants.py runs them on builds with one planted mistake each,
to show every such mistake is caught by at least one pin.

What pins what:
  * E4M3 decode: the format's fixed points (tests/golden/format_fixed_points.json)
    and torch's independent float8_e4m3fn decode of all 256 codes;
  * BF16 rounding: hand-derived ties, carries, overflow and subnormal cases, and
    torch's binary32 -> bfloat16 cast on binary32 inputs (a single rounding);
  * the GEMM: a hand-worked example (tests/golden/hand_worked_k256_n130.json),
    identity and all-ones closed forms, exact brute force with rational
    arithmetic on tiny shapes, zero blocks, pad columns, linearity, sums on exact
    BF16 midpoints, NaN flow;
  * the quantisers and W8A8: torch restatements, each block's or group's maximum
    mapping to +-448, rational brute force, unit-code closed forms.
"""
from __future__ import annotations

import json
import math
from fractions import Fraction
from pathlib import Path

import numpy as np
import pytest
import torch

import workloads

GOLDEN = Path(__file__).resolve().parent / "golden"


# ---------------------------------------------------------------- helpers --
def _e4m3_torch(codes: np.ndarray) -> np.ndarray:
    t = torch.from_numpy(np.ascontiguousarray(codes, dtype=np.uint8))
    return t.view(torch.float8_e4m3fn).to(torch.float64).numpy()


def _bf16_value(code: int) -> float:
    return float(np.array([code << 16], dtype=np.uint32).view(np.float32)[0])


def _rne_bf16_exact(x: Fraction) -> int:
    """Exact round-to-nearest-even of a rational to BF16 bits, by rational
    arithmetic (an independent route from the oracle's frexp/nearbyint)."""
    if x == 0:
        return 0
    neg = x < 0
    a = -x if neg else x
    e = a.numerator.bit_length() - a.denominator.bit_length()
    if Fraction(2) ** e > a:
        e -= 1
    q = max(e - 7, -133)
    units = round(a / Fraction(2) ** q)       # Python rounds Fractions half-to-even
    v = units * Fraction(2) ** q
    if v >= Fraction(2) ** 128:
        bits = 0x7F80
    else:
        bits = int(np.array([float(v)], dtype=np.float32).view(np.uint32)[0] >> 16)
    return bits | (0x8000 if neg else 0)


def _rand_bf16(shape, gen, scale=1.0):
    return (torch.randn(shape, generator=gen) * scale).to(torch.bfloat16)


def _codes(t_bf16: torch.Tensor) -> np.ndarray:
    return t_bf16.contiguous().view(torch.int16).numpy().view(np.uint16)


def _brute_force(A_codes, W_codes, scale, M, N, K, lda):
    """Exact C by rational sums of exactly-representable terms."""
    a = A_codes.reshape(M, lda)[:, :K]
    af = a.astype(np.uint32) << 16
    af = af.view(np.float32).astype(np.float64)
    wf = _e4m3_torch(W_codes.reshape(N, K))
    s = scale.reshape((N + 127) // 128, K // 128).astype(np.float64)
    out = np.zeros((M, N), dtype=np.uint16)
    exact = np.zeros((M, N))
    for m in range(M):
        for n in range(N):
            srow = np.repeat(s[n // 128], 128)
            tot = sum((Fraction(float(af[m, k])) * Fraction(float(wf[n, k])) * Fraction(float(srow[k]))
                       for k in range(K)), Fraction(0))
            out[m, n] = _rne_bf16_exact(tot)
            exact[m, n] = float(tot)
    return out, exact


# ------------------------------------------------------------------- pins --
def pin_e4m3_fixed_points(o):
    g = json.loads((GOLDEN / "format_fixed_points.json").read_text())
    for row in g["e4m3"]:
        code = int(row["code"], 16)
        got = o.e4m3_to_double(code)
        if row["value"] == "nan":
            assert math.isnan(got), row
        else:
            assert got == row["value"], (row, got)
            assert math.copysign(1.0, got) == math.copysign(1.0, row["value"]), row


def pin_e4m3_all_codes_vs_torch(o):
    ref = _e4m3_torch(np.arange(256, dtype=np.uint8))
    got = np.array([o.e4m3_to_double(c) for c in range(256)])
    nan = np.isnan(ref)
    assert np.array_equal(nan, np.isnan(got))
    assert np.array_equal(ref[~nan], got[~nan])
    assert np.array_equal(np.signbit(ref[~nan]), np.signbit(got[~nan]))
    # strictly increasing over the non-negative finite codes
    pos = got[:0x7F]
    assert np.all(np.diff(pos) > 0)


def _parse_x(s: str) -> float:
    if s == "nan":
        return float("nan")
    return float(eval(s.replace("^", "**"), {"__builtins__": {}}))


def pin_bf16_fixed_points(o):
    g = json.loads((GOLDEN / "format_fixed_points.json").read_text())
    for row in g["bf16_rne"]:
        x = _parse_x(row["x"])
        assert o.bf16_rne(x) == int(row["bf16"], 16), (row, hex(o.bf16_rne(x)))


def pin_bf16_vs_torch_on_binary32(o):
    gen = torch.Generator().manual_seed(11)
    xs = torch.cat([
        torch.randn(4000, generator=gen) * 10.0 ** torch.randint(-30, 30, (4000,), generator=gen),
        torch.randn(1000, generator=gen) * 1e-39,                        # binary32 subnormals
        (torch.randint(-2 ** 20, 2 ** 20, (1000,), generator=gen) * 2.0 ** -14) + 0.5,
    ]).to(torch.float32)
    ref = xs.to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    got = np.array([o.bf16_rne(float(x)) for x in xs.tolist()], dtype=np.uint16)
    assert np.array_equal(ref, got)
    # BF16 -> double is the binary32 reading of the upper half
    for c in [0x0001, 0x3F80, 0xC020, 0x7F7F, 0x8000, 0x0080]:
        assert o.bf16_to_double(c) == _bf16_value(c)


def pin_hand_worked_example(o):
    g = json.loads((GOLDEN / "hand_worked_k256_n130.json").read_text())
    M, N, K, lda, ldc = g["M"], g["N"], g["K"], g["a_row_stride"], g["c_row_stride"]
    A = np.full((M, lda), 1e30, dtype=np.float32)
    for m in range(M):
        for k in range(K):
            A[m, k] = (1.0 if k % 2 == 0 else -0.5) * (1 if m == 0 else 2)
    A_codes = _codes(torch.from_numpy(A).to(torch.bfloat16))
    W = np.empty((N, K), dtype=np.uint8)
    W[:, :128] = 0x38
    W[:, 128:] = 0x40
    W[129, :] = 0xB0
    scale = np.array(g["inputs"]["scale"], dtype=np.float32)
    C0 = np.full((M, ldc), 0x7FC0, dtype=np.uint16)
    C, exact, _ = o.gemm(A_codes, W, scale, M, N, K, a_row_stride=lda, C=C0, c_row_stride=ldc,
                         want_exact=True)
    for e in g["expected"]:
        assert exact[e["m"], e["n"]] == e["value"], e
        assert C[e["m"], e["n"]] == int(e["bf16"], 16), (e, hex(C[e["m"], e["n"]]))
    assert np.all(C[:, N:] == 0x7FC0)


def pin_identity_weights(o):
    gen = torch.Generator().manual_seed(3)
    for (M, N, K) in [(3, 256, 256), (2, 200, 256)]:
        A = _codes(_rand_bf16((M, K), gen))
        W = np.zeros((N, K), dtype=np.uint8)
        for n in range(N):
            W[n, n] = 0x38                       # 1.0
        scale = np.ones(((N + 127) // 128, K // 128), dtype=np.float32)
        C, _, _ = o.gemm(A, W, scale, M, N, K)
        assert np.array_equal(C, A[:, :N]), "identity weights must reproduce A"


def pin_all_ones_closed_form(o):
    gen = torch.Generator().manual_seed(5)
    M, N, K = 3, 384, 512
    A_t = _rand_bf16((M, K), gen)
    A = _codes(A_t)
    W = np.full((N, K), 0x38, dtype=np.uint8)
    e = torch.randint(-6, 7, (3, 4), generator=gen).numpy()
    scale = (2.0 ** e).astype(np.float32)        # powers of two: every product exact
    _, exact, _ = o.gemm(A, W, scale, M, N, K, want_exact=True)
    a = A_t.to(torch.float64).numpy()
    bsum = a.reshape(M, K // 128, 128).sum(axis=2)  # exact in float64 for these values
    for n in [0, 127, 128, 255, 256, 383]:
        want = (bsum * scale[n // 128][None, :].astype(np.float64)).sum(axis=1)
        assert np.array_equal(exact[:, n], want), n


def pin_brute_force_tiny(o):
    gen = torch.Generator().manual_seed(7)
    for (M, N, K, lda) in [(1, 128, 128, 128), (3, 130, 256, 264), (2, 9, 384, 384),
                           (4, 257, 128, 136)]:
        A = _codes(_rand_bf16((M, lda), gen, scale=3.0))
        W = torch.randint(0, 256, (N, K), generator=gen, dtype=torch.int32).to(torch.uint8).numpy()
        W[(W == 0x7F) | (W == 0xFF)] = 0x01
        nb, kb = (N + 127) // 128, K // 128
        scale = (2.0 ** (torch.rand((nb, kb), generator=gen) * 12 - 6)).to(torch.float32).numpy()
        C, exact, absum = o.gemm(A, W, scale, M, N, K, a_row_stride=lda, want_exact=True)
        want, want_exact = _brute_force(A, W, scale, M, N, K, lda)
        assert np.array_equal(C, want), (M, N, K)
        assert np.all(np.abs(exact - want_exact) <= K * 2.0 ** -52 * absum)


def pin_zero_block(o):
    gen = torch.Generator().manual_seed(9)
    M, N, K = 2, 256, 384
    A = _codes(_rand_bf16((M, K), gen))
    W = torch.randint(0, 0x7E, (N, K), generator=gen, dtype=torch.int32).to(torch.uint8).numpy()
    scale = (torch.rand((2, 3), generator=gen) + 0.5).numpy().astype(np.float32)
    scale[1, 2] = 0.0
    W2 = W.copy()
    W2[128:256, 256:384] = 0                           # zero codes under the zero scale
    _, e1, _ = o.gemm(A, W, scale, M, N, K, want_exact=True)
    _, e2, _ = o.gemm(A, W2, scale, M, N, K, want_exact=True)
    assert np.array_equal(e1, e2)
    # dropping the block's K range for the affected rows gives the same sums
    A3 = A.reshape(M, K)[:, :256].copy()
    _, e3, _ = o.gemm(A3, W2[:, :256].copy(), scale[:, :2].copy(), M, N, 256, want_exact=True)
    assert np.array_equal(e1[:, 128:], e3[:, 128:])


def pin_pads_untouched_and_ignored(o):
    gen = torch.Generator().manual_seed(13)
    M, N, K, lda, ldc = 3, 130, 256, 272, 140
    A_full = _codes(_rand_bf16((M, lda), gen))
    A_full[:, K:] = 0x7FC0                      # NaN in A's pad must not be read
    W = torch.randint(0, 0x7E, (N, K), generator=gen, dtype=torch.int32).to(torch.uint8).numpy()
    scale = np.ones((2, 2), dtype=np.float32)
    C0 = np.full((M, ldc), 0x1234, dtype=np.uint16)
    C, _, _ = o.gemm(A_full, W, scale, M, N, K, a_row_stride=lda, C=C0, c_row_stride=ldc)
    assert np.all(C[:, N:] == 0x1234)
    Cc, _, _ = o.gemm(np.ascontiguousarray(A_full[:, :K]), W, scale, M, N, K)
    assert np.array_equal(C[:, :N], Cc)


def pin_linearity(o):
    gen = torch.Generator().manual_seed(17)
    M, N, K = 2, 160, 256
    A = _codes(_rand_bf16((M, K), gen))
    W = torch.randint(0, 0x7E, (N, K), generator=gen, dtype=torch.int32).to(torch.uint8).numpy()
    scale = (torch.rand((2, 2), generator=gen) + 0.1).numpy().astype(np.float32)
    _, e1, ab = o.gemm(A, W, scale, M, N, K, want_exact=True)
    _, e2, _ = o.gemm(A, W, scale * 2, M, N, K, want_exact=True)
    assert np.array_equal(e2, 2 * e1)
    # the same permutation of K inside each block, applied to A and W
    perm = np.concatenate([b * 128 + np.random.default_rng(1).permutation(128) for b in range(2)])
    _, e3, _ = o.gemm(np.ascontiguousarray(A.reshape(M, K)[:, perm]),
                      np.ascontiguousarray(W[:, perm]), scale, M, N, K, want_exact=True)
    assert np.all(np.abs(e3 - e1) <= K * 2.0 ** -52 * ab)


def pin_output_rounding_ties(o):
    """Sums that land exactly on a midpoint between two BF16 neighbours round to the
    one with an even last bit: 1 + 2^-8 lies halfway between 1 and 1 + 2^-7 (-> 1),
    1 + 3*2^-8 halfway between 1 + 2^-7 and 1 + 2^-6 (-> 1 + 2^-6); the same with
    the sign flipped. Closed forms of round-to-nearest-even on the GEMM's output."""
    M, N, K = 4, 128, 128
    A = np.zeros((M, K), dtype=np.float32)
    A[0, :2] = [1.0, 2.0 ** -8]
    A[1, :2] = [1.0, 3 * 2.0 ** -8]
    A[2, :2] = [-1.0, -(2.0 ** -8)]
    A[3, :2] = [-1.0, -3 * 2.0 ** -8]
    W = np.full((N, K), 0x38, dtype=np.uint8)                 # every weight 1.0
    C, _, _ = o.gemm(_codes(torch.from_numpy(A).to(torch.bfloat16)), W,
                     np.ones((1, 1), np.float32), M, N, K)
    want = [0x3F80, 0x3F82, 0xBF80, 0xBF82]                     # 1, 1 + 2^-6, -1, -(1 + 2^-6)
    for m in range(M):
        assert np.all(C[m] == want[m]), (m, hex(int(C[m, 0])))


def pin_nan_propagation(o):
    gen = torch.Generator().manual_seed(19)
    M, N, K = 2, 128, 128
    A = _codes(_rand_bf16((M, K), gen))
    W = np.full((N, K), 0x38, dtype=np.uint8)
    W[7, 100] = 0x7F
    C, _, _ = o.gemm(A, W, np.ones((1, 1), np.float32), M, N, K)
    isnan = (C & 0x7F80) == 0x7F80
    isnan &= (C & 0x007F) != 0
    assert isnan[:, 7].all() and isnan.sum() == M


# ---- weight block quantiser pins ------------------------------------------

def pin_e4m3_encode_round_trip(o):
    """Every finite code encodes back to itself (the encoder inverts the decoder)."""
    for c in range(256):
        if (c & 0x7F) == 0x7F:
            continue
        assert o.e4m3_encode(o.e4m3_to_double(c)) == c, hex(c)
    assert o.e4m3_encode(float("nan")) & 0x7F == 0x7F
    assert o.e4m3_encode(1e6) == 0x7E and o.e4m3_encode(-1e6) == 0xFE   # saturation


def pin_e4m3_encode_ties_vs_torch(o):
    """Exact midpoints between neighbouring codes round to the even code, and
    random values round as torch's float8_e4m3fn cast (an independent encoder)."""
    vals = []
    for c in range(0x7E):
        a, b = o.e4m3_to_double(c), o.e4m3_to_double(c + 1)
        vals += [(a + b) / 2, -(a + b) / 2, a + (b - a) / 3, b - (b - a) / 5]
    g = torch.Generator().manual_seed(31)
    vals += (torch.randn(20000, generator=g) * 64).tolist()
    x = torch.tensor(vals, dtype=torch.float32)
    ref = x.clamp(-448, 448).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    got = np.array([o.e4m3_encode(float(v)) for v in x.numpy()], dtype=np.uint8)
    assert np.array_equal(ref, got), int((ref != got).sum())
    for c in range(0x7E):   # the tie itself: even mantissa wins
        mid = (o.e4m3_to_double(c) + o.e4m3_to_double(c + 1)) / 2
        if float(np.float32(mid)) == mid:
            assert o.e4m3_encode(mid) == (c if c % 2 == 0 else c + 1), hex(c)


def pin_quantizer_vs_recipe(o):
    """Blocks, ragged N, a zero block and a row pitch: the oracle quantiser equals
    the input recipe's torch implementation code for code and scale for scale."""
    g = torch.Generator().manual_seed(32)
    N, K, ld = 300, 384, 400
    w = torch.randn(N, ld, generator=g) * 0.02
    w[128:256, 128:256] = 0.0                                   # one zero block
    w[5, 7] = 3.0                                               # an outlier
    codes, scales = o.quantize_weights(w.numpy(), N, K, w_row_stride=ld)
    rc, rs = workloads.block_quantize_e4m3(w[:, :K].contiguous())
    assert np.array_equal(codes, rc.numpy())
    assert np.array_equal(scales, rs.numpy())
    assert scales[1, 1] == 0.0 and not codes[128:256, 128:256].any()


def pin_quantizer_block_maximum(o):
    """The largest |w| of a block encodes as +-448 and dequantises within one E4M3
    step of the original: a closed form of scale = amax / 448."""
    g = torch.Generator().manual_seed(33)
    w = torch.randn(256, 256, generator=g)
    codes, scales = o.quantize_weights(w.numpy(), 256, 256)
    for nb in range(2):
        for kb in range(2):
            blk = w[nb * 128:(nb + 1) * 128, kb * 128:(kb + 1) * 128]
            amax = float(blk.abs().max())
            assert scales[nb, kb] == np.float32(np.float32(amax) / np.float32(448.0))
            r, c = divmod(int(blk.abs().argmax()), 128)
            assert codes[nb * 128 + r, kb * 128 + c] & 0x7F == 0x7E
            deq = np.array([o.e4m3_to_double(int(x)) for x in
                            codes[nb * 128:(nb + 1) * 128, kb * 128].tolist()]) * scales[nb, kb]
            step = 2.0 ** np.floor(np.log2(np.maximum(np.abs(blk[:, 0].numpy()), 1e-30))) / 8
            assert np.all(np.abs(deq - blk[:, 0].numpy()) <= np.maximum(step, 2.0 ** -9 * scales[nb, kb]))


# ---- W8A8 pins (activation quantiser and FP8 x FP8 product) ----------------

def _torch_act_quant(a_bf16: torch.Tensor):
    """Independent torch statement of the per-token 128-group quantiser."""
    M, K = a_bf16.shape
    x = a_bf16.float().reshape(M, K // 128, 128)
    amax = x.abs().amax(dim=2)
    s = amax / 448.0
    safe = torch.where(s > 0, s, torch.ones_like(s))
    c = (x / safe[:, :, None]).clamp(-448, 448).to(torch.float8_e4m3fn).view(torch.uint8)
    c[s == 0] = 0
    return c.reshape(M, K).numpy(), s.t().contiguous().numpy()


def pin_act_quantizer_vs_torch(o):
    g = torch.Generator().manual_seed(41)
    M, K, ld = 5, 512, 520
    a = (torch.randn(M, ld, generator=g) * 3).to(torch.bfloat16)
    a[2, 128:256] = 0                                           # a zero group
    codes, scales = o.quantize_activations(_codes(a), M, K, a_row_stride=ld)
    rc, rs = _torch_act_quant(a[:, :K])
    assert np.array_equal(codes, rc) and np.array_equal(scales, rs)
    assert scales[1, 2] == 0 and not codes[2, 128:256].any()


def pin_act_quantizer_group_maximum(o):
    """Each (token, 128-group) gets its own scale fl32(amax) / 448 and its largest
    |a| encodes as +-448, while groups with a much smaller maximum keep their own
    finer scale (a closed form of the per-group rule)."""
    g = torch.Generator().manual_seed(44)
    M, K = 3, 384
    a = torch.randn(M, K, generator=g)
    a[:, 128:256] *= 1e-3                                       # a quiet middle group
    a[1, 300] = 50.0                                            # a loud entry in the last group
    a = a.to(torch.bfloat16)
    codes, scales = o.quantize_activations(_codes(a), M, K)
    af = a.float()
    for m in range(M):
        for gi in range(K // 128):
            grp = af[m, gi * 128:(gi + 1) * 128]
            amax = float(grp.abs().max())
            assert scales[gi, m] == np.float32(np.float32(amax) / np.float32(448.0)), (m, gi)
            j = int(grp.abs().argmax())
            assert codes[m, gi * 128 + j] & 0x7F == 0x7E, (m, gi)
    assert np.all(scales[1] < 1e-2 * scales[0])                # the quiet group's own scale


def pin_w8a8_reduces_to_w8a16(o):
    """With unit activation scales the W8A8 product is the W8A16 product of the
    activations' E4M3 values (exact in BF16), bit for bit."""
    g = torch.Generator().manual_seed(42)
    M, N, K = 3, 200, 256
    aq = torch.randint(0, 256, (M, K), generator=g, dtype=torch.uint8)
    aq[(aq & 0x7F) == 0x7F] = 0x38                              # no NaN codes
    w = torch.randn(N, K, generator=g) * 0.05
    wc, ws = workloads.block_quantize_e4m3(w)
    ones = np.ones((K // 128, M), dtype=np.float32)
    c8, _, _ = o.w8a8_gemm(aq.numpy(), ones, wc.numpy(), ws.numpy(), M, N, K)
    vals = _e4m3_torch(aq.numpy().reshape(-1)).reshape(M, K)
    a16 = _codes(torch.from_numpy(vals.astype(np.float32)).to(torch.bfloat16))
    c16, _, _ = o.gemm(a16, wc.numpy(), ws.numpy(), M, N, K)
    assert np.array_equal(c8, c16)


def pin_w8a8_brute_force_tiny(o):
    """Exact rational sums on tiny shapes with random group and block scales."""
    g = torch.Generator().manual_seed(43)
    M, N, K = 2, 130, 256
    aq = torch.randint(0, 0x7E, (M, K), generator=g, dtype=torch.uint8)
    wq = torch.randint(0, 0x7E, (N, K), generator=g, dtype=torch.uint8)
    sa = (torch.rand(K // 128, M, generator=g) + 0.5).numpy().astype(np.float32)
    sw = (torch.rand((N + 127) // 128, K // 128, generator=g) + 0.5).numpy().astype(np.float32)
    sign = torch.randint(0, 2, (M, K), generator=g, dtype=torch.uint8) << 7
    aq = aq | sign
    got, _, _ = o.w8a8_gemm(aq.numpy(), sa, wq.numpy(), sw, M, N, K)
    av = _e4m3_torch(aq.numpy().reshape(-1)).reshape(M, K)
    wv = _e4m3_torch(wq.numpy().reshape(-1)).reshape(N, K)
    for m in range(M):
        for n in (0, 1, 127, 128, 129):
            tot = Fraction(0)
            for k in range(K):
                tot += (Fraction(float(av[m, k])) * Fraction(float(sa[k // 128, m]))) * \
                       (Fraction(float(wv[n, k])) * Fraction(float(sw[n // 128, k // 128])))
            assert got[m, n] == _rne_bf16_exact(tot), (m, n)


def pin_w8a8_scales_closed_form(o):
    """With every code 1.0, the W8A8 output is sum over K groups of 128 * a_scale *
    w_scale; powers of two keep every term and sum exact, so the value is known in
    closed form and each activation scale must enter exactly once."""
    g = torch.Generator().manual_seed(45)
    M, N, K = 3, 256, 512
    aq = np.full((M, K), 0x38, dtype=np.uint8)
    wq = np.full((N, K), 0x38, dtype=np.uint8)
    sa = (2.0 ** torch.randint(-4, 5, (K // 128, M), generator=g)).numpy().astype(np.float32)
    sw = (2.0 ** torch.randint(-4, 5, (N // 128, K // 128), generator=g)).numpy().astype(np.float32)
    _, exact, _ = o.w8a8_gemm(aq, sa, wq, sw, M, N, K, want_exact=True)
    for m in range(M):
        for n in (0, 127, 128, 255):
            want = sum(128.0 * float(sa[kb, m]) * float(sw[n // 128, kb]) for kb in range(K // 128))
            assert exact[m, n] == want, (m, n)


PINS = [pin_e4m3_fixed_points, pin_e4m3_all_codes_vs_torch, pin_bf16_fixed_points,
        pin_bf16_vs_torch_on_binary32, pin_hand_worked_example, pin_identity_weights,
        pin_all_ones_closed_form, pin_brute_force_tiny, pin_zero_block,
        pin_pads_untouched_and_ignored, pin_linearity, pin_output_rounding_ties,
        pin_nan_propagation,
        pin_e4m3_encode_round_trip, pin_e4m3_encode_ties_vs_torch, pin_quantizer_vs_recipe,
        pin_quantizer_block_maximum,
        pin_act_quantizer_vs_torch, pin_act_quantizer_group_maximum, pin_w8a8_reduces_to_w8a16,
        pin_w8a8_brute_force_tiny, pin_w8a8_scales_closed_form]


@pytest.mark.parametrize("pin", PINS, ids=[p.__name__ for p in PINS])
def test_pin(pin, oracle_lib):
    pin(oracle_lib)
