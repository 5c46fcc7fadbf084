"""Seeded synthetic inputs for the W8A16 block-scaled GEMM.

This module is shared by the CUDA path's tests/bench and by the oracle's tests.
It holds none of the GEMM's arithmetic: it draws random numbers with torch's CPU
generator and encodes weights to FP8 E4M3 with torch's own ``float8_e4m3fn``
cast (round-to-nearest-even), after clamping to +-448 so the cast never
overflows. No value here comes from either the oracle or the CUDA library.

Weight format (page "metrale_model_layers/layers/ops/w8a16_gemm_pipelined_m32.rs",
doc comment of ``w8a16_gemm_pipelined_m32_strided``): W ``[N, K]`` E4M3 with one
FP32 ``block_scale`` per 128x128 block, grid ``[ceil(N/128), K/128]``. The block
quantiser used to make such weights: scale = amax(|w| over the block) / 448,
code = e4m3_rne(clamp(w / scale, -448, 448)); a block whose amax is 0 gets scale
0 and all-zero codes.

Recipe, in draw order from ``torch.Generator().manual_seed(seed)``:
  1. A ~ N(0, 1) in FP32 over the full pitch ``[M, a_row_stride]`` (pad columns
     are random too);
  2. W ~ N(0, w_std) in FP32, ``[N, K]``;
  3. extras: a fraction of A's elements (chosen by ``randperm``) multiplied by an
     outlier factor; optional per-block power-of-two spreads of W (drawn with
     ``randint``); listed zero blocks of W.
  Then A is rounded to BF16 (torch RNE) and W is block-quantised.
C is pre-filled: used region with the BF16 NaN 0xFFFF (catches unwritten
outputs), pad columns ``n >= N`` with 0x7FC0 (must stay untouched).
"""
from __future__ import annotations

from dataclasses import dataclass, field

import numpy as np
import torch

C_USED_SENTINEL = 0xFFFF
C_PAD_FILL = 0x7FC0
E4M3_MAX = 448.0


@dataclass(frozen=True)
class Workload:
    name: str
    M: int
    N: int
    K: int
    seed: int
    a_row_stride: int | None = None
    c_row_stride: int | None = None
    zero_blocks: tuple = ()          # ((nb, kb), ...) blocks of W forced to 0
    outlier_frac: float = 0.0        # fraction of A elements scaled by outlier_mult
    outlier_mult: float = 50.0
    w_std: float = 0.02
    block_spread: int = 0            # >0: each W block scaled by 2^U{-s..s}
    note: str = ""

    @property
    def lda(self) -> int:
        return self.a_row_stride or self.K

    @property
    def ldc(self) -> int:
        return self.c_row_stride or self.N

    def roofline_bytes(self) -> int:
        """N*K + 4*ceil(N/128)*(K/128) + 2*M*K + 2*M*N: W, scales, A and C once."""
        nb = (self.N + 127) // 128
        return self.N * self.K + 4 * nb * (self.K // 128) + 2 * self.M * self.K + 2 * self.M * self.N

    def flops(self) -> int:
        return 2 * self.M * self.N * self.K


# The five workloads the operation is measured on (decode GEMV, fused QKV, the
# strided multi-sequence tier, and a multi-tile prefill-sized call).
CONFIGS: dict[str, Workload] = {w.name: w for w in [
    Workload("tiny_m1_n256_k256", 1, 256, 256, seed=0, note="contiguous, scales [2,2]"),
    Workload("decode_gemv_m1_n4096_k4096", 1, 4096, 4096, seed=1,
             note="decode GEMV, contiguous, scales [32,32]"),
    Workload("skinny_qkv_m8_n12288_k4096", 8, 12288, 4096, seed=2, zero_blocks=((48, 16),),
             note="fused-QKV shape, one all-zero W block with scale 0"),
    Workload("strided_m32_n14336_k5120", 32, 14336, 5120, seed=3, a_row_stride=5184,
             c_row_stride=14400, note="a pitch 5184 (random pad), c pitch 14400 (pad 0x7FC0)"),
    Workload("multitile_m128_n28672_k8192", 128, 28672, 8192, seed=4, outlier_frac=0.01,
             outlier_mult=50.0, note="1% of A elements x50"),
]}
CONFIG_ORDER = list(CONFIGS)


def bf16_codes(t: torch.Tensor) -> np.ndarray:
    """uint16 numpy view of a BF16 tensor's bits."""
    return t.contiguous().view(torch.int16).numpy().view(np.uint16)


def block_quantize_e4m3(w: torch.Tensor, block: int = 128):
    """FP32 [N, K] -> (uint8 E4M3 codes [N, K], FP32 scales [ceil(N/128), K/128]).

    Processed one 128-row block-row at a time to bound host memory.
    """
    N, K = w.shape
    assert K % block == 0
    nb, kb = (N + block - 1) // block, K // block
    codes = torch.empty((N, K), dtype=torch.uint8)
    scales = torch.empty((nb, kb), dtype=torch.float32)
    for i in range(nb):
        rows = w[i * block:(i + 1) * block]
        r = rows.shape[0]
        blk = rows.reshape(r, kb, block)
        amax = blk.abs().amax(dim=(0, 2))                      # [kb]
        s = (amax / E4M3_MAX).to(torch.float32)
        safe = torch.where(s > 0, s, torch.ones_like(s))
        q = (blk / safe[None, :, None]).clamp(-E4M3_MAX, E4M3_MAX)
        c = q.to(torch.float8_e4m3fn).view(torch.uint8)
        c[:, s == 0, :] = 0
        codes[i * block:i * block + r] = c.reshape(r, K)
        scales[i] = s
    return codes, scales


@dataclass
class Case:
    wl: Workload
    A: torch.Tensor          # BF16 [M, lda]
    W: torch.Tensor          # uint8 [N, K] E4M3 codes
    scale: torch.Tensor      # FP32 [ceil(N/128), K/128]
    C0: torch.Tensor         # BF16 [M, ldc] pre-filled output
    extra: dict = field(default_factory=dict)

    # numpy views of the raw codes (what the oracle consumes)
    def A_np(self):
        return bf16_codes(self.A)

    def W_np(self):
        return self.W.numpy()

    def scale_np(self):
        return self.scale.numpy()

    def C0_np(self):
        return bf16_codes(self.C0)


def make_case(wl: Workload | str, **overrides) -> Case:
    if isinstance(wl, str):
        wl = CONFIGS[wl]
    if overrides:
        wl = Workload(**{**wl.__dict__, **overrides})
    M, N, K = wl.M, wl.N, wl.K
    lda, ldc = wl.lda, wl.ldc
    g = torch.Generator().manual_seed(wl.seed)
    a = torch.randn((M, lda), generator=g, dtype=torch.float32)
    w = torch.randn((N, K), generator=g, dtype=torch.float32) * wl.w_std
    if wl.outlier_frac > 0:
        cnt = int(round(wl.outlier_frac * M * lda))
        idx = torch.randperm(M * lda, generator=g)[:cnt]
        a.view(-1)[idx] *= wl.outlier_mult
    nb, kb = (N + 127) // 128, K // 128
    if wl.block_spread > 0:
        e = torch.randint(-wl.block_spread, wl.block_spread + 1, (nb, kb), generator=g)
        f = torch.pow(2.0, e.to(torch.float32))
        for i in range(nb):
            w[i * 128:(i + 1) * 128] *= f[i].repeat_interleave(128)[None, :]
    for (bn, bk) in wl.zero_blocks:
        w[bn * 128:(bn + 1) * 128, bk * 128:(bk + 1) * 128] = 0.0
    A = a.to(torch.bfloat16)
    W, scale = block_quantize_e4m3(w)
    C0 = torch.full((M, ldc), C_PAD_FILL, dtype=torch.int32).to(torch.int16)
    C0[:, :N] = np.int16(np.uint16(C_USED_SENTINEL).view(np.int16))
    C0 = C0.view(torch.bfloat16)
    return Case(wl, A, W, scale, C0)


def random_codes_case(M: int, N: int, K: int, seed: int, lda=None, ldc=None) -> Case:
    """Every E4M3 code (NaNs excluded) drawn uniformly, scales drawn log-uniform
    over 2^-8..2^8: exercises subnormal, max-magnitude and negative-zero codes."""
    lda = lda or K
    ldc = ldc or N
    g = torch.Generator().manual_seed(seed)
    A = torch.randn((M, lda), generator=g).to(torch.bfloat16)
    W = torch.randint(0, 256, (N, K), generator=g, dtype=torch.int32).to(torch.uint8)
    W[(W == 0x7F) | (W == 0xFF)] = 0x7E
    nb, kb = (N + 127) // 128, K // 128
    scale = torch.pow(2.0, torch.rand((nb, kb), generator=g) * 16 - 8).to(torch.float32)
    C0 = torch.full((M, ldc), C_PAD_FILL, dtype=torch.int32).to(torch.int16)
    C0[:, :N] = np.int16(np.uint16(C_USED_SENTINEL).view(np.int16))
    wl = Workload(f"random_codes_m{M}_n{N}_k{K}", M, N, K, seed, lda if lda != K else None,
                  ldc if ldc != N else None)
    return Case(wl, A, W, scale, C0.view(torch.bfloat16))
