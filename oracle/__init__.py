"""CPU oracle for the W8A16 block-scaled GEMM (ctypes wrapper of w8a16_oracle.c).

TEST INFRASTRUCTURE ONLY. Only tests/, ``__graft_entry__.smoke()`` and bench.py's
CPU-baseline / reference leg may import this package. The product library under
``fp8_weight_only_gemm_gb300/`` never imports it, and this package imports
nothing from the product.

What it computes is the plain definition of the operation documented on the page
"metrale_model_layers/layers/ops/w8a16_gemm_pipelined_m32.rs" (doc comment of
``w8a16_gemm_pipelined_m32_strided``: A ``[M, a_row_stride]`` BF16 with the first
K columns read, W ``[N, K]`` FP8 E4M3, ``block_scale`` ``[N/128, K/128]`` FP32, C
``[M, c_row_stride]`` BF16 with the first N columns written; doc comment of
``W8A16_M32_K_BLOCK``: one scale block per 128-K step):

    C[m, n] = bf16_rne( sum_k A[m, k] * e4m3(W[n, k]) * scale[n // 128, k // 128] )

summed in FP64 in k order and rounded once. Pins (tests/test_oracle_pins.py):
all 256 E4M3 codes against the format's fixed points and an independent library
decode, BF16 rounding on ties / carries / subnormals / overflow, identity and
all-ones closed forms, brute force on tiny shapes, zero blocks, linearity, and
mutation tests showing each pin catches a planted mistake.
"""
from __future__ import annotations

import ctypes
import hashlib
import os
import platform
import subprocess
from pathlib import Path

import numpy as np

_HERE = Path(__file__).resolve().parent
_SRC = _HERE / "w8a16_oracle.c"
_BUILD = _HERE / "_build"

_u16p = ctypes.POINTER(ctypes.c_uint16)
_u8p = ctypes.POINTER(ctypes.c_uint8)
_f32p = ctypes.POINTER(ctypes.c_float)
_f64p = ctypes.POINTER(ctypes.c_double)


def _src_tag(source: bytes) -> str:
    h = hashlib.sha1(source).hexdigest()[:12]
    return f"{h}_{platform.machine()}"


def build(outdir: Path | None = None, source: str | None = None) -> Path:
    """Compile the oracle with gcc (no fast-math, no FP contraction) and return
    the path of the shared library.

    ``source`` replaces the text of w8a16_oracle.c; only the mutation tests pass
    one (a copy with one planted mistake, compiled into their own directory).
    """
    outdir = Path(outdir) if outdir is not None else _BUILD
    outdir.mkdir(parents=True, exist_ok=True)
    text = _SRC.read_bytes() if source is None else source.encode()
    lib = outdir / f"liboracle_w8a16_{_src_tag(text)}.so"
    if lib.exists():
        return lib
    src = _SRC
    if source is not None:
        src = outdir / f"w8a16_oracle_{_src_tag(text)}.c"
        src.write_bytes(text)
    tmp = lib.with_suffix(f".tmp{os.getpid()}.so")
    cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-ffp-contract=off",
           "-fno-fast-math", "-pthread", str(src), "-o", str(tmp), "-lm"]
    subprocess.run(cmd, check=True, capture_output=True)
    os.replace(tmp, lib)
    return lib


def source_text() -> str:
    """The oracle's C source."""
    return _SRC.read_text()


class Oracle:
    """One loaded build of the oracle."""

    def __init__(self, outdir: Path | None = None, source: str | None = None):
        self.path = build(outdir, source)
        lib = ctypes.CDLL(str(self.path))
        lib.oracle_e4m3_to_double.argtypes = [ctypes.c_uint8]
        lib.oracle_e4m3_to_double.restype = ctypes.c_double
        lib.oracle_bf16_to_double.argtypes = [ctypes.c_uint16]
        lib.oracle_bf16_to_double.restype = ctypes.c_double
        lib.oracle_double_to_bf16_rne.argtypes = [ctypes.c_double]
        lib.oracle_double_to_bf16_rne.restype = ctypes.c_uint16
        lib.oracle_w8a16_gemm.argtypes = [
            _u16p, ctypes.c_uint32, _u8p, _f32p, _u16p, ctypes.c_uint32,
            ctypes.c_uint32, ctypes.c_uint32, ctypes.c_uint32, _f64p, _f64p, ctypes.c_int]
        lib.oracle_w8a16_gemm.restype = ctypes.c_int
        lib.oracle_e4m3_encode_rne.argtypes = [ctypes.c_float]
        lib.oracle_e4m3_encode_rne.restype = ctypes.c_uint8
        lib.oracle_quantize_weights.argtypes = [_f32p, ctypes.c_uint32, ctypes.c_uint32,
                                                ctypes.c_uint32, _u8p, _f32p]
        lib.oracle_quantize_weights.restype = ctypes.c_int
        lib.oracle_quantize_activations.argtypes = [_u16p, ctypes.c_uint32, ctypes.c_uint32,
                                                    ctypes.c_uint32, _u8p, _f32p]
        lib.oracle_quantize_activations.restype = ctypes.c_int
        lib.oracle_w8a8_gemm.argtypes = [
            _u8p, ctypes.c_uint32, _f32p, _u8p, _f32p, _u16p, ctypes.c_uint32,
            ctypes.c_uint32, ctypes.c_uint32, ctypes.c_uint32, _f64p, _f64p, ctypes.c_int]
        lib.oracle_w8a8_gemm.restype = ctypes.c_int
        self.lib = lib

    # -- scalar codecs -----------------------------------------------------
    def e4m3_to_double(self, code: int) -> float:
        return self.lib.oracle_e4m3_to_double(int(code) & 0xFF)

    def bf16_to_double(self, code: int) -> float:
        return self.lib.oracle_bf16_to_double(int(code) & 0xFFFF)

    def bf16_rne(self, x: float) -> int:
        return int(self.lib.oracle_double_to_bf16_rne(float(x)))

    def e4m3_encode(self, x: float) -> int:
        """E4M3 code of the FP32 value x: nearest, ties to even, saturating."""
        return int(self.lib.oracle_e4m3_encode_rne(float(x)))

    # -- the weight block quantiser -----------------------------------------
    def quantize_weights(self, W, N, K, w_row_stride=None):
        """(codes uint8 [N, K], scales float32 [ceil(N/128), K/128]) of the FP32
        weights W (``N * w_row_stride`` elements)."""
        import numpy as np
        ld = K if w_row_stride is None else int(w_row_stride)
        W = np.ascontiguousarray(np.asarray(W, dtype=np.float32).reshape(-1))
        if W.size < N * ld:
            raise ValueError("W too small")
        codes = np.zeros(N * K, dtype=np.uint8)
        scales = np.zeros(((N + 127) // 128) * (K // 128), dtype=np.float32)
        rc = self.lib.oracle_quantize_weights(
            W.ctypes.data_as(_f32p), ld, N, K, codes.ctypes.data_as(_u8p),
            scales.ctypes.data_as(_f32p))
        if rc != 0:
            raise ValueError(f"oracle_quantize_weights rejected N={N} K={K} ld={ld}")
        return codes.reshape(N, K), scales.reshape((N + 127) // 128, K // 128)

    # -- the GEMM ----------------------------------------------------------
    def gemm(self, A, W, scale, M, N, K, a_row_stride=None, C=None, c_row_stride=None,
             threads=None, want_exact=False):
        """C[m, n] for all m < M, n < N.

        A: uint16 array of BF16 codes, ``M * a_row_stride`` elements (any shape).
        W: uint8 array of E4M3 codes, ``N * K`` elements. scale: float32,
        ``ceil(N/128) * K/128`` elements. C (optional): uint16 array of
        ``M * c_row_stride`` elements, updated in place (pad columns untouched).
        Returns (C as [M, c_row_stride] uint16, exact [M, N] f64 or None,
        absum [M, N] f64 or None).
        """
        a_row_stride = K if a_row_stride is None else int(a_row_stride)
        c_row_stride = N if c_row_stride is None else int(c_row_stride)
        A = np.ascontiguousarray(A, dtype=np.uint16).reshape(-1)
        W = np.ascontiguousarray(W, dtype=np.uint8).reshape(-1)
        scale = np.ascontiguousarray(scale, dtype=np.float32).reshape(-1)
        assert A.size >= (M - 1) * a_row_stride + K
        assert W.size == N * K
        assert scale.size == ((N + 127) // 128) * (K // 128)
        if C is None:
            C = np.zeros(M * c_row_stride, dtype=np.uint16)
        C = np.ascontiguousarray(C, dtype=np.uint16).reshape(-1).copy()
        assert C.size >= (M - 1) * c_row_stride + N
        exact = np.zeros(M * N, dtype=np.float64) if want_exact else None
        absum = np.zeros(M * N, dtype=np.float64) if want_exact else None
        rc = self.lib.oracle_w8a16_gemm(
            A.ctypes.data_as(_u16p), a_row_stride, W.ctypes.data_as(_u8p),
            scale.ctypes.data_as(_f32p), C.ctypes.data_as(_u16p), c_row_stride, M, N, K,
            exact.ctypes.data_as(_f64p) if exact is not None else None,
            absum.ctypes.data_as(_f64p) if absum is not None else None,
            int(threads or os.cpu_count() or 1))
        if rc != 0:
            raise ValueError(f"oracle rejected M={M} N={N} K={K} strides=({a_row_stride},{c_row_stride})")
        Cv = C.reshape(M, c_row_stride) if C.size == M * c_row_stride else C
        return (Cv,
                exact.reshape(M, N) if exact is not None else None,
                absum.reshape(M, N) if absum is not None else None)

    # -- W8A8: the activation quantiser and the FP8 x FP8 product ------------
    def quantize_activations(self, A, M, K, a_row_stride=None):
        """(codes uint8 [M, K], scales float32 [K/128, M]) of BF16 activations A
        (uint16 codes, ``M * a_row_stride`` elements)."""
        ld = K if a_row_stride is None else int(a_row_stride)
        A = np.ascontiguousarray(A, dtype=np.uint16).reshape(-1)
        assert A.size >= (M - 1) * ld + K
        codes = np.zeros(M * K, dtype=np.uint8)
        scales = np.zeros((K // 128) * M, dtype=np.float32)
        rc = self.lib.oracle_quantize_activations(A.ctypes.data_as(_u16p), ld, M, K,
                                                  codes.ctypes.data_as(_u8p),
                                                  scales.ctypes.data_as(_f32p))
        if rc != 0:
            raise ValueError(f"oracle_quantize_activations rejected M={M} K={K} ld={ld}")
        return codes.reshape(M, K), scales.reshape(K // 128, M)

    def w8a8_gemm(self, Aq, a_scale, W, scale, M, N, K, a_row_stride=None, C=None,
                  c_row_stride=None, threads=None, want_exact=False):
        """C[m, n] of the W8A8 product (see oracle_w8a8_gemm); same returns as gemm()."""
        a_row_stride = K if a_row_stride is None else int(a_row_stride)
        c_row_stride = N if c_row_stride is None else int(c_row_stride)
        Aq = np.ascontiguousarray(Aq, dtype=np.uint8).reshape(-1)
        a_scale = np.ascontiguousarray(a_scale, dtype=np.float32).reshape(-1)
        W = np.ascontiguousarray(W, dtype=np.uint8).reshape(-1)
        scale = np.ascontiguousarray(scale, dtype=np.float32).reshape(-1)
        assert Aq.size >= (M - 1) * a_row_stride + K and a_scale.size == (K // 128) * M
        assert W.size == N * K and scale.size == ((N + 127) // 128) * (K // 128)
        if C is None:
            C = np.zeros(M * c_row_stride, dtype=np.uint16)
        C = np.ascontiguousarray(C, dtype=np.uint16).reshape(-1).copy()
        exact = np.zeros(M * N, dtype=np.float64) if want_exact else None
        absum = np.zeros(M * N, dtype=np.float64) if want_exact else None
        rc = self.lib.oracle_w8a8_gemm(
            Aq.ctypes.data_as(_u8p), a_row_stride, a_scale.ctypes.data_as(_f32p),
            W.ctypes.data_as(_u8p), scale.ctypes.data_as(_f32p), C.ctypes.data_as(_u16p),
            c_row_stride, M, N, K,
            exact.ctypes.data_as(_f64p) if exact is not None else None,
            absum.ctypes.data_as(_f64p) if absum is not None else None,
            int(threads or os.cpu_count() or 1))
        if rc != 0:
            raise ValueError(f"oracle_w8a8_gemm rejected M={M} N={N} K={K}")
        Cv = C.reshape(M, c_row_stride) if C.size == M * c_row_stride else C
        return (Cv,
                exact.reshape(M, N) if exact is not None else None,
                absum.reshape(M, N) if absum is not None else None)


_DEFAULT: Oracle | None = None


def get() -> Oracle:
    """The unmutated oracle, built on first use."""
    global _DEFAULT
    if _DEFAULT is None:
        _DEFAULT = Oracle()
    return _DEFAULT
