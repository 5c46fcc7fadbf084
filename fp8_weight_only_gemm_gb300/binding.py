"""ctypes binding of libw8a16.so: argument marshalling only.

Every step of the operation runs in the library's CUDA kernels; this module only
turns torch tensors into pointers, pitches and a stream handle, and turns the
library's error codes into exceptions. There is no fallback: if the library is
not built or not loadable, every call raises.
"""
from __future__ import annotations

import ctypes
import re
from pathlib import Path

PKG = Path(__file__).resolve().parent
LIB_PATH = PKG / "_build" / "libw8a16.so"
HEADER = PKG.parent / "include" / "w8a16.h"

# Values mirrored from include/w8a16.h (checked against the header by the tests).
W8A16_OK = 0
FLAG_PDL = 1
VARIANT_AUTO, VARIANT_SIMT, VARIANT_TC, VARIANT_TC8, VARIANT_W8A8, VARIANT_PRESPLIT, VARIANT_GEMV = (
    0, 1, 2, 3, 4, 5, 6)
VARIANT_STREAM = 7
STATUS_OK, STATUS_WAIT_TIMEOUT = 0, 1
WEIGHTS_F32, WEIGHTS_BF16 = 0, 1


class Plan(ctypes.Structure):
    _fields_ = [("variant", ctypes.c_int32), ("token_tile", ctypes.c_uint32),
                ("split_k", ctypes.c_uint32), ("stages", ctypes.c_uint32),
                ("ctas_per_sm", ctypes.c_uint32), ("grid", ctypes.c_uint32 * 3),
                ("block", ctypes.c_uint32 * 3), ("cluster", ctypes.c_uint32 * 3),
                ("smem_bytes", ctypes.c_uint32), ("tmem_cols", ctypes.c_uint32),
                ("tail_tiles", ctypes.c_uint32), ("tail_split", ctypes.c_uint32)]

    def as_dict(self) -> dict:
        return {"variant": self.variant, "token_tile": self.token_tile, "split_k": self.split_k,
                "stages": self.stages, "ctas_per_sm": self.ctas_per_sm, "grid": list(self.grid),
                "block": list(self.block), "cluster": list(self.cluster),
                "smem_bytes": self.smem_bytes, "tmem_cols": self.tmem_cols,
                "tail_tiles": self.tail_tiles, "tail_split": self.tail_split}


class W8A16Error(RuntimeError):
    def __init__(self, code: int, message: str):
        super().__init__(f"w8a16 error {code}: {message}")
        self.code = code


_VP, _U32, _I32, _INT = ctypes.c_void_p, ctypes.c_uint32, ctypes.c_int32, ctypes.c_int
_U64 = ctypes.c_uint64
_SIGS = {
    "w8a16_gemm": (_INT, [_VP, _U32, _VP, _VP, _VP, _U32, _U32, _U32, _U32, _VP]),
    "w8a16_gemm_contiguous": (_INT, [_VP, _VP, _VP, _VP, _U32, _U32, _U32, _VP]),
    "w8a16_gemm_ex": (_INT, [_VP, _U32, _VP, _VP, _VP, _U32, _U32, _U32, _U32, _U32, _VP]),
    "w8a16_gemm_host": (_INT, [_VP, _U32, _VP, _VP, _VP, _U32, _U32, _U32, _U32, _VP, _VP, _VP,
                               _VP, _INT, _VP]),
    "w8a16_check_args": (_INT, [_VP, _U32, _VP, _VP, _VP, _U32, _U32, _U32, _U32]),
    "w8a16_plan_for": (_INT, [_U32, _U32, _U32, _U32, ctypes.POINTER(_U32), ctypes.POINTER(Plan)]),
    "w8a16_plan_current": (_INT, [_U32, _U32, _U32, ctypes.POINTER(Plan)]),
    "w8a16_cluster_capacity": (_INT, [_I32, _U32, _U32, ctypes.POINTER(_U32)]),
    "w8a16_plan_variant": (_INT, [_U32, _U32, _U32, _I32, _U32, _U32, _U32, ctypes.POINTER(Plan)]),
    "w8a16_gemm_with_plan": (_INT, [_VP, _U32, _VP, _VP, _VP, _U32, _U32, _U32, _U32,
                                    ctypes.POINTER(Plan), _U32, _VP]),
    "w8a16_quantize_weights": (_INT, [_VP, _U32, _U32, _U32, _U32, _VP, _VP, _VP]),
    "w8a16_quantize_activations": (_INT, [_VP, _U32, _U32, _U32, _VP, _VP, _U32, _VP]),
    "w8a16_workspace_bytes": (_U64, [_U32, _U32]),
    "w8a16_workspace_bytes_for": (_U64, [_U32, _U32, _U32]),
    "w8a16_plan_ws": (_INT, [_U32, _U32, _U32, _U64, ctypes.POINTER(Plan)]),
    "w8a16_gemm_noalloc": (_INT, [_VP, _U32, _VP, _VP, _VP, _U32, _U32, _U32, _U32, _U32, _VP]),
    "w8a16_noalloc_scratch_bytes": (_U64, []),
    "w8a16_split_activations": (_INT, [_VP, _U32, _U32, _U32, _VP, _U64, _VP]),
    "w8a16_gemm_split_terms": (_INT, [_VP, _U64, _VP, _VP, _VP, _U32, _U32, _U32, _U32, _U32, _VP]),
    "w8a16_gemm_ws": (_INT, [_VP, _U32, _VP, _VP, _VP, _U32, _U32, _U32, _U32, ctypes.POINTER(Plan), _VP,
                             _U64, _U32, _VP]),
    "w8a16_gemm_w8a8": (_INT, [_VP, _U32, _VP, _U32, _VP, _VP, _VP, _U32, _U32, _U32, _U32, _U32,
                               _VP]),
    "w8a16_gemm_w8a8_with_plan": (_INT, [_VP, _U32, _VP, _U32, _VP, _VP, _VP, _U32, _U32, _U32,
                                         _U32, ctypes.POINTER(Plan), _U32, _VP]),
    "w8a16_last_error": (ctypes.c_char_p, []),
    "w8a16_strerror": (ctypes.c_char_p, [_INT]),
    "w8a16_device_status": (_INT, [_VP, _INT, ctypes.POINTER(_U32), ctypes.POINTER(_U32),
                                   ctypes.POINTER(_U32)]),
    "w8a16_selftest_wait_timeout": (_INT, [_U32, _VP]),
    "w8a16_version": (ctypes.c_char_p, []),
}

_lib = None


def header_functions() -> list[str]:
    """Names of the functions include/w8a16.h declares."""
    text = HEADER.read_text()
    return sorted(set(re.findall(r"W8A16_API\s+(?:int|uint64_t|const char \*)\s*(w8a16_\w+)\s*\(", text)))


def load(path: Path | str | None = None):
    """Load the library (once). Raises if it has not been built."""
    global _lib
    if _lib is not None and path is None:
        return _lib
    p = Path(path) if path else LIB_PATH
    if not p.exists():
        raise RuntimeError(f"{p} is missing: build it first (python -m fp8_weight_only_gemm_gb300.build "
                           "or __graft_entry__.build()); there is no fallback path")
    lib = ctypes.CDLL(str(p))
    for name, (res, args) in _SIGS.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    if path is None:
        _lib = lib
    return lib


def last_error() -> str:
    return load().w8a16_last_error().decode()


def strerror(code: int) -> str:
    return load().w8a16_strerror(code).decode()


def _check(rc: int):
    if rc != W8A16_OK:
        raise W8A16Error(rc, last_error() or strerror(rc))


def _stream_handle(stream) -> int | None:
    import torch
    if stream is None:
        stream = torch.cuda.current_stream()
    return int(stream.cuda_stream) if hasattr(stream, "cuda_stream") else int(stream)


# -------------------------------------------------------------- pure host --
def check_args(M, N, K, a_row_stride, c_row_stride, A=0, W=0, scale=0, C=0) -> int:
    return load().w8a16_check_args(A or None, a_row_stride, W or None, scale or None, C or None,
                                   c_row_stride, M, N, K)


def plan_for(M, N, K, sm_count=152, cluster_ctas=None) -> dict:
    """Pure planner. cluster_ctas: optional 17-entry table (index = cluster size)
    of co-resident CTAs, as cluster_capacity() reports for a device."""
    p = Plan()
    tab = None
    if cluster_ctas is not None:
        tab = (_U32 * 17)(*[int(x) for x in cluster_ctas])
    _check(load().w8a16_plan_for(M, N, K, sm_count, tab, ctypes.byref(p)))
    return p.as_dict()


def plan_current(M, N, K) -> dict:
    """The plan w8a16_gemm uses on the current device."""
    p = Plan()
    _check(load().w8a16_plan_current(M, N, K, ctypes.byref(p)))
    return p.as_dict()


def plan_ws(M, N, K, workspace_bytes) -> dict:
    """The plan gemm_ws takes with a workspace of that many bytes (plan=None) on the
    current device."""
    p = Plan()
    _check(load().w8a16_plan_ws(M, N, K, workspace_bytes, ctypes.byref(p)))
    return p.as_dict()


def cluster_capacity(token_tile, stages, variant=VARIANT_TC) -> list[int]:
    out = (_U32 * 17)()
    _check(load().w8a16_cluster_capacity(variant, token_tile, stages, out))
    return list(out)


def plan_variant(M, N, K, variant=VARIANT_TC, split_k=0, stages=0, sm_count=152) -> Plan:
    p = Plan()
    _check(load().w8a16_plan_variant(M, N, K, variant, split_k, stages, sm_count, ctypes.byref(p)))
    return p


# ----------------------------------------------------------- device calls --
# The library sees plain pointers and cannot tell host memory, another device's
# memory or a short buffer from a good one; a kernel handed any of them would
# fault. So every tensor entry point checks placement, dtypes and extents here,
# before it calls the library.
_CODE_DTYPES = ("uint8", "float8_e4m3fn")


def _on_one_gpu(*tensors):
    dev = tensors[0].device
    for t in tensors:
        if not t.is_cuda:
            raise ValueError("all tensors must be on a CUDA device")
        if t.device != dev:
            raise ValueError(f"all tensors must be on one device (got {dev} and {t.device})")


def _scale_shape(scale, N, K, name="block_scale"):
    """Block scales cover the [N, K] weights: [ceil(N/128), K/128]. Checked when K
    is a multiple of 128; otherwise the library reports K itself."""
    want = ((N + 127) // 128, K // 128)
    if K % 128 == 0 and tuple(scale.shape) != want:
        raise ValueError(f"{name} must be {list(want)} for N={N}, K={K}; got {list(scale.shape)}")


def _is_codes(t) -> bool:
    return str(t.dtype).rsplit(".", 1)[-1] in _CODE_DTYPES


def _shapes(A, W, scale, C):
    import torch
    if A.dim() != 2 or W.dim() != 2:
        raise ValueError("A and W must be 2-D")
    if A.dtype != torch.bfloat16:
        raise TypeError(f"A must be bfloat16, got {A.dtype}")
    if W.dtype not in (torch.uint8, torch.float8_e4m3fn):
        raise TypeError(f"W must be uint8 E4M3 codes or float8_e4m3fn, got {W.dtype}")
    if scale.dtype != torch.float32:
        raise TypeError(f"block_scale must be float32, got {scale.dtype}")
    if A.stride(1) != 1 or (C is not None and C.stride(1) != 1):
        raise ValueError("A and C rows must be contiguous (stride 1 along K / N)")
    if not W.is_contiguous() or not scale.is_contiguous():
        raise ValueError("W and block_scale must be contiguous")
    M, K = A.shape
    N, Kw = W.shape
    if Kw != K:
        raise ValueError(f"A has K={K} columns, W has {Kw}")
    _scale_shape(scale, N, K)
    return M, N, K


def gemm(A, W, scale, C=None, *, stream=None, plan: Plan | None = None, flags: int = 0):
    """C[:, :N] = A @ dequant(W)^T on the GPU. A: bf16 [M, K] (any row pitch, rows
    contiguous); W: uint8/float8_e4m3fn [N, K]; scale: fp32 [ceil(N/128), K/128];
    C: optional bf16 [M, >=N] output view (allocated [M, N] if None)."""
    import torch
    M, N, K = _shapes(A, W, scale, C)
    if C is None:
        C = torch.empty((M, N), dtype=torch.bfloat16, device=A.device)
    if C.dtype != torch.bfloat16 or C.shape[0] != M or C.shape[1] < N:
        raise ValueError("C must be bfloat16 [M, >=N]")
    _on_one_gpu(A, W, scale, C)
    lib = load()
    args = (A.data_ptr(), A.stride(0), W.data_ptr(), scale.data_ptr(), C.data_ptr(), C.stride(0),
            M, N, K)
    with torch.cuda.device(A.device):
        s = _stream_handle(stream)
        if plan is None:
            rc = lib.w8a16_gemm_ex(*args, flags, s)
        else:
            rc = lib.w8a16_gemm_with_plan(*args, ctypes.byref(plan), flags, s)
    _check(rc)
    return C


def workspace_bytes(M: int, K: int) -> int:
    """Workspace bytes of the pre-split path of gemm_ws at (M, K)."""
    return int(load().w8a16_workspace_bytes(M, K))


def workspace_bytes_for(M: int, N: int, K: int) -> int:
    """Workspace bytes with which gemm_ws takes its fastest plan at (M, N, K) on the
    current device."""
    return int(load().w8a16_workspace_bytes_for(M, N, K))


def gemm_ws(A, W, scale, C=None, *, workspace=None, stream=None, plan: Plan | None = None,
            flags: int = 0):
    """gemm() through w8a16_gemm_ws. workspace: a CUDA uint8 tensor, 16-byte aligned
    (workspace_bytes_for(M, N, K) bytes give the fastest plan; workspace_bytes(M, K)
    the pre-split plan above 16 tokens); None allocates one of the larger of the two
    with torch for this call (a caller that repeats calls should keep one); False
    passes none."""
    import torch
    M, N, K = _shapes(A, W, scale, C)
    if C is None:
        C = torch.empty((M, N), dtype=torch.bfloat16, device=A.device)
    if C.dtype != torch.bfloat16 or C.shape[0] != M or C.shape[1] < N:
        raise ValueError("C must be bfloat16 [M, >=N]")
    _on_one_gpu(A, W, scale, C)
    if workspace is not None and workspace is not False:
        if workspace.dtype != torch.uint8 or not workspace.is_contiguous():
            raise ValueError("workspace must be a contiguous uint8 tensor")
        _on_one_gpu(A, workspace)
    lib = load()
    if workspace is None:
        with torch.cuda.device(A.device):
            need = max(workspace_bytes_for(M, N, K), workspace_bytes(M, K))
        workspace = torch.empty(max(16, need), dtype=torch.uint8, device=A.device)
    ws_ptr, ws_bytes = (None, 0) if workspace is False else (workspace.data_ptr(), workspace.numel())
    with torch.cuda.device(A.device):
        rc = lib.w8a16_gemm_ws(A.data_ptr(), A.stride(0), W.data_ptr(), scale.data_ptr(), C.data_ptr(),
                               C.stride(0), M, N, K, ctypes.byref(plan) if plan is not None else None,
                               ws_ptr, ws_bytes, flags, _stream_handle(stream))
    _check(rc)
    return C


def gemm_noalloc(A, W, scale, C=None, *, stream=None, flags: int = 0):
    """gemm() through w8a16_gemm_noalloc (the library's fixed scratch buffer; calls
    must not overlap in time)."""
    import torch
    M, N, K = _shapes(A, W, scale, C)
    if C is None:
        C = torch.empty((M, N), dtype=torch.bfloat16, device=A.device)
    if C.dtype != torch.bfloat16 or C.shape[0] != M or C.shape[1] < N:
        raise ValueError("C must be bfloat16 [M, >=N]")
    _on_one_gpu(A, W, scale, C)
    with torch.cuda.device(A.device):
        rc = load().w8a16_gemm_noalloc(A.data_ptr(), A.stride(0), W.data_ptr(), scale.data_ptr(),
                                       C.data_ptr(), C.stride(0), M, N, K, flags, _stream_handle(stream))
    _check(rc)
    return C


def gemm_noalloc_ptr(A_ptr, a_row_stride, W_ptr, scale_ptr, C_ptr, c_row_stride, M, N, K, stream=0,
                     flags: int = 0) -> int:
    """Raw-pointer w8a16_gemm_noalloc (returns the library's code; does not raise)."""
    return load().w8a16_gemm_noalloc(A_ptr or None, a_row_stride, W_ptr or None, scale_ptr or None,
                                     C_ptr or None, c_row_stride, M, N, K, flags, stream or None)


def noalloc_scratch_bytes() -> int:
    return int(load().w8a16_noalloc_scratch_bytes())


def gemm_ws_ptr(A_ptr, a_row_stride, W_ptr, scale_ptr, C_ptr, c_row_stride, M, N, K, ws_ptr, ws_bytes,
                stream=0, plan: Plan | None = None, flags: int = 0) -> int:
    """Raw-pointer w8a16_gemm_ws (returns the library's code; does not raise)."""
    return load().w8a16_gemm_ws(A_ptr or None, a_row_stride, W_ptr or None, scale_ptr or None, C_ptr or None,
                                c_row_stride, M, N, K, ctypes.byref(plan) if plan is not None else None,
                                ws_ptr or None, ws_bytes, flags, stream or None)


def split_activations(A, workspace=None, *, stream=None):
    """w8a16_split_activations: the two E4M3 terms of BF16 A [M, K] (row pitch A.stride(0))
    and their factors, written into `workspace` (a CUDA uint8 tensor of at least
    workspace_bytes(M, K) bytes; None allocates one with torch). Returns the workspace."""
    import torch
    if A.dim() != 2 or A.dtype != torch.bfloat16 or A.stride(1) != 1:
        raise ValueError("A must be a bfloat16 [M, K] tensor with unit column stride")
    M, K = A.shape
    if workspace is None:
        workspace = torch.empty(max(16, workspace_bytes(M, K)), dtype=torch.uint8, device=A.device)
    if workspace.dtype != torch.uint8 or not workspace.is_contiguous():
        raise ValueError("workspace must be a contiguous uint8 tensor")
    _on_one_gpu(A, workspace)
    with torch.cuda.device(A.device):
        rc = load().w8a16_split_activations(A.data_ptr(), A.stride(0), M, K, workspace.data_ptr(),
                                            workspace.numel(), _stream_handle(stream))
    _check(rc)
    return workspace


def gemm_split_terms(workspace, M, W, scale, C=None, *, stream=None, flags: int = 0):
    """w8a16_gemm_split_terms: C [M, >=N] = the product of the activations that
    split_activations() wrote into `workspace` (for M tokens) with W and scale."""
    import torch
    if W.dim() != 2 or not _is_codes(W):
        raise ValueError("W must be a uint8 or float8_e4m3fn [N, K] tensor")
    N, K = W.shape
    _scale_shape(scale, N, K)
    if C is None:
        C = torch.empty((M, N), dtype=torch.bfloat16, device=W.device)
    if C.dtype != torch.bfloat16 or C.shape[0] != M or C.shape[1] < N or C.stride(1) != 1:
        raise ValueError("C must be bfloat16 [M, >=N] with unit column stride")
    if workspace.dtype != torch.uint8 or not workspace.is_contiguous():
        raise ValueError("workspace must be a contiguous uint8 tensor")
    _on_one_gpu(workspace, W, scale, C)
    with torch.cuda.device(W.device):
        rc = load().w8a16_gemm_split_terms(workspace.data_ptr(), workspace.numel(), W.data_ptr(),
                                           scale.data_ptr(), C.data_ptr(), C.stride(0), M, N, K, flags,
                                           _stream_handle(stream))
    _check(rc)
    return C


def gemm_ptr(A_ptr, a_row_stride, W_ptr, scale_ptr, C_ptr, c_row_stride, M, N, K, stream=0,
             plan: Plan | None = None, flags: int = 0) -> int:
    """Raw-pointer call (returns the library's code; does not raise)."""
    lib = load()
    if plan is None:
        return lib.w8a16_gemm_ex(A_ptr, a_row_stride, W_ptr, scale_ptr, C_ptr, c_row_stride, M, N,
                                 K, flags, stream or None)
    return lib.w8a16_gemm_with_plan(A_ptr, a_row_stride, W_ptr, scale_ptr, C_ptr, c_row_stride,
                                    M, N, K, ctypes.byref(plan), flags, stream or None)


def gemm_host(A_host, W_host, scale_host, C_host, dA, dW, dScale, dC, *, copy_weights=True,
              stream=None):
    """Host-buffer call: the library queues H2D copies, the GEMM and the D2H copy.
    Host tensors should be pinned; the device buffers take A and C at the host
    tensors' row pitches (dA, dC), W as [N, K] and the scales at their shape."""
    import torch
    M, N, K = _shapes(A_host, W_host, scale_host, C_host)
    if C_host.dtype != torch.bfloat16 or C_host.shape[0] != M or C_host.shape[1] < N:
        raise ValueError("C_host must be bfloat16 [M, >=N]")
    if any(t.is_cuda for t in (A_host, W_host, scale_host, C_host)):
        raise ValueError("A_host, W_host, scale_host and C_host must be in host memory")
    _on_one_gpu(dA, dW, dScale, dC)
    for name, d, h, rows, cols in (("dA", dA, A_host, M, K), ("dC", dC, C_host, M, N)):
        if (d.dtype != torch.bfloat16 or d.dim() != 2 or d.stride(1) != 1 or d.stride(0) != h.stride(0)
                or d.shape[0] < rows or d.shape[1] < cols):
            raise ValueError(f"{name} must be bfloat16 with at least [{rows}, {cols}] at row pitch {h.stride(0)}")
    if not _is_codes(dW) or not dW.is_contiguous() or tuple(dW.shape) != (N, K):
        raise ValueError(f"dW must be contiguous E4M3 codes [{N}, {K}]")
    if dScale.dtype != torch.float32 or not dScale.is_contiguous() or dScale.shape != scale_host.shape:
        raise ValueError(f"dScale must be contiguous float32 {list(scale_host.shape)}")
    with torch.cuda.device(dA.device):
        rc = load().w8a16_gemm_host(
            A_host.data_ptr(), A_host.stride(0), W_host.data_ptr(), scale_host.data_ptr(),
            C_host.data_ptr(), C_host.stride(0), M, N, K, dA.data_ptr(), dW.data_ptr(),
            dScale.data_ptr(), dC.data_ptr(), 1 if copy_weights else 0, _stream_handle(stream))
    _check(rc)
    return C_host


def quantize_weights(W, *, stream=None):
    """(codes uint8 [N, K], block_scale float32 [ceil(N/128), K/128]) of a CUDA
    float32 or bfloat16 [N, K] weight tensor (rows contiguous, any row pitch)."""
    import torch
    if W.dim() != 2 or W.stride(1) != 1:
        raise ValueError("W must be 2-D with contiguous rows")
    if W.dtype == torch.float32:
        wt = WEIGHTS_F32
    elif W.dtype == torch.bfloat16:
        wt = WEIGHTS_BF16
    else:
        raise TypeError(f"W must be float32 or bfloat16, got {W.dtype}")
    if not W.is_cuda:
        raise ValueError("W must be on a CUDA device")
    N, K = W.shape
    codes = torch.empty((N, K), dtype=torch.uint8, device=W.device)
    scale = torch.empty(((N + 127) // 128, K // 128 if K % 128 == 0 else 1), dtype=torch.float32,
                        device=W.device)
    with torch.cuda.device(W.device):
        rc = load().w8a16_quantize_weights(W.data_ptr(), wt, W.stride(0), N, K, codes.data_ptr(),
                                           scale.data_ptr(), _stream_handle(stream))
    _check(rc)
    return codes, scale


def quantize_activations(A, *, stream=None):
    """(codes uint8 [M, K], scales float32 [K/128, S]) of CUDA bfloat16 activations
    [M, K] (rows contiguous, any pitch); S = M rounded up to a multiple of 4, the
    columns past M unused."""
    import torch
    if A.dim() != 2 or A.stride(1) != 1 or A.dtype != torch.bfloat16 or not A.is_cuda:
        raise ValueError("A must be a CUDA bfloat16 [M, K] tensor with contiguous rows")
    M, K = A.shape
    S = (M + 3) // 4 * 4
    codes = torch.empty((M, K), dtype=torch.uint8, device=A.device)
    scales = torch.zeros((max(K // 128, 1), S), dtype=torch.float32, device=A.device)
    with torch.cuda.device(A.device):
        rc = load().w8a16_quantize_activations(A.data_ptr(), A.stride(0), M, K, codes.data_ptr(),
                                               scales.data_ptr(), S, _stream_handle(stream))
    _check(rc)
    return codes, scales


def gemm_w8a8(A_codes, a_scale, W, scale, C=None, *, stream=None, plan: Plan | None = None,
              flags: int = 0):
    """C[:, :N] (bf16) = (A_codes x a_scale) @ (W x block scales)^T on the GPU.
    A_codes: uint8 [M, K] (row pitch a multiple of 16 bytes); a_scale: float32
    [K/128, >=M] (row pitch a multiple of 4); W: uint8 [N, K]; scale: float32
    [ceil(N/128), K/128]; C: optional bf16 [M, >=N]."""
    import torch
    if A_codes.dim() != 2 or not _is_codes(A_codes) or A_codes.stride(1) != 1:
        raise ValueError("A_codes must be 2-D E4M3 codes (uint8 or float8_e4m3fn) with contiguous rows")
    M, K = A_codes.shape
    if (a_scale.dim() != 2 or a_scale.dtype != torch.float32 or a_scale.stride(1) != 1
            or a_scale.shape[0] < K // 128 or a_scale.shape[1] < M):
        raise ValueError(f"a_scale must be float32 with at least [{K // 128}, {M}] and contiguous rows")
    if W.dim() != 2 or not _is_codes(W) or not W.is_contiguous() or W.shape[1] != K:
        raise ValueError(f"W must be contiguous E4M3 codes [N, {K}]")
    N = W.shape[0]
    if scale.dtype != torch.float32 or not scale.is_contiguous():
        raise ValueError("block_scale must be contiguous float32")
    _scale_shape(scale, N, K)
    if C is None:
        C = torch.empty((M, N), dtype=torch.bfloat16, device=A_codes.device)
    if C.dtype != torch.bfloat16 or C.dim() != 2 or C.stride(1) != 1 or C.shape[0] != M or C.shape[1] < N:
        raise ValueError("C must be bfloat16 [M, >=N] with contiguous rows")
    _on_one_gpu(A_codes, a_scale, W, scale, C)
    args = (A_codes.data_ptr(), A_codes.stride(0), a_scale.data_ptr(), a_scale.stride(0), W.data_ptr(),
            scale.data_ptr(), C.data_ptr(), C.stride(0), M, N, K)
    with torch.cuda.device(A_codes.device):
        s = _stream_handle(stream)
        if plan is None:
            rc = load().w8a16_gemm_w8a8(*args, flags, s)
        else:
            rc = load().w8a16_gemm_w8a8_with_plan(*args, ctypes.byref(plan), flags, s)
    _check(rc)
    return C


def gemm_w8a8_ptr(A_ptr, a_row_stride, a_scale_ptr, a_scale_stride, W_ptr, scale_ptr, C_ptr,
                  c_row_stride, M, N, K, stream=0, flags: int = 0) -> int:
    """Raw-pointer W8A8 call (returns the library's code; does not raise)."""
    return load().w8a16_gemm_w8a8(A_ptr or None, a_row_stride, a_scale_ptr or None, a_scale_stride,
                                  W_ptr or None, scale_ptr or None, C_ptr or None, c_row_stride, M, N,
                                  K, flags, stream or None)


def quantize_weights_ptr(W_ptr, w_dtype, w_row_stride, N, K, codes_ptr, scale_ptr, stream=0) -> int:
    """Raw-pointer call (returns the library's code; does not raise)."""
    return load().w8a16_quantize_weights(W_ptr or None, w_dtype, w_row_stride, N, K, codes_ptr or None,
                                         scale_ptr or None, stream or None)


def device_status(stream=None, clear=False) -> tuple[int, int, int]:
    st, wh, de = ctypes.c_uint32(), ctypes.c_uint32(), ctypes.c_uint32()
    _check(load().w8a16_device_status(_stream_handle(stream), 1 if clear else 0, ctypes.byref(st),
                                      ctypes.byref(wh), ctypes.byref(de)))
    return st.value, wh.value, de.value


def selftest_wait_timeout(timeout_us: int, stream=None):
    _check(load().w8a16_selftest_wait_timeout(timeout_us, _stream_handle(stream)))


def version() -> str:
    return load().w8a16_version().decode()
