"""Block-scaled FP8 (E4M3) quantization, GEMM and on-policy weight sync for
GB300 (sm_103a).

A thin ctypes binding over ``libfp8bs.so`` (C ABI in ``include/fp8bs.h``).
PyTorch provides device memory and streams; every step of the computation
runs in the library's CUDA kernels.  There is no CPU path: every call raises
if the compiled library or a CUDA device is missing.

Shapes follow ``torch.nn.Linear``: X [M, K], W [N, K], Y = X W^T.
"""
from __future__ import annotations

import ctypes as C
import os
from dataclasses import dataclass
from typing import Optional, Sequence

import torch

__all__ = [
    "FP8Error", "QTensor", "SyncEntry", "library", "quantize_group", "quantize_block", "quantize_mx",
    "param_requantize", "requantize_transposed", "dispatch_quantize_mx", "rmsnorm_quantize", "swiglu_quantize", "permute_rows_mx", "gemm", "grouped_gemm", "sync_payload_size", "sync_pack", "sync_install", "sync_install_noalloc",
    "status_poll", "check_wait_expiry", "mx_scale_bytes", "mx_grouped_scale_bytes",
    "RECIPE_BLOCKWISE", "RECIPE_MX", "RECIPE_BLOCKWISE_POW2", "LAYOUT_GROUP_1x128", "LAYOUT_BLOCK_128x128", "LAYOUT_MX_1x32",
    "LAYOUT_MX_1x32_GROUPED",
]

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libfp8bs.so")

RECIPE_BLOCKWISE, RECIPE_MX, RECIPE_BLOCKWISE_POW2 = 1, 2, 3
LAYOUT_GROUP_1x128, LAYOUT_BLOCK_128x128, LAYOUT_MX_1x32, LAYOUT_MX_1x32_GROUPED = 1, 2, 3, 4
AXIS_K, AXIS_M = 0, 1
OP = {"fwd": 0, "dgrad": 1, "wgrad": 2}
OUT_BF16, OUT_F32 = 0, 1
SYNC_FP8, SYNC_BF16 = 1, 2

_STATUS = {0: "FP8_OK", 1: "FP8_ERR_INVALID_ARG", 2: "FP8_ERR_ALIGNMENT", 3: "FP8_ERR_UNSUPPORTED",
           4: "FP8_ERR_BAD_PAYLOAD", 5: "FP8_ERR_CHECKSUM", 6: "FP8_ERR_TIMEOUT", 7: "FP8_ERR_CUDA",
           8: "FP8_ERR_CAPACITY"}


class FP8Error(RuntimeError):
    def __init__(self, status: int, message: str):
        super().__init__(f"{_STATUS.get(status, status)}: {message}")
        self.status = status


class _Tensor(C.Structure):
    _fields_ = [("codes", C.c_void_p), ("scales", C.c_void_p), ("rows", C.c_int64), ("cols", C.c_int64),
                ("recipe", C.c_int32), ("layout", C.c_int32)]


class _SyncEntry(C.Structure):
    _fields_ = [("tag", C.c_uint64), ("kind", C.c_int32), ("reserved", C.c_int32), ("t", _Tensor)]


_lib = None


def library() -> C.CDLL:
    """The loaded CUDA library (raises if it has not been built)."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(LIB_PATH):
        raise FP8Error(7, f"{LIB_PATH} is missing: run __graft_entry__.build() first")
    lib = C.CDLL(LIB_PATH)
    P, I64, I32, S = C.c_void_p, C.c_int64, C.c_int32, C.c_void_p
    TP = C.POINTER(_Tensor)
    EP = C.POINTER(_SyncEntry)
    sigs = {
        "fp8_quantize_group": [P, I64, I64, I64, I32, TP, S],
        "fp8_quantize_block": [P, I64, I64, I64, TP, TP, S],
        "fp8_quantize_mx": [P, I64, I64, I64, TP, S],
        "fp8_quantize_mx_transposed": [P, I64, I64, I64, TP, S],
        "fp8_param_requantize": [P, P, I64, I64, I64, TP, TP, S],
        "fp8_requantize_transposed": [TP, TP, S],
        "fp8_check_wait_expiry": [I64, S],
        "fp8_dispatch_quantize_mx": [P, I64, I64, I64, P, C.c_int32, P, C.c_int32, TP, S],
        "fp8_rmsnorm_quantize": [P, P, I64, I64, I64, C.c_float, P, I64, P, TP, S],
        "fp8_swiglu_quantize": [P, I64, I64, I64, P, I64, TP, S],
        "fp8_permute_rows_mx": [TP, P, P, I32, TP, S],
        "fp8_gemm_blockscaled": [TP, TP, P, I64, I32, I32, TP, S],
        "fp8_grouped_gemm": [TP, TP, P, I32, I64, P, I64, S],
        "fp8_sync_payload_size": [EP, I32, C.POINTER(C.c_uint64)],
        "fp8_sync_pack": [EP, I32, P, C.c_uint64, C.POINTER(C.c_uint64), S],
        "fp8_sync_install": [P, C.c_uint64, EP, I32, S],
        "fp8_sync_install_noalloc": [P, C.c_uint64, EP, I32, S],
        "fp8_status_poll": [S],
    }
    for name, args in sigs.items():
        fn = getattr(lib, name)
        fn.argtypes = args
        fn.restype = C.c_int
    lib.fp8_last_error.restype = C.c_char_p
    lib.fp8_last_error.argtypes = []
    lib.fp8_abi_version.restype = C.c_int32
    lib.fp8_mx_scale_bytes.restype = C.c_int64
    lib.fp8_mx_scale_bytes.argtypes = [I64, I64]
    lib.fp8_mx_grouped_scale_bytes.restype = C.c_int64
    lib.fp8_mx_grouped_scale_bytes.argtypes = [I64, I64, I32]
    _lib = lib
    return lib


def _check(status: int):
    if status != 0:
        raise FP8Error(status, library().fp8_last_error().decode())


def _stream(stream) -> int:
    if stream is None:
        stream = torch.cuda.current_stream()
    return stream.cuda_stream


def _dev(t: torch.Tensor) -> torch.device:
    if not t.is_cuda:
        raise FP8Error(1, "inputs must be CUDA tensors (there is no CPU path)")
    return t.device


@dataclass
class QTensor:
    """A quantized matrix: E4M3 codes [rows, cols] (uint8) and its scales."""
    codes: torch.Tensor
    scales: torch.Tensor
    rows: int
    cols: int
    recipe: int
    layout: int

    def c(self) -> _Tensor:
        return _Tensor(self.codes.data_ptr(), self.scales.data_ptr(), self.rows, self.cols, self.recipe,
                       self.layout)


def mx_scale_bytes(rows: int, cols: int) -> int:
    return int(library().fp8_mx_scale_bytes(rows, cols))


def mx_grouped_scale_bytes(total_rows: int, cols: int, groups: int) -> int:
    return int(library().fp8_mx_grouped_scale_bytes(total_rows, cols, groups))


def _bf16_2d(x: torch.Tensor) -> torch.Tensor:
    if x.dtype != torch.bfloat16 or x.dim() != 2 or x.stride(1) != 1:
        raise FP8Error(1, "expected a 2-D bf16 tensor with unit column stride")
    return x


# ---------------------------------------------------------------- quantizers
def _scales_for(rows: int, cols: int, pow2: bool, fp32_shape, dev) -> torch.Tensor:
    if pow2:
        return torch.empty((mx_scale_bytes(rows, cols),), dtype=torch.uint8, device=dev)
    return torch.empty(fp32_shape, dtype=torch.float32, device=dev)


def quantize_group(x: torch.Tensor, axis: str = "K", out: Optional[QTensor] = None, stream=None,
                   pow2: bool = False) -> QTensor:
    """1x128 groups along K (axis='K') or 128x1 groups along M written
    transposed (axis='M', the WGrad operand layout).  pow2=True: power-of-two
    scales as E8M0 bytes in the MX layout (RECIPE_BLOCKWISE_POW2).  `out`
    may supply preallocated codes/scales."""
    x = _bf16_2d(x)
    M, K = x.shape
    dev = _dev(x)
    recipe = RECIPE_BLOCKWISE_POW2 if pow2 else RECIPE_BLOCKWISE
    layout = LAYOUT_MX_1x32 if pow2 else LAYOUT_GROUP_1x128
    if axis == "K":
        q = out or QTensor(torch.empty((M, K), dtype=torch.uint8, device=dev),
                           _scales_for(M, K, pow2, (K // 128, M), dev), M, K, recipe, layout)
        ax = AXIS_K
    elif axis == "M":
        q = out or QTensor(torch.empty((K, M), dtype=torch.uint8, device=dev),
                           _scales_for(K, M, pow2, (M // 128, K), dev), K, M, recipe, layout)
        ax = AXIS_M
    else:
        raise FP8Error(1, f"axis must be 'K' or 'M', got {axis!r}")
    t = q.c()
    _check(library().fp8_quantize_group(x.data_ptr(), M, K, x.stride(0), ax, C.byref(t), _stream(stream)))
    return q


def requantize_transposed(q: QTensor, out: Optional[QTensor] = None, stream=None) -> QTensor:
    """128x1 transposed quantization (the WGrad operand) of the fp32
    dequantization of a saved 1x128 FP8 tensor [M, K]: codes [K, M], scales
    [M/128, K]."""
    if q.recipe != RECIPE_BLOCKWISE or q.layout != LAYOUT_GROUP_1x128:
        raise FP8Error(1, "requantize_transposed takes a 1x128 blockwise tensor")
    M, K = q.rows, q.cols
    dev = _dev(q.codes)
    out = out or QTensor(torch.empty((K, M), dtype=torch.uint8, device=dev),
                         torch.empty((M // 128, K), dtype=torch.float32, device=dev), K, M, RECIPE_BLOCKWISE,
                         LAYOUT_GROUP_1x128)
    a, b = q.c(), out.c()
    _check(library().fp8_requantize_transposed(C.byref(a), C.byref(b), _stream(stream)))
    return out


def quantize_block(w: torch.Tensor, transposed: bool = False, out: Optional[QTensor] = None,
                   out_t: Optional[QTensor] = None, stream=None, pow2: bool = False):
    """128x128 blocks; with transposed=True also returns the transposed copy
    (codes [K, N], scales [K/128, N/128]) used as the DGrad B operand.
    pow2=True: power-of-two scales in the MX layout (RECIPE_BLOCKWISE_POW2)."""
    w = _bf16_2d(w)
    N, K = w.shape
    dev = _dev(w)
    recipe = RECIPE_BLOCKWISE_POW2 if pow2 else RECIPE_BLOCKWISE
    layout = LAYOUT_MX_1x32 if pow2 else LAYOUT_BLOCK_128x128
    q = out or QTensor(torch.empty((N, K), dtype=torch.uint8, device=dev),
                       _scales_for(N, K, pow2, (N // 128, K // 128), dev), N, K, recipe, layout)
    qt = None
    if transposed:
        qt = out_t or QTensor(torch.empty((K, N), dtype=torch.uint8, device=dev),
                              _scales_for(K, N, pow2, (K // 128, N // 128), dev), K, N, recipe, layout)
    t = q.c()
    tt = qt.c() if qt is not None else None
    _check(library().fp8_quantize_block(w.data_ptr(), N, K, w.stride(0), C.byref(t),
                                        C.byref(tt) if tt is not None else None, _stream(stream)))
    return (q, qt) if transposed else q


def param_requantize(master: torch.Tensor, delta: Optional[torch.Tensor] = None, transposed: bool = False,
                     out: Optional[QTensor] = None, out_t: Optional[QTensor] = None, stream=None,
                     pow2: bool = False):
    """fp8_param: Q(W) of an fp32 master [N, K] in 128x128 blocks.  With a
    delta, master += delta (fp32, in place) first.  Returns the FP8 weight
    (and its transposed copy when transposed=True)."""
    if master.dtype != torch.float32 or master.dim() != 2 or master.stride(1) != 1:
        raise TypeError("master must be a row-major 2-D float32 tensor")
    N, K = master.shape
    dev = _dev(master)
    if delta is not None:
        if delta.dtype != torch.float32 or delta.shape != master.shape or delta.stride() != master.stride():
            raise TypeError("delta must be a float32 tensor with the master's shape and strides")
        if delta.device != master.device:
            raise TypeError("delta must be on the master's device")
    recipe = RECIPE_BLOCKWISE_POW2 if pow2 else RECIPE_BLOCKWISE
    layout = LAYOUT_MX_1x32 if pow2 else LAYOUT_BLOCK_128x128
    q = out or QTensor(torch.empty((N, K), dtype=torch.uint8, device=dev),
                       _scales_for(N, K, pow2, (N // 128, K // 128), dev), N, K, recipe, layout)
    qt = None
    if transposed:
        qt = out_t or QTensor(torch.empty((K, N), dtype=torch.uint8, device=dev),
                              _scales_for(K, N, pow2, (K // 128, N // 128), dev), K, N, recipe, layout)
    t = q.c()
    tt = qt.c() if qt is not None else None
    _check(library().fp8_param_requantize(master.data_ptr(), delta.data_ptr() if delta is not None else None, N, K,
                                          master.stride(0), C.byref(t), C.byref(tt) if tt is not None else None,
                                          _stream(stream)))
    return (q, qt) if transposed else q


def _activation_out(rows: int, cols: int, recipe: int, dev) -> QTensor:
    if recipe == RECIPE_BLOCKWISE:
        return QTensor(torch.empty((rows, cols), dtype=torch.uint8, device=dev),
                       torch.empty((cols // 128, rows), dtype=torch.float32, device=dev), rows, cols, recipe,
                       LAYOUT_GROUP_1x128)
    if recipe in (RECIPE_BLOCKWISE_POW2, RECIPE_MX):
        return QTensor(torch.empty((rows, cols), dtype=torch.uint8, device=dev),
                       torch.empty((mx_scale_bytes(rows, cols),), dtype=torch.uint8, device=dev), rows, cols, recipe,
                       LAYOUT_MX_1x32)
    raise ValueError(f"unsupported activation recipe {recipe}")


def rmsnorm_quantize(x: torch.Tensor, gamma: torch.Tensor, eps: float = 1e-6, recipe: int = RECIPE_BLOCKWISE,
                     want_y: bool = False, want_rstd: bool = False, out: Optional[QTensor] = None,
                     y: Optional[torch.Tensor] = None, rstd: Optional[torch.Tensor] = None, stream=None):
    """RMSNorm of bf16 rows fused with their quantization.  Returns the FP8
    activation, plus y (bf16) and rstd (fp32) when asked for."""
    x = _bf16_2d(x)
    M, K = x.shape
    dev = _dev(x)
    if gamma.dtype != torch.bfloat16 or gamma.shape != (K,) or not gamma.is_contiguous():
        raise TypeError("gamma must be a contiguous bf16 vector of length K")
    q = out or _activation_out(M, K, recipe, dev)
    if want_y and y is None:
        y = torch.empty((M, K), dtype=torch.bfloat16, device=dev)
    if want_rstd and rstd is None:
        rstd = torch.empty((M,), dtype=torch.float32, device=dev)
    t = q.c()
    _check(library().fp8_rmsnorm_quantize(x.data_ptr(), gamma.data_ptr(), M, K, x.stride(0), float(eps),
                                          y.data_ptr() if y is not None else None, y.stride(0) if y is not None else 0,
                                          rstd.data_ptr() if rstd is not None else None, C.byref(t), _stream(stream)))
    res = (q,) + ((y,) if want_y else ()) + ((rstd,) if want_rstd else ())
    return res if len(res) > 1 else q


def swiglu_quantize(gu: torch.Tensor, recipe: int = RECIPE_BLOCKWISE, want_h: bool = False,
                    out: Optional[QTensor] = None, h: Optional[torch.Tensor] = None, stream=None):
    """silu(gate) * up of a [M, 2F] bf16 tensor (gate | up) fused with the
    quantization of the [M, F] result.  Returns the FP8 activation (and h)."""
    gu = _bf16_2d(gu)
    M, F2 = gu.shape
    if F2 % 2:
        raise ValueError("gu must have an even number of columns (gate | up)")
    F = F2 // 2
    dev = _dev(gu)
    q = out or _activation_out(M, F, recipe, dev)
    if want_h and h is None:
        h = torch.empty((M, F), dtype=torch.bfloat16, device=dev)
    t = q.c()
    _check(library().fp8_swiglu_quantize(gu.data_ptr(), M, F, gu.stride(0), h.data_ptr() if h is not None else None,
                                         h.stride(0) if h is not None else 0, C.byref(t), _stream(stream)))
    return (q, h) if want_h else q


def quantize_mx(x: torch.Tensor, out: Optional[QTensor] = None, stream=None, transposed: bool = False) -> QTensor:
    """MXFP8: 1x32 blocks, E8M0 scales in the tensor-core atom layout.
    transposed=True: 32x1 blocks along the rows, codes written transposed
    [K, R] (the MXFP8 backward operands W^T, dY^T, X^T)."""
    x = _bf16_2d(x)
    R, K = x.shape
    dev = _dev(x)
    if transposed:
        q = out or QTensor(torch.empty((K, R), dtype=torch.uint8, device=dev),
                           torch.empty((mx_scale_bytes(K, R),), dtype=torch.uint8, device=dev), K, R, RECIPE_MX,
                           LAYOUT_MX_1x32)
        t = q.c()
        _check(library().fp8_quantize_mx_transposed(x.data_ptr(), R, K, x.stride(0), C.byref(t), _stream(stream)))
        return q
    q = out or QTensor(torch.empty((R, K), dtype=torch.uint8, device=dev),
                torch.empty((mx_scale_bytes(R, K),), dtype=torch.uint8, device=dev), R, K, RECIPE_MX,
                LAYOUT_MX_1x32)
    t = q.c()
    _check(library().fp8_quantize_mx(x.data_ptr(), R, K, x.stride(0), C.byref(t), _stream(stream)))
    return q


def permute_rows_mx(q: QTensor, gather: torch.Tensor, offsets: torch.Tensor, out: Optional[QTensor] = None,
                    stream=None) -> QTensor:
    """Gathers MX rows into expert-contiguous groups (dst row i = src row
    gather[i]); offsets int32 [G+1] on the device."""
    if gather.dtype != torch.int32 or offsets.dtype != torch.int32:
        raise FP8Error(1, "gather and offsets must be int32")
    total = gather.numel()
    G = offsets.numel() - 1
    dev = _dev(q.codes)
    out = out or QTensor(torch.empty((total, q.cols), dtype=torch.uint8, device=dev),
                  torch.empty((mx_grouped_scale_bytes(total, q.cols, G),), dtype=torch.uint8, device=dev),
                  total, q.cols, RECIPE_MX, LAYOUT_MX_1x32_GROUPED)
    src, dst = q.c(), out.c()
    _check(library().fp8_permute_rows_mx(C.byref(src), gather.data_ptr(), offsets.data_ptr(), G, C.byref(dst),
                                         _stream(stream)))
    return out


def dispatch_quantize_mx(x: torch.Tensor, dst_index: torch.Tensor, offsets: torch.Tensor, total: int,
                         out: Optional[QTensor] = None, stream=None) -> QTensor:
    """MoE dispatch fused with the MX quantization: every token row of x is
    quantized once and written to dst rows dst_index[t, :] (int32 [T, top_k],
    -1 = dropped) of a total-row grouped MXFP8 tensor."""
    x = _bf16_2d(x)
    if dst_index.dtype != torch.int32 or offsets.dtype != torch.int32 or dst_index.dim() != 2:
        raise FP8Error(1, "dst_index must be int32 [T, top_k], offsets int32")
    T, K = x.shape
    if dst_index.shape[0] != T or not dst_index.is_contiguous():
        raise FP8Error(1, "dst_index must be a contiguous [T, top_k] tensor")
    G = offsets.numel() - 1
    dev = _dev(x)
    out = out or QTensor(torch.empty((total, K), dtype=torch.uint8, device=dev),
                         torch.empty((mx_grouped_scale_bytes(total, K, G),), dtype=torch.uint8, device=dev),
                         total, K, RECIPE_MX, LAYOUT_MX_1x32_GROUPED)
    dst = out.c()
    _check(library().fp8_dispatch_quantize_mx(x.data_ptr(), T, K, x.stride(0), dst_index.data_ptr(),
                                              dst_index.shape[1], offsets.data_ptr(), G, C.byref(dst),
                                              _stream(stream)))
    return out


# ---------------------------------------------------------------- GEMMs
def gemm(A: QTensor, B: QTensor, op: str = "fwd", out_dtype=torch.bfloat16, quantize_output: bool = False,
         out: Optional[torch.Tensor] = None, out_q: Optional[QTensor] = None, stream=None):
    """D = A B^T with fp32 accumulation.  Returns D, or (D, QTensor of D)
    when quantize_output (1x128 for blockwise, 1x32 for MXFP8, 1x128 with
    power-of-two scales for the blockwise power-of-two recipe)."""
    M, N = A.rows, B.rows
    dev = _dev(A.codes)
    if out is None:
        out = torch.empty((M, N), dtype=out_dtype, device=dev)
    dq = out_q
    if quantize_output and dq is None:
        if A.recipe == RECIPE_BLOCKWISE:
            dq = QTensor(torch.empty((M, N), dtype=torch.uint8, device=dev),
                         torch.empty((N // 128, M), dtype=torch.float32, device=dev), M, N, RECIPE_BLOCKWISE,
                         LAYOUT_GROUP_1x128)
        else:
            dq = QTensor(torch.empty((M, N), dtype=torch.uint8, device=dev),
                         torch.empty((mx_scale_bytes(M, N),), dtype=torch.uint8, device=dev), M, N, A.recipe,
                         LAYOUT_MX_1x32)
    a, b = A.c(), B.c()
    dqc = dq.c() if dq is not None else None
    dt = OUT_F32 if out.dtype == torch.float32 else OUT_BF16
    _check(library().fp8_gemm_blockscaled(C.byref(a), C.byref(b), out.data_ptr(), out.stride(0), dt, OP[op],
                                          C.byref(dqc) if dqc is not None else None, _stream(stream)))
    return (out, dq) if quantize_output else out


def grouped_gemm(A: QTensor, B_stack: QTensor, offsets: torch.Tensor, N: int, out: Optional[torch.Tensor] = None,
                 stream=None) -> torch.Tensor:
    """Per-expert D[off_g:off_g+1] = A_g W_g^T (MXFP8)."""
    G = offsets.numel() - 1
    if out is None:
        out = torch.empty((A.rows, N), dtype=torch.bfloat16, device=_dev(A.codes))
    a, b = A.c(), B_stack.c()
    _check(library().fp8_grouped_gemm(C.byref(a), C.byref(b), offsets.data_ptr(), G, N, out.data_ptr(),
                                      out.stride(0), _stream(stream)))
    return out


# ---------------------------------------------------------------- weight sync
@dataclass
class SyncEntry:
    """One tensor of a weight-sync payload: a QTensor, or a bf16 tensor kept
    in high precision (norms, embeddings)."""
    tag: int
    tensor: object  # QTensor or bf16 torch.Tensor

    def c(self) -> _SyncEntry:
        if isinstance(self.tensor, QTensor):
            return _SyncEntry(self.tag, SYNC_FP8, 0, self.tensor.c())
        t = self.tensor
        if t.dtype != torch.bfloat16 or t.dim() != 2 or not t.is_contiguous():
            raise FP8Error(1, "bf16 sync entries must be contiguous 2-D bf16 tensors")
        return _SyncEntry(self.tag, SYNC_BF16, 0, _Tensor(t.data_ptr(), None, t.shape[0], t.shape[1], 0, 0))


def _entries(entries: Sequence[SyncEntry]):
    arr = (_SyncEntry * max(1, len(entries)))()
    for i, e in enumerate(entries):
        arr[i] = e.c()
    return arr


def sync_payload_size(entries: Sequence[SyncEntry]) -> int:
    n = C.c_uint64(0)
    _check(library().fp8_sync_payload_size(_entries(entries), len(entries), C.byref(n)))
    return int(n.value)


def sync_pack(entries: Sequence[SyncEntry], payload: Optional[torch.Tensor] = None, stream=None) -> torch.Tensor:
    """Packs the trainer's FP8 codes + scales (and bf16 tensors) into one
    device payload."""
    size = sync_payload_size(entries)
    if payload is None:
        dev = entries[0].tensor.codes.device if isinstance(entries[0].tensor, QTensor) else entries[0].tensor.device
        payload = torch.empty((size,), dtype=torch.uint8, device=dev)
    used = C.c_uint64(0)
    _check(library().fp8_sync_pack(_entries(entries), len(entries), payload.data_ptr(), payload.numel(),
                                   C.byref(used), _stream(stream)))
    return payload[: used.value]


def sync_install(payload: torch.Tensor, dst: Sequence[SyncEntry], stream=None, check: bool = True):
    """Installs a payload into the rollout-side tensors (no quantizer runs).
    With check=True the device-side checksum verdict is read back and a
    mismatch raises FP8Error(FP8_ERR_CHECKSUM)."""
    _check(library().fp8_sync_install(payload.data_ptr(), payload.numel(), _entries(dst), len(dst),
                                      _stream(stream)))
    if check:
        status_poll(stream)


def sync_install_noalloc(payload: torch.Tensor, dst: Sequence[SyncEntry], stream=None):
    """sync_install for callers that cannot allocate device memory: the
    library's fixed scratch array is used instead (at most 128 entries;
    installs are ordered on the device, as for sync_install).  Blocks until
    the copy is done; a checksum
    mismatch raises FP8Error(FP8_ERR_CHECKSUM)."""
    _check(library().fp8_sync_install_noalloc(payload.data_ptr(), payload.numel(), _entries(dst), len(dst),
                                              _stream(stream)))


def check_wait_expiry(limit_ns: int = 20_000_000, stream=None) -> None:
    """Runs the library's bounded-wait failure path on the device (a wait
    that nothing completes, given up after limit_ns); the next status_poll()
    raises FP8Error with FP8_ERR_TIMEOUT."""
    _check(library().fp8_check_wait_expiry(int(limit_ns), _stream(stream)))


def status_poll(stream=None):
    _check(library().fp8_status_poll(_stream(stream)))
