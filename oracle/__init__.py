"""CPU oracle for block-scaled FP8 (E4M3): ctypes marshalling over fp8_oracle.c.

TEST INFRASTRUCTURE ONLY.  The product package never imports this module;
only tests, the smoke check and the benchmark's CPU-baseline leg do.  All
arithmetic lives in fp8_oracle.c (plain C, fp64/IEEE fp32, no fast-math);
this file only converts numpy arrays to pointers and back.

bf16 tensors are passed as their uint16 bit patterns.
"""
from __future__ import annotations

import ctypes as C
import os

import numpy as np

from ._build import build_oracle, library_path

_lib = None

_P = C.c_void_p
_I64 = C.c_int64


def load():
    """Loads (building first if needed) the oracle shared library."""
    global _lib
    if _lib is not None:
        return _lib
    path = build_oracle()  # rebuilds when fp8_oracle.c is newer than the library
    lib = C.CDLL(path)
    sig = {
        "oracle_e4m3_decode": (C.c_double, [C.c_uint8]),
        "oracle_e4m3_encode_f64": (C.c_uint8, [C.c_double]),
        "oracle_e4m3_encode_f32": (C.c_uint8, [C.c_float]),
        "oracle_e4m3_encode_array": (None, [_P, _I64, _P]),
        "oracle_e4m3_decode_array": (None, [_P, _I64, _P]),
        "oracle_quant_group_1x128": (None, [_P, _I64, _I64, _I64, _P, _P]),
        "oracle_quant_group_128x1_T": (None, [_P, _I64, _I64, _I64, _P, _P]),
        "oracle_quant_block_128x128": (None, [_P, _I64, _I64, _I64, _P, _P, _P, _P]),
        "oracle_mx_scale_offset": (_I64, [_I64, _I64, _I64]),
        "oracle_mx_scale_bytes": (_I64, [_I64, _I64]),
        "oracle_quant_mx_1x32": (None, [_P, _I64, _I64, _I64, _P, _P]),
        "oracle_quant_mx_32x1_T": (None, [_P, _I64, _I64, _I64, _P, _P]),
        "oracle_pow2_exponent": (C.c_int, [C.c_float]),
        "oracle_quant_group_1x128_pow2": (None, [_P, _I64, _I64, _I64, _P, _P]),
        "oracle_quant_group_128x1_T_pow2": (None, [_P, _I64, _I64, _I64, _P, _P]),
        "oracle_quant_block_128x128_pow2": (None, [_P, _I64, _I64, _I64, _P, _P, _P, _P]),
        "oracle_param_update": (None, [_P, _P, _I64, _I64, _I64]),
        "oracle_quant_block_128x128_f32": (None, [_P, _I64, _I64, _I64, _P, _P, _P, _P]),
        "oracle_quant_block_128x128_f32_pow2": (None, [_P, _I64, _I64, _I64, _P, _P, _P, _P]),
        "oracle_requant_1x128_to_128x1_T": (None, [_P, _P, _I64, _I64, _P, _P]),
        "oracle_bf16_round_f64": (C.c_uint16, [C.c_double]),
        "oracle_rmsnorm": (None, [_P, _P, _I64, _I64, _I64, C.c_float, _P, _P]),
        "oracle_swiglu": (None, [_P, _I64, _I64, _I64, _P]),
        "oracle_dequant_group": (None, [_P, _P, _I64, _I64, _P]),
        "oracle_dequant_block": (None, [_P, _P, _I64, _I64, _P]),
        "oracle_dequant_mx": (None, [_P, _P, _I64, _I64, _P]),
        "oracle_gemm_ref": (None, [_P, _P, _I64, _I64, _I64, _P, _P]),
        "oracle_gemm_ref_sampled": (None, [_P, _P, _I64, _P, _P, _I64, _P, _P]),
        "oracle_naive_requant_per_tensor": (C.c_float, [_P, _P, _I64, _I64, _P]),
        "oracle_sync_word_term": (C.c_uint64, [C.c_uint64, C.c_uint64]),
        "oracle_sync_checksum": (C.c_uint64, [_P, C.c_uint64]),
        "oracle_sync_payload_size": (C.c_uint64, [_P, C.c_int32]),
        "oracle_sync_pack": (C.c_uint64, [_P, C.c_int32, _P, C.c_uint64]),
        "oracle_sync_install": (C.c_int32, [_P, C.c_uint64, _P, C.c_int32]),
        "oracle_set_threads": (None, [C.c_int32]),
        "oracle_max_threads": (C.c_int32, []),
    }
    for name, (res, args) in sig.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    _lib = lib
    return lib


def set_threads(n: int) -> None:
    """Thread count of the oracle's OpenMP loops (timing only)."""
    load().oracle_set_threads(int(n))


def max_threads() -> int:
    return int(load().oracle_max_threads())


def _ptr(a: np.ndarray):
    assert a.flags["C_CONTIGUOUS"], "oracle arrays must be C-contiguous"
    return a.ctypes.data_as(C.c_void_p)


def _bits(x) -> np.ndarray:
    x = np.ascontiguousarray(x)
    if x.dtype != np.uint16:
        raise TypeError("bf16 inputs are passed as uint16 bit patterns")
    return x


# ---------------------------------------------------------------- scalars
def e4m3_decode(codes) -> np.ndarray:
    c = np.ascontiguousarray(codes, dtype=np.uint8)
    out = np.empty(c.shape, dtype=np.float64)
    load().oracle_e4m3_decode_array(_ptr(c), c.size, _ptr(out))
    return out


def e4m3_encode(values) -> np.ndarray:
    v = np.ascontiguousarray(values, dtype=np.float32)
    out = np.empty(v.shape, dtype=np.uint8)
    load().oracle_e4m3_encode_array(_ptr(v), v.size, _ptr(out))
    return out


def e4m3_encode_exact(value: float) -> int:
    """Encodes one exact real value (a Python float / fp64)."""
    return int(load().oracle_e4m3_encode_f64(float(value)))


# ---------------------------------------------------------------- quantizers
def quant_group_1x128(x_bits):
    x = _bits(x_bits)
    M, K = x.shape
    codes = np.empty((M, K), np.uint8)
    scales = np.empty((K // 128, M), np.float32)
    load().oracle_quant_group_1x128(_ptr(x), M, K, K, _ptr(codes), _ptr(scales))
    return codes, scales


def quant_group_128x1_T(x_bits):
    x = _bits(x_bits)
    M, K = x.shape
    codes_t = np.empty((K, M), np.uint8)
    scales = np.empty((M // 128, K), np.float32)
    load().oracle_quant_group_128x1_T(_ptr(x), M, K, K, _ptr(codes_t), _ptr(scales))
    return codes_t, scales


def quant_block_128x128(w_bits, transposed: bool = False):
    w = _bits(w_bits)
    N, K = w.shape
    codes = np.empty((N, K), np.uint8)
    scales = np.empty((N // 128, K // 128), np.float32)
    if transposed:
        codes_t = np.empty((K, N), np.uint8)
        scales_t = np.empty((K // 128, N // 128), np.float32)
        load().oracle_quant_block_128x128(_ptr(w), N, K, K, _ptr(codes), _ptr(scales),
                                          _ptr(codes_t), _ptr(scales_t))
        return codes, scales, codes_t, scales_t
    load().oracle_quant_block_128x128(_ptr(w), N, K, K, _ptr(codes), _ptr(scales), None, None)
    return codes, scales


def mx_scale_offset(r: int, kb: int, K: int) -> int:
    return int(load().oracle_mx_scale_offset(r, kb, K))


def mx_scale_bytes(R: int, K: int) -> int:
    return int(load().oracle_mx_scale_bytes(R, K))


def quant_mx_1x32(x_bits):
    x = _bits(x_bits)
    R, K = x.shape
    codes = np.empty((R, K), np.uint8)
    scales = np.empty((mx_scale_bytes(R, K),), np.uint8)
    load().oracle_quant_mx_1x32(_ptr(x), R, K, K, _ptr(codes), _ptr(scales))
    return codes, scales


def quant_mx_32x1_T(x_bits):
    """32x1 MX blocks along the rows, codes transposed [K][R] (MX backward)."""
    x = _bits(x_bits)
    R, K = x.shape
    codes_t = np.empty((K, R), np.uint8)
    scales_t = np.empty((mx_scale_bytes(K, R),), np.uint8)
    load().oracle_quant_mx_32x1_T(_ptr(x), R, K, K, _ptr(codes_t), _ptr(scales_t))
    return codes_t, scales_t


def pow2_exponent(amax: float) -> int:
    return int(load().oracle_pow2_exponent(float(amax)))


def quant_group_1x128_pow2(x_bits):
    """1x128 groups, power-of-two scales as E8M0 bytes in the MX atom layout."""
    x = _bits(x_bits)
    M, K = x.shape
    codes = np.empty((M, K), np.uint8)
    scales = np.empty((mx_scale_bytes(M, K),), np.uint8)
    load().oracle_quant_group_1x128_pow2(_ptr(x), M, K, K, _ptr(codes), _ptr(scales))
    return codes, scales


def quant_group_128x1_T_pow2(x_bits):
    x = _bits(x_bits)
    M, K = x.shape
    codes_t = np.empty((K, M), np.uint8)
    scales_t = np.empty((mx_scale_bytes(K, M),), np.uint8)
    load().oracle_quant_group_128x1_T_pow2(_ptr(x), M, K, K, _ptr(codes_t), _ptr(scales_t))
    return codes_t, scales_t


def quant_block_128x128_pow2(w_bits, transposed: bool = False):
    w = _bits(w_bits)
    N, K = w.shape
    codes = np.empty((N, K), np.uint8)
    scales = np.empty((mx_scale_bytes(N, K),), np.uint8)
    if transposed:
        codes_t = np.empty((K, N), np.uint8)
        scales_t = np.empty((mx_scale_bytes(K, N),), np.uint8)
        load().oracle_quant_block_128x128_pow2(_ptr(w), N, K, K, _ptr(codes), _ptr(scales),
                                               _ptr(codes_t), _ptr(scales_t))
        return codes, scales, codes_t, scales_t
    load().oracle_quant_block_128x128_pow2(_ptr(w), N, K, K, _ptr(codes), _ptr(scales), None, None)
    return codes, scales


# ---------------------------------------------------------------- fp8_param
def _f32(x) -> np.ndarray:
    x = np.ascontiguousarray(x)
    if x.dtype != np.float32:
        raise TypeError("fp32 master weights are passed as float32 arrays")
    return x


def param_update(master, delta) -> np.ndarray:
    """W_t = W_{t-1} + dW in fp32 (returns a new array)."""
    m = _f32(master).copy()
    d = _f32(delta)
    assert m.shape == d.shape and m.ndim == 2
    load().oracle_param_update(_ptr(m), _ptr(d), m.shape[0], m.shape[1], m.shape[1])
    return m


def quant_block_128x128_f32(w, transposed: bool = False, pow2: bool = False):
    """Q(W) of an fp32 master: 128x128 blocks, fp32 scales [N/128][K/128] or
    (pow2) E8M0 bytes in the MX atom layout."""
    w = _f32(w)
    N, K = w.shape
    codes = np.empty((N, K), np.uint8)
    if pow2:
        scales = np.empty((mx_scale_bytes(N, K),), np.uint8)
        scales_t = np.empty((mx_scale_bytes(K, N),), np.uint8) if transposed else None
        fn = load().oracle_quant_block_128x128_f32_pow2
    else:
        scales = np.empty((N // 128, K // 128), np.float32)
        scales_t = np.empty((K // 128, N // 128), np.float32) if transposed else None
        fn = load().oracle_quant_block_128x128_f32
    codes_t = np.empty((K, N), np.uint8) if transposed else None
    fn(_ptr(w), N, K, K, _ptr(codes), _ptr(scales),
       _ptr(codes_t) if transposed else None, _ptr(scales_t) if transposed else None)
    if transposed:
        return codes, scales, codes_t, scales_t
    return codes, scales


# ---------------------------------------------------------------- saved activation -> WGrad operand
def requant_1x128_to_128x1_T(codes, scales):
    """The 128x1 transposed quantization of the fp32 dequantization of a
    1x128-quantized [M, K] tensor: (codes^T [K, M], scales [M/128, K])."""
    c = np.ascontiguousarray(codes, np.uint8)
    s = np.ascontiguousarray(scales, np.float32)
    M, K = c.shape
    assert s.shape == (K // 128, M)
    codes_t = np.empty((K, M), np.uint8)
    scales_t = np.empty((M // 128, K), np.float32)
    load().oracle_requant_1x128_to_128x1_T(_ptr(c), _ptr(s), M, K, _ptr(codes_t), _ptr(scales_t))
    return codes_t, scales_t


# ---------------------------------------------------------------- fused producers
def bf16_round(values) -> np.ndarray:
    """bf16 bit patterns nearest to each (fp64) value."""
    v = np.asarray(values, np.float64)
    fn = load().oracle_bf16_round_f64
    return np.array([fn(float(a)) for a in v.ravel()], np.uint16).reshape(v.shape)


def rmsnorm(x_bits, gamma_bits, eps: float):
    """RMSNorm in fp64, output rounded to bf16: (y bits [M, K], rstd fp32 [M])."""
    x = _bits(x_bits)
    g = _bits(gamma_bits)
    M, K = x.shape
    assert g.shape == (K,)
    y = np.empty((M, K), np.uint16)
    rstd = np.empty((M,), np.float32)
    load().oracle_rmsnorm(_ptr(x), _ptr(g), M, K, K, float(eps), _ptr(y), _ptr(rstd))
    return y, rstd


def swiglu(gu_bits):
    """silu(gate) * up of a [M, 2F] row pair in fp64, rounded to bf16: [M, F]."""
    gu = _bits(gu_bits)
    M, F2 = gu.shape
    F = F2 // 2
    h = np.empty((M, F), np.uint16)
    load().oracle_swiglu(_ptr(gu), M, F, F2, _ptr(h))
    return h


# ---------------------------------------------------------------- dequant
def dequant_group(codes, scales):
    codes = np.ascontiguousarray(codes, np.uint8)
    scales = np.ascontiguousarray(scales, np.float32)
    R, K = codes.shape
    out = np.empty((R, K), np.float64)
    load().oracle_dequant_group(_ptr(codes), _ptr(scales), R, K, _ptr(out))
    return out


def dequant_block(codes, scales):
    codes = np.ascontiguousarray(codes, np.uint8)
    scales = np.ascontiguousarray(scales, np.float32)
    R, K = codes.shape
    out = np.empty((R, K), np.float64)
    load().oracle_dequant_block(_ptr(codes), _ptr(scales), R, K, _ptr(out))
    return out


def dequant_mx(codes, scales):
    codes = np.ascontiguousarray(codes, np.uint8)
    scales = np.ascontiguousarray(scales, np.uint8)
    R, K = codes.shape
    out = np.empty((R, K), np.float64)
    load().oracle_dequant_mx(_ptr(codes), _ptr(scales), R, K, _ptr(out))
    return out


# ---------------------------------------------------------------- GEMM
def gemm_ref(a_deq, b_deq):
    """ref = A . B^T and mag = |A| . |B|^T, both fp64; A [M,K], B [N,K]."""
    a = np.ascontiguousarray(a_deq, np.float64)
    b = np.ascontiguousarray(b_deq, np.float64)
    M, K = a.shape
    N = b.shape[0]
    assert b.shape[1] == K
    ref = np.empty((M, N), np.float64)
    mag = np.empty((M, N), np.float64)
    load().oracle_gemm_ref(_ptr(a), _ptr(b), M, N, K, _ptr(ref), _ptr(mag))
    return ref, mag


def gemm_ref_sampled(a_deq, b_deq, ms, ns):
    a = np.ascontiguousarray(a_deq, np.float64)
    b = np.ascontiguousarray(b_deq, np.float64)
    ms = np.ascontiguousarray(ms, np.int64)
    ns = np.ascontiguousarray(ns, np.int64)
    K = a.shape[1]
    ref = np.empty(ms.shape, np.float64)
    mag = np.empty(ms.shape, np.float64)
    load().oracle_gemm_ref_sampled(_ptr(a), _ptr(b), K, _ptr(ms), _ptr(ns), ms.size,
                                   _ptr(ref), _ptr(mag))
    return ref, mag


def gemm_tolerance(ref, mag):
    """Per-element bound |gpu - ref| <= 2e-3 * mag + 2^-8 * |ref|."""
    return 2e-3 * np.asarray(mag) + (2.0 ** -8) * np.abs(np.asarray(ref))


# ---------------------------------------------------------------- sync
def naive_requant_per_tensor(codes, block_scales):
    codes = np.ascontiguousarray(codes, np.uint8)
    block_scales = np.ascontiguousarray(block_scales, np.float32)
    N, K = codes.shape
    out = np.empty((N, K), np.uint8)
    s = load().oracle_naive_requant_per_tensor(_ptr(codes), _ptr(block_scales), N, K, _ptr(out))
    return out, float(s)


def sync_word_term(w: int, i: int) -> int:
    """The checksum's term for payload word w at word index i."""
    return int(load().oracle_sync_word_term(w & 0xFFFFFFFFFFFFFFFF, i & 0xFFFFFFFFFFFFFFFF))


class _Entry(C.Structure):
    _fields_ = [
        ("tag", C.c_uint64),
        ("kind", C.c_uint32),
        ("recipe", C.c_uint32),
        ("rows", C.c_int64),
        ("cols", C.c_int64),
        ("scale_layout", C.c_uint32),
        ("data", C.c_void_p),
        ("scales", C.c_void_p),
    ]


KIND_FP8, KIND_BF16 = 1, 2
RECIPE_NONE, RECIPE_BLOCKWISE, RECIPE_MX, RECIPE_BLOCKWISE_POW2 = 0, 1, 2, 3
LAYOUT_NONE, LAYOUT_GROUP_1x128, LAYOUT_BLOCK_128x128, LAYOUT_MX_1x32 = 0, 1, 2, 3


def _entries(specs):
    """specs: list of dicts with tag, kind, recipe, rows, cols, layout, data
    (np.uint8 / np.uint16 array) and scales (np array or None)."""
    arr = (_Entry * max(1, len(specs)))()
    keep = []
    for i, s in enumerate(specs):
        data = np.ascontiguousarray(s["data"])
        keep.append(data)
        sc = s.get("scales")
        if sc is not None:
            sc = np.ascontiguousarray(sc)
            keep.append(sc)
        arr[i] = _Entry(s["tag"], s["kind"], s["recipe"], s["rows"], s["cols"], s["layout"],
                        data.ctypes.data, None if sc is None else sc.ctypes.data)
    return arr, keep


def sync_payload_size(specs) -> int:
    arr, _keep = _entries(specs)
    return int(load().oracle_sync_payload_size(arr, len(specs)))


def sync_pack(specs) -> np.ndarray:
    arr, _keep = _entries(specs)
    total = int(load().oracle_sync_payload_size(arr, len(specs)))
    out = np.zeros((total,), np.uint8)
    used = load().oracle_sync_pack(arr, len(specs), _ptr(out), total)
    assert used == total
    return out


def sync_install(payload, dst_specs) -> int:
    """Writes into the dst specs' data/scales arrays (which must be writable,
    C-contiguous numpy arrays).  Returns 0 ok, 1 bad payload, 2 checksum."""
    p = np.ascontiguousarray(payload, np.uint8)
    arr, _keep = _entries(dst_specs)
    for s, k in zip(dst_specs, range(len(dst_specs))):
        assert s["data"].flags["C_CONTIGUOUS"] and s["data"].flags["WRITEABLE"]
    return int(load().oracle_sync_install(_ptr(p), p.size, arr, len(dst_specs)))


def sync_checksum(payload) -> int:
    p = np.ascontiguousarray(payload, np.uint8)
    return int(load().oracle_sync_checksum(_ptr(p), p.size))
