"""Host-side checks of the C ABI (no GPU needed): the library builds and
loads, exports every function include/fp8bs.h declares, and rejects bad
arguments before touching the device."""
import ctypes as C
import os
import re

import pytest

import block_scaled_fp8_e4m3_gb300 as fp8

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    from block_scaled_fp8_e4m3_gb300 import _build
    _build.build()
    return fp8.library()


def _declared_functions():
    src = open(os.path.join(ROOT, "include", "fp8bs.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"^\s*(?:fp8_status|int64_t|int32_t|const char\*)\s+(fp8_\w+)\s*\(", src, re.M)))


def test_exports_every_declared_symbol(lib):
    names = _declared_functions()
    assert len(names) >= 14
    for n in names:
        assert hasattr(lib, n), n


def test_abi_version(lib):
    assert lib.fp8_abi_version() == 1


def test_scale_buffer_sizes(lib):
    assert fp8.mx_scale_bytes(128, 128) == 512
    assert fp8.mx_scale_bytes(129, 32) == 2 * 512
    assert fp8.mx_scale_bytes(2048, 4096) == 16 * 32 * 512
    assert fp8.mx_grouped_scale_bytes(300, 256, 3) == (3 + 3) * 2 * 512


def _t(rows, cols, recipe, layout, codes=0x10000, scales=0x20000):
    return fp8._Tensor(codes, scales, rows, cols, recipe, layout)


@pytest.mark.parametrize("case,expect", [
    ("group_k_bad_K", 3), ("group_m_bad_M", 3), ("block_bad_N", 3), ("mx_bad_K", 3),
    ("misaligned", 2), ("bad_ld", 1), ("wrong_layout", 1), ("wrong_shape", 1), ("null_out", 1),
    ("gemm_bad_K", 3), ("gemm_K_mismatch", 1), ("gemm_bad_N", 3),
    ("mx_t_bad_R", 3), ("mx_t_wrong_shape", 1),
    ("param_bad_N", 3), ("param_bad_ld", 2), ("param_wrong_recipe", 1),
])
def test_argument_validation_happens_on_host(lib, case, expect):
    x = 0x100000                                   # never dereferenced: validation fails first
    s = None
    if case == "group_k_bad_K":
        t = _t(4, 100, 1, 1)
        st = lib.fp8_quantize_group(x, 4, 100, 100 + 4, 0, C.byref(t), s)
    elif case == "group_m_bad_M":
        t = _t(256, 100, 1, 1)
        st = lib.fp8_quantize_group(x, 100, 256, 256, 1, C.byref(t), s)
    elif case == "block_bad_N":
        t = _t(100, 128, 1, 2)
        st = lib.fp8_quantize_block(x, 100, 128, 128, C.byref(t), None, s)
    elif case == "mx_bad_K":
        t = _t(4, 40, 2, 3)
        st = lib.fp8_quantize_mx(x, 4, 40, 40, C.byref(t), s)
    elif case == "mx_t_bad_R":
        t = _t(64, 100, 2, 3)
        st = lib.fp8_quantize_mx_transposed(x, 100, 64, 64, C.byref(t), s)
    elif case == "mx_t_wrong_shape":
        t = _t(128, 64, 2, 3)                      # must be (K, R) = (64, 128)
        st = lib.fp8_quantize_mx_transposed(x, 128, 64, 64, C.byref(t), s)
    elif case == "param_bad_N":
        t = _t(100, 128, 1, 2)
        st = lib.fp8_param_requantize(x, None, 100, 128, 128, C.byref(t), None, s)
    elif case == "param_bad_ld":
        t = _t(128, 128, 1, 2)
        st = lib.fp8_param_requantize(x, None, 128, 128, 130, C.byref(t), None, s)
    elif case == "param_wrong_recipe":
        t = _t(128, 128, 2, 3)                     # MXFP8 is not an fp8_param recipe
        st = lib.fp8_param_requantize(x, x, 128, 128, 128, C.byref(t), None, s)
    elif case == "misaligned":
        t = _t(4, 128, 1, 1)
        st = lib.fp8_quantize_group(x + 2, 4, 128, 128, 0, C.byref(t), s)
    elif case == "bad_ld":
        t = _t(4, 128, 1, 1)
        st = lib.fp8_quantize_group(x, 4, 128, 64, 0, C.byref(t), s)
    elif case == "wrong_layout":
        t = _t(4, 128, 1, 2)
        st = lib.fp8_quantize_group(x, 4, 128, 128, 0, C.byref(t), s)
    elif case == "wrong_shape":
        t = _t(5, 128, 1, 1)
        st = lib.fp8_quantize_group(x, 4, 128, 128, 0, C.byref(t), s)
    elif case == "null_out":
        st = lib.fp8_quantize_group(x, 4, 128, 128, 0, None, s)
    elif case == "gemm_bad_K":
        a, b = _t(4, 100, 1, 1), _t(128, 100, 1, 2)
        st = lib.fp8_gemm_blockscaled(C.byref(a), C.byref(b), x, 128, 0, 0, None, s)
    elif case == "gemm_K_mismatch":
        a, b = _t(4, 128, 1, 1), _t(128, 256, 1, 2)
        st = lib.fp8_gemm_blockscaled(C.byref(a), C.byref(b), x, 128, 0, 0, None, s)
    elif case == "gemm_bad_N":
        a, b = _t(4, 128, 1, 1), _t(100, 128, 1, 2)
        st = lib.fp8_gemm_blockscaled(C.byref(a), C.byref(b), x, 128, 0, 0, None, s)
    assert st == expect, lib.fp8_last_error()
    assert len(lib.fp8_last_error()) > 0


def test_sync_payload_size_matches_oracle(lib, orc):
    """The library's payload layout (host computation) equals the oracle's."""
    from block_scaled_fp8_e4m3_gb300 import synth
    specs = [(0x1, 1, 1, 256, 384, 2), (0x2, 1, 1, 130, 256, 1), (0x3, 1, 2, 100, 96, 3), (0x4, 2, 0, 3, 70, 0)]
    arr = (fp8._SyncEntry * 4)()
    oracle_specs = []
    import numpy as np
    for i, (tag, kind, recipe, r, c, layout) in enumerate(specs):
        arr[i] = fp8._SyncEntry(tag, kind, 0, fp8._Tensor(0x1000, 0x2000 if kind == 1 else None, r, c,
                                                         recipe, layout))
        oracle_specs.append(dict(tag=tag, kind=kind, recipe=recipe, rows=r, cols=c, layout=layout,
                                 data=np.zeros(1, np.uint8), scales=None))
    n = C.c_uint64(0)
    assert lib.fp8_sync_payload_size(arr, 4, C.byref(n)) == 0
    assert n.value == orc.sync_payload_size(oracle_specs)
