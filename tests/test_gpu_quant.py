"""GPU parity of the quantizers: codes and scales byte-identical to the
oracle on seeded inputs, small ragged cases through the full-size workloads."""
import numpy as np
import pytest
import torch

import block_scaled_fp8_e4m3_gb300 as fp8
from block_scaled_fp8_e4m3_gb300 import synth
from gpu_util import (DEV, assert_bytes_equal, oracle_block, oracle_group_k, oracle_group_m, oracle_mx, to_np)

pytestmark = pytest.mark.gpu


def _dev(x):
    return x.to(DEV)


@pytest.mark.parametrize("shape,seed", [((1, 128), 1), ((17, 256), 2), ((300, 640), 3), ((1000, 384), 4)])
def test_group_k_small(shape, seed):
    x = synth.random_bf16(shape, seed=seed, outliers=True)
    q = fp8.quantize_group(_dev(x), "K")
    codes, scales = oracle_group_k(x)
    assert_bytes_equal(to_np(q.codes), codes, "codes")
    assert_bytes_equal(to_np(q.scales), scales, "scales")


@pytest.mark.parametrize("shape,seed", [((128, 8), 5), ((256, 200), 6), ((384, 520), 7)])
def test_group_m_small(shape, seed):
    x = synth.random_bf16(shape, seed=seed, outliers=True)
    q = fp8.quantize_group(_dev(x), "M")
    codes_t, scales = oracle_group_m(x)
    assert_bytes_equal(to_np(q.codes), codes_t, "codes^T")
    assert_bytes_equal(to_np(q.scales), scales, "scales")


@pytest.mark.parametrize("shape,seed", [((128, 128), 8), ((384, 640), 9)])
def test_block_small(shape, seed):
    w = synth.random_bf16(shape, seed=seed, std=0.02)
    q, qt = fp8.quantize_block(_dev(w), transposed=True)
    c, s, ct, st = oracle_block(w, transposed=True)
    assert_bytes_equal(to_np(q.codes), c, "codes")
    assert_bytes_equal(to_np(q.scales), s, "scales")
    assert_bytes_equal(to_np(qt.codes), ct, "codes^T")
    assert_bytes_equal(to_np(qt.scales), st, "scales^T")
    q2 = fp8.quantize_block(_dev(w))
    assert_bytes_equal(to_np(q2.codes), c, "codes without transpose")


@pytest.mark.parametrize("shape,seed", [((1, 32), 10), ((5, 96), 11), ((130, 160), 12), ((513, 2048), 13)])
def test_mx_small(shape, seed):
    x = synth.random_bf16(shape, seed=seed, outliers=True)
    q = fp8.quantize_mx(_dev(x))
    codes, scales = oracle_mx(x)
    assert_bytes_equal(to_np(q.codes), codes, "codes")
    assert_bytes_equal(to_np(q.scales), scales, "scales")


def test_special_values():
    """Zero groups, negative zeros, subnormal bf16 inputs, huge values, a
    group whose maximum is negative."""
    x = torch.zeros((130, 256), dtype=torch.float32)
    x[1, :128] = -0.0
    x[2, 5] = -3.0
    x[2, 6] = 1.0
    x[3, :] = torch.linspace(-1e-38, 1e-38, 256)        # bf16 subnormals
    x[4, :] = torch.linspace(-3e38, 3e38, 256)
    x[5, 0] = 1e-30
    x[5, 1] = 1e30
    x = x.to(torch.bfloat16)
    for fn, orc in ((lambda t: fp8.quantize_group(t, "K"), oracle_group_k), (fp8.quantize_mx, oracle_mx)):
        q = fn(_dev(x))
        c, s = orc(x)
        assert_bytes_equal(to_np(q.codes), c, "codes")
        assert_bytes_equal(to_np(q.scales), s, "scales")
    xm = x[:128].contiguous()
    q = fp8.quantize_group(_dev(xm), "M")
    c, s = oracle_group_m(xm)
    assert_bytes_equal(to_np(q.codes), c, "codes^T")
    assert_bytes_equal(to_np(q.scales), s, "scales")


def test_empty_inputs():
    x = torch.empty((0, 256), dtype=torch.bfloat16, device=DEV)
    q = fp8.quantize_group(x, "K")
    assert q.codes.numel() == 0
    q = fp8.quantize_mx(x)
    assert q.codes.numel() == 0
    torch.cuda.synchronize()


def test_strided_input():
    base = synth.random_bf16((64, 1024), seed=14, outliers=True)
    view = _dev(base)[:, 256:768]                          # ld = 1024, 512 columns
    q = fp8.quantize_group(view, "K")
    c, s = oracle_group_k(base[:, 256:768].contiguous())
    assert_bytes_equal(to_np(q.codes), c, "codes")
    assert_bytes_equal(to_np(q.scales), s, "scales")


# ---------------------------------------------------------------- full size
@pytest.fixture(scope="module")
def mlp():
    return synth.mlp()


def test_full_mlp_activation_1x128(mlp):
    X = mlp.tensors["X"]
    q = fp8.quantize_group(_dev(X), "K")
    c, s = oracle_group_k(X)
    assert_bytes_equal(to_np(q.codes), c, "codes")
    assert_bytes_equal(to_np(q.scales), s, "scales")


def test_full_mlp_weight_128x128(mlp):
    W = mlp.tensors["W"]
    q, qt = fp8.quantize_block(_dev(W), transposed=True)
    c, s, ct, st = oracle_block(W, transposed=True)
    assert_bytes_equal(to_np(q.codes), c, "codes")
    assert_bytes_equal(to_np(q.scales), s, "scales")
    assert_bytes_equal(to_np(qt.codes), ct, "codes^T")


def test_full_backward_128x1():
    wl = synth.backward()
    for name in ("dY", "X"):
        t = wl.tensors[name]
        q = fp8.quantize_group(_dev(t), "M")
        c, s = oracle_group_m(t)
        assert_bytes_equal(to_np(q.codes), c, f"{name} codes^T")
        assert_bytes_equal(to_np(q.scales), s, f"{name} scales")


def test_full_mx():
    wl = synth.mx()
    for name in ("X", "W"):
        t = wl.tensors[name]
        q = fp8.quantize_mx(_dev(t))
        c, s = oracle_mx(t)
        assert_bytes_equal(to_np(q.codes), c, f"{name} codes")
        assert_bytes_equal(to_np(q.scales), s, f"{name} scales")
