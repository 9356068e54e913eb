"""GPU parity of the blockwise recipe with power-of-two scales: the
quantizers byte for byte against the oracle (codes and E8M0 bytes in the MX
layout), the GEMMs (run on the block-scaled MMA) within |gpu - ref| <=
2e-3 sum|ab| + 2^-8 |ref| of the oracle's fp64 product of the dequantized
operands, the fused quantization of Y, and a weight-sync round trip."""
import numpy as np
import pytest
import torch

import block_scaled_fp8_e4m3_gb300 as fp8
import oracle
from block_scaled_fp8_e4m3_gb300 import synth
from gpu_util import DEV, assert_bytes_equal, assert_gemm_close, bf16_dev_to_f64, sampled_gemm_check, to_np

pytestmark = pytest.mark.gpu


def _o(fn, t, **kw):
    return fn(synth.bf16_bits(t), **kw)


@pytest.mark.parametrize("M,K", [(1, 128), (130, 384), (257, 512), (8192, 4096)])
def test_group_1x128(M, K):
    x = synth.random_bf16((M, K), seed=M + K, outliers=True)
    q = fp8.quantize_group(x.to(DEV), "K", pow2=True)
    c, s = _o(oracle.quant_group_1x128_pow2, x)
    assert q.recipe == fp8.RECIPE_BLOCKWISE_POW2 and q.layout == fp8.LAYOUT_MX_1x32
    assert_bytes_equal(to_np(q.codes), c, "codes")
    assert_bytes_equal(to_np(q.scales), s, "scales")


@pytest.mark.parametrize("M,K", [(128, 8), (256, 392), (8192, 4096)])
def test_group_128x1_transposed(M, K):
    x = synth.random_bf16((M, K), seed=M * 3 + K, outliers=True)
    q = fp8.quantize_group(x.to(DEV), "M", pow2=True)
    c, s = _o(oracle.quant_group_128x1_T_pow2, x)
    assert (q.rows, q.cols) == (K, M)
    assert_bytes_equal(to_np(q.codes), c, "codes")
    assert_bytes_equal(to_np(q.scales), s, "scales")


@pytest.mark.parametrize("N,K", [(128, 128), (256, 384), (12288, 4096)])
def test_block_128x128_with_transpose(N, K):
    w = synth.random_bf16((N, K), seed=N + 7 * K, std=0.02)
    q, qt = fp8.quantize_block(w.to(DEV), transposed=True, pow2=True)
    c, s, ct, st = _o(oracle.quant_block_128x128_pow2, w, transposed=True)
    assert_bytes_equal(to_np(q.codes), c, "codes")
    assert_bytes_equal(to_np(q.scales), s, "scales")
    assert_bytes_equal(to_np(qt.codes), ct, "codes^T")
    assert_bytes_equal(to_np(qt.scales), st, "scales^T")


def test_special_values():
    x = torch.zeros((128, 256), dtype=torch.float32)
    x[0, :] = 0.0                                   # an all-zero group: e = 0
    x[1, 0] = float("inf")
    x[2, 3] = float("nan")
    x[3, :] = -0.0
    x[4, :128] = 1e-38                               # tiny: exponent clamped at -127
    x[5, 0] = 3.0e38
    x[6, 128:] = torch.linspace(-448.0, 448.0, 128)  # amax/448 = 1: e = 0
    x[7, :] = 448.5                                  # rounds up to 2 (bf16 448.0 or 450.0)
    xb = x.to(torch.bfloat16)
    q = fp8.quantize_group(xb.to(DEV), "K", pow2=True)
    c, s = _o(oracle.quant_group_1x128_pow2, xb)
    assert_bytes_equal(to_np(q.codes), c, "codes")
    assert_bytes_equal(to_np(q.scales), s, "scales")
    qb = fp8.quantize_block(xb.to(DEV)[:, :128].contiguous(), pow2=True)
    cb, sb = _o(oracle.quant_block_128x128_pow2, xb[:, :128].contiguous())
    assert_bytes_equal(to_np(qb.codes), cb, "block codes")
    assert_bytes_equal(to_np(qb.scales), sb, "block scales")


def _deq(c, s):
    return oracle.dequant_mx(c, s)


@pytest.mark.parametrize("M,N,K", [(128, 256, 128), (300, 512, 512), (1, 128, 256), (640, 1280, 384)])
def test_gemm_fwd(M, N, K):
    X = synth.random_bf16((M, K), seed=M + N + K + 5, outliers=True)
    W = synth.random_bf16((N, K), seed=M + N + K + 6, std=0.02)
    qx = fp8.quantize_group(X.to(DEV), "K", pow2=True)
    qw = fp8.quantize_block(W.to(DEV), pow2=True)
    Y = fp8.gemm(qx, qw, "fwd")
    ref, mag = oracle.gemm_ref(_deq(*_o(oracle.quant_group_1x128_pow2, X)),
                               _deq(*_o(oracle.quant_block_128x128_pow2, W)))
    assert_gemm_close(bf16_dev_to_f64(Y), ref, mag, f"pow2 fwd {M}x{N}x{K}")


def test_gemm_fwd_fused_quant():
    M, N, K = 260, 512, 640
    X = synth.random_bf16((M, K), seed=91, outliers=True)
    W = synth.random_bf16((N, K), seed=92, std=0.02)
    qx = fp8.quantize_group(X.to(DEV), "K", pow2=True)
    qw = fp8.quantize_block(W.to(DEV), pow2=True)
    Y, qy = fp8.gemm(qx, qw, "fwd", quantize_output=True)
    assert qy.recipe == fp8.RECIPE_BLOCKWISE_POW2
    q2 = fp8.quantize_group(Y, "K", pow2=True)
    assert_bytes_equal(to_np(qy.codes), to_np(q2.codes), "fused codes")
    assert_bytes_equal(to_np(qy.scales), to_np(q2.scales), "fused scales")
    c, s = _o(oracle.quant_group_1x128_pow2, Y.cpu())
    assert_bytes_equal(to_np(qy.codes), c, "fused codes vs oracle")
    assert_bytes_equal(to_np(qy.scales), s, "fused scales vs oracle")


@pytest.mark.parametrize("M,Nw,Kw", [(256, 256, 384), (384, 512, 256)])
def test_gemm_dgrad_wgrad(M, Nw, Kw):
    dY = synth.random_bf16((M, Nw), seed=M + Nw, std=1e-3)
    W = synth.random_bf16((Nw, Kw), seed=Nw + Kw, std=0.02)
    X = synth.random_bf16((M, Kw), seed=M + Kw, outliers=True)
    q_dy = fp8.quantize_group(dY.to(DEV), "K", pow2=True)
    _, q_wt = fp8.quantize_block(W.to(DEV), transposed=True, pow2=True)
    dX = fp8.gemm(q_dy, q_wt, "dgrad")
    _, _, ct, st = _o(oracle.quant_block_128x128_pow2, W, transposed=True)
    ref, mag = oracle.gemm_ref(_deq(*_o(oracle.quant_group_1x128_pow2, dY)), _deq(ct, st))
    assert_gemm_close(bf16_dev_to_f64(dX), ref, mag, "pow2 dgrad")
    q_dyt = fp8.quantize_group(dY.to(DEV), "M", pow2=True)
    q_xt = fp8.quantize_group(X.to(DEV), "M", pow2=True)
    dW = fp8.gemm(q_dyt, q_xt, "wgrad")
    ref, mag = oracle.gemm_ref(_deq(*_o(oracle.quant_group_128x1_T_pow2, dY)),
                               _deq(*_o(oracle.quant_group_128x1_T_pow2, X)))
    assert_gemm_close(bf16_dev_to_f64(dW), ref, mag, "pow2 wgrad")


def test_gemm_full_mlp_sampled():
    """The dense-MLP shape 8192x4096x12288 with power-of-two scales, checked
    on sampled outputs against the oracle's per-element reference."""
    wl = synth.mlp()
    X, W = wl.tensors["X"], wl.tensors["W"]
    qx = fp8.quantize_group(X.to(DEV), "K", pow2=True)
    qw = fp8.quantize_block(W.to(DEV), pow2=True)
    Y = fp8.gemm(qx, qw, "fwd")
    a = _deq(*_o(oracle.quant_group_1x128_pow2, X))
    b = _deq(*_o(oracle.quant_block_128x128_pow2, W))
    sampled_gemm_check(Y, a, b, "pow2 fwd 8192x4096x12288 sampled", seed=12)


def test_sync_round_trip():
    w = synth.random_bf16((384, 512), seed=33, std=0.02)
    q = fp8.quantize_block(w.to(DEV), pow2=True)
    entries = [fp8.SyncEntry(7, q)]
    payload = fp8.sync_pack(entries)
    dst = fp8.QTensor(torch.zeros_like(q.codes), torch.zeros_like(q.scales), q.rows, q.cols, q.recipe, q.layout)
    fp8.sync_install(payload, [fp8.SyncEntry(7, dst)])
    assert torch.equal(dst.codes, q.codes) and torch.equal(dst.scales, q.scales)
    spec = [dict(tag=7, kind=oracle.KIND_FP8, recipe=oracle.RECIPE_BLOCKWISE_POW2, rows=384, cols=512,
                 layout=oracle.LAYOUT_MX_1x32,
                 data=to_np(q.codes), scales=to_np(q.scales))]
    assert_bytes_equal(to_np(payload), oracle.sync_pack(spec), "payload vs oracle")
