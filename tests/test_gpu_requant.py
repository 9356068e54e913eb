"""GPU parity of the WGrad operand built from a saved 1x128 FP8 activation:
codes and scales byte-equal to the oracle (fp32 dequantization, then the
128x1 transposed quantization), at small ragged sizes and at full size, and
WGrad on that operand within the GEMM tolerance."""
import numpy as np
import pytest
import torch

import block_scaled_fp8_e4m3_gb300 as fp8
import oracle
from block_scaled_fp8_e4m3_gb300 import synth
from gpu_util import DEV, assert_bytes_equal, assert_gemm_close, bf16_dev_to_f64, to_np

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("M,K", [(128, 128), (256, 384), (384, 1024), (8192, 4096)])
def test_requantize_transposed(M, K):
    x = synth.random_bf16((M, K), seed=M + 5 * K, outliers=True)
    q = fp8.quantize_group(x.to(DEV), "K")
    qt = fp8.requantize_transposed(q)
    c, s = oracle.quant_group_1x128(synth.bf16_bits(x))
    ct, st = oracle.requant_1x128_to_128x1_T(c, s)
    assert (qt.rows, qt.cols) == (K, M)
    assert_bytes_equal(to_np(qt.codes), ct, "codes^T")
    assert_bytes_equal(to_np(qt.scales), st, "scales")


def test_zero_and_tiny_groups():
    x = torch.zeros((256, 256), dtype=torch.float32)
    x[:, 128:] = torch.linspace(-1e-30, 1e-30, 128)
    x[0:128, 5] = 3.0e30
    xb = x.to(torch.bfloat16)
    q = fp8.quantize_group(xb.to(DEV), "K")
    qt = fp8.requantize_transposed(q)
    c, s = oracle.quant_group_1x128(synth.bf16_bits(xb))
    ct, st = oracle.requant_1x128_to_128x1_T(c, s)
    assert_bytes_equal(to_np(qt.codes), ct, "codes^T")
    assert_bytes_equal(to_np(qt.scales), st, "scales")


def test_wgrad_on_the_requantized_operand():
    M, Nw, Kw = 384, 256, 512
    dY = synth.random_bf16((M, Nw), seed=31, std=1e-3)
    X = synth.random_bf16((M, Kw), seed=32, outliers=True)
    q_dyt = fp8.quantize_group(dY.to(DEV), "M")
    q_xt = fp8.requantize_transposed(fp8.quantize_group(X.to(DEV), "K"))
    dW = fp8.gemm(q_dyt, q_xt, "wgrad")
    c1, s1 = oracle.quant_group_128x1_T(synth.bf16_bits(dY))
    cx, sx = oracle.quant_group_1x128(synth.bf16_bits(X))
    c2, s2 = oracle.requant_1x128_to_128x1_T(cx, sx)
    ref, mag = oracle.gemm_ref(oracle.dequant_group(c1, s1), oracle.dequant_group(c2, s2))
    assert_gemm_close(bf16_dev_to_f64(dW), ref, mag, "wgrad on the re-quantized X")
