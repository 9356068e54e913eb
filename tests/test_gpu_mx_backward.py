"""GPU parity of the MXFP8 backward path: the 32x1 transposed quantizer byte
for byte against the oracle, and DGrad (dX = dY W with B = W^T) and WGrad
(dW = dY^T X) on the block-scaled MMA within |gpu - ref| <= 2e-3 sum|ab| +
2^-8 |ref| of the oracle's fp64 product of the dequantized operands."""
import numpy as np
import pytest

import block_scaled_fp8_e4m3_gb300 as fp8
import oracle
from block_scaled_fp8_e4m3_gb300 import synth
from gpu_util import DEV, assert_bytes_equal, assert_gemm_close, bf16_dev_to_f64, sampled_gemm_check, to_np

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("R,K", [(128, 8), (256, 200), (384, 1000), (8192, 4096)])
def test_transposed_quantizer(R, K):
    x = synth.random_bf16((R, K), seed=R + 3 * K, outliers=True)
    q = fp8.quantize_mx(x.to(DEV), transposed=True)
    c, s = oracle.quant_mx_32x1_T(synth.bf16_bits(x))
    assert (q.rows, q.cols) == (K, R)
    assert_bytes_equal(to_np(q.codes), c, "codes")
    assert_bytes_equal(to_np(q.scales), s, "scales")


@pytest.mark.parametrize("M,Nw,Kw", [(256, 256, 384), (384, 512, 256), (8192, 4096, 4096)])
def test_dgrad_wgrad(M, Nw, Kw):
    dY = synth.random_bf16((M, Nw), seed=M + Nw + 1, std=1e-3)
    W = synth.random_bf16((Nw, Kw), seed=Nw + Kw + 2, std=0.02)
    X = synth.random_bf16((M, Kw), seed=M + Kw + 3, outliers=True)
    q_dy = fp8.quantize_mx(dY.to(DEV))
    q_wt = fp8.quantize_mx(W.to(DEV), transposed=True)
    dX = fp8.gemm(q_dy, q_wt, "dgrad")
    a = oracle.dequant_mx(*oracle.quant_mx_1x32(synth.bf16_bits(dY)))
    b = oracle.dequant_mx(*oracle.quant_mx_32x1_T(synth.bf16_bits(W)))
    q_dyt = fp8.quantize_mx(dY.to(DEV), transposed=True)
    q_xt = fp8.quantize_mx(X.to(DEV), transposed=True)
    dW = fp8.gemm(q_dyt, q_xt, "wgrad")
    at = oracle.dequant_mx(*oracle.quant_mx_32x1_T(synth.bf16_bits(dY)))
    bt = oracle.dequant_mx(*oracle.quant_mx_32x1_T(synth.bf16_bits(X)))
    if M * Nw * Kw <= 2 ** 27:
        ref, mag = oracle.gemm_ref(a, b)
        assert_gemm_close(bf16_dev_to_f64(dX), ref, mag, f"mx dgrad {M}x{Nw}x{Kw}")
        ref, mag = oracle.gemm_ref(at, bt)
        assert_gemm_close(bf16_dev_to_f64(dW), ref, mag, f"mx wgrad {M}x{Nw}x{Kw}")
    else:
        sampled_gemm_check(dX, a, b, "mx dgrad full sampled", seed=4)
        sampled_gemm_check(dW, at, bt, "mx wgrad full sampled", seed=5)
