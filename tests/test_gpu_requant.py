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


def test_quotients_at_rounding_midpoints():
    """Dequantized values x' whose quotient by the (non-power-of-two) 128x1
    scale lies at or within 10 ulps of an E4M3 rounding midpoint: the codes of
    the IEEE quotient, byte for byte.  Block b of 128 rows shifts every row
    scale by b - 10 ulps; row 0 of each block sets the column maxima."""
    v = oracle.e4m3_decode(np.arange(127, dtype=np.uint8))
    mids = (v[:-1] + v[1:]) / 2                                   # 126 midpoints
    sc = 7.77
    blocks = 21
    M, K = 128 * blocks, 256
    e = -(np.arange(K) % 7)                                       # column j holds +-2^e, e in [-6, 0]
    col_codes = ((e + 7) << 3).astype(np.uint8) | np.where(np.arange(K) % 2 == 1, 0x80, 0).astype(np.uint8)
    codes = np.zeros((M, K), np.uint8)
    srow = np.ones((K // 128, M), np.float32)
    for b in range(blocks):
        r0 = 128 * b
        codes[r0] = 0x7E                                          # 448 * 7.77: the column maximum
        srow[:, r0] = np.float32(sc)
        s_mid = ((mids * sc).astype(np.float32).view(np.int32) + (b - 10)).view(np.float32)
        codes[r0 + 1:r0 + 127] = col_codes
        srow[:, r0 + 1:r0 + 127] = s_mid
    q = fp8.QTensor(torch.from_numpy(codes).to(DEV), torch.from_numpy(srow).to(DEV), M, K, fp8.RECIPE_BLOCKWISE,
                    fp8.LAYOUT_GROUP_1x128)
    qt = fp8.requantize_transposed(q)
    ct, st = oracle.requant_1x128_to_128x1_T(codes, srow)
    assert_bytes_equal(to_np(qt.codes), ct, "codes^T")
    assert_bytes_equal(to_np(qt.scales), st, "scales")
    assert len(np.unique(ct)) > 200
    # the inputs do separate the IEEE quotient from the plain product with RN(1/s)
    xd = (oracle.e4m3_decode(codes).astype(np.float32) * srow[0][:, None]).astype(np.float32)
    naive = oracle.e4m3_encode((xd * np.repeat(np.float32(1) / st, 128, axis=0)).astype(np.float32))
    assert (naive.T != ct).any()


def test_random_row_scales_full_significands():
    """Saved codes with arbitrary fp32 row scales (full significands,
    log-uniform over 2^-24..2^24, so every quotient x' / s has a full
    significand too) and all finite codes: codes and scales byte-equal to the
    oracle over 2048 x 1024, which spans 16 x 16 tiles of the kernel."""
    rng = np.random.default_rng(1234)
    M, K = 2048, 1024
    codes = rng.integers(0, 256, size=(M, K), dtype=np.uint8)
    codes[(codes & 0x7F) == 0x7F] ^= 0x01                        # no NaN codes: 0x7F -> 0x7E
    srow = np.exp2(rng.uniform(-24.0, 24.0, size=(K // 128, M))).astype(np.float32)
    q = fp8.QTensor(torch.from_numpy(codes).to(DEV), torch.from_numpy(srow).to(DEV), M, K, fp8.RECIPE_BLOCKWISE,
                    fp8.LAYOUT_GROUP_1x128)
    qt = fp8.requantize_transposed(q)
    ct, st = oracle.requant_1x128_to_128x1_T(codes, srow)
    assert_bytes_equal(to_np(qt.codes), ct, "codes^T")
    assert_bytes_equal(to_np(qt.scales), st, "scales")


def test_nan_codes_in_the_saved_activation():
    """E4M3 NaN codes (0x7F, 0xFF) in the saved activation: as documented
    for fp8_requantize_transposed, each gives a NaN code (either sign) at its
    transposed position and stays out of its group's scale; every other code
    and every scale equals the oracle's."""
    x = synth.random_bf16((256, 256), seed=91, outliers=True)
    q = fp8.quantize_group(x.to(DEV), "K")
    codes = to_np(q.codes).copy()
    rng = np.random.default_rng(92)
    pos = rng.choice(codes.size, size=40, replace=False)
    codes.flat[pos[:20]] = 0x7F
    codes.flat[pos[20:]] = 0xFF
    srow = to_np(q.scales)
    qn = fp8.QTensor(torch.from_numpy(codes).to(DEV), torch.from_numpy(srow).to(DEV), 256, 256, fp8.RECIPE_BLOCKWISE,
                     fp8.LAYOUT_GROUP_1x128)
    qt = fp8.requantize_transposed(qn)
    ct, st = oracle.requant_1x128_to_128x1_T(codes, srow)
    got = to_np(qt.codes)
    nan_g, nan_r = (got & 0x7F) == 0x7F, (ct & 0x7F) == 0x7F
    assert np.array_equal(nan_g, nan_r)
    assert nan_g.sum() == 40
    assert_bytes_equal(np.where(nan_g, 0x7F, got).astype(np.uint8), np.where(nan_r, 0x7F, ct).astype(np.uint8),
                       "codes^T outside the NaN positions")
    assert_bytes_equal(to_np(qt.scales), st, "scales")
