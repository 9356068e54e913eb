"""Pins the oracle's fp8_param step ("Deep dive: FP8 quantization with FP32
and power-of-two block scales": the optimizer updates the FP32 master and
the FP8 storage is recomputed from it each step as Q(W_t)).  The update is
checked against the exact sum, the fp32-input block quantizers against the
already-pinned bf16 ones on bf16-representable values and against an
independent numpy division plus a nearest-value search on full-mantissa
values, and the scale corner cases by their definitions."""
import numpy as np
import pytest
import torch

from block_scaled_fp8_e4m3_gb300 import synth
from test_oracle_e4m3 import _brute_force_encode


def _master(shape, seed, std=0.02):
    return (np.random.default_rng(seed).standard_normal(shape) * std).astype(np.float32)


def test_update_is_the_exact_sum_rounded_to_fp32(orc):
    w = _master((128, 256), 1)
    rng = np.random.default_rng(2)
    d = (rng.choice([-1.0, 1.0], w.shape) * 1e-6 * rng.uniform(0.5, 1.0, w.shape)).astype(np.float32)
    got = orc.param_update(w, d)
    # |d| / |w| >= 2^-29 almost everywhere: the fp64 sum is exact, so its
    # rounding to fp32 is the correctly rounded fp32 sum
    exact = w.astype(np.float64) + d.astype(np.float64)
    assert np.array_equal(got, exact.astype(np.float32))
    assert not np.array_equal(got, w)                  # the update is not lost in the add
    assert np.array_equal(orc.param_update(w, np.zeros_like(w)), w)


@pytest.mark.parametrize("pow2", [False, True])
def test_fp32_quantizer_equals_the_bf16_one_on_bf16_values(orc, pow2):
    x = synth.random_bf16((256, 384), seed=3, outliers=True) * 0.02
    bits = synth.bf16_bits(x)
    w = x.float().numpy()
    got = orc.quant_block_128x128_f32(w, transposed=True, pow2=pow2)
    ref = (orc.quant_block_128x128_pow2 if pow2 else orc.quant_block_128x128)(bits, transposed=True)
    for g, r in zip(got, ref):
        assert np.array_equal(g, r)


def test_fp32_scale_and_codes_full_mantissa(orc):
    w = _master((256, 256), 4)
    w[5, 7] = 0.25                                      # a large outlier in block (0, 0)
    codes, scales = orc.quant_block_128x128_f32(w)
    for nb in range(2):
        for kb in range(2):
            blk = w[128 * nb:128 * (nb + 1), 128 * kb:128 * (kb + 1)]
            s = np.float32(np.abs(blk).max()) / np.float32(448.0)   # numpy's IEEE fp32 division
            assert scales[nb, kb] == s
            q = (blk / s).astype(np.float32)            # fp32 quotients, as the recipe rounds them
            want = _brute_force_encode(q.astype(np.float64))
            assert np.array_equal(codes[128 * nb:128 * (nb + 1), 128 * kb:128 * (kb + 1)], want), (nb, kb)


def test_fp32_scale_is_the_ieee_quotient_for_many_maxima(orc):
    rng = np.random.default_rng(8)
    KB = 96
    w = _master((128, 128 * KB), 9)
    w *= np.repeat(np.exp2(rng.uniform(-30, 30, KB)), 128).astype(np.float32)[None, :]
    _, scales = orc.quant_block_128x128_f32(w)
    amax = np.abs(w).reshape(128, KB, 128).max(axis=(0, 2))
    assert np.array_equal(scales[0], amax.astype(np.float32) / np.float32(448.0))
    # a product with the rounded reciprocal differs for some of them
    assert not np.array_equal(scales[0], amax.astype(np.float32) * np.float32(1.0 / 448.0))


def test_fp32_pow2_codes_full_mantissa(orc):
    w = _master((128, 256), 5)
    codes, scales = orc.quant_block_128x128_f32(w, pow2=True)
    for kb in range(2):
        blk = w[:, 128 * kb:128 * (kb + 1)]
        a = float(np.abs(blk).max())
        e = orc.pow2_exponent(a)
        t = float(np.float32(a) / np.float32(448.0))
        assert 2.0 ** e >= t > 2.0 ** (e - 1)
        assert np.array_equal(codes[:, 128 * kb:128 * (kb + 1)],
                              _brute_force_encode(blk.astype(np.float64) * 2.0 ** -e))
        for r in (0, 31, 32, 127):
            for q in range(4):
                assert scales[orc.mx_scale_offset(r, 4 * kb + q, 256)] == e + 127


def test_requantization_error_does_not_accumulate(orc):
    """Q(W_t) depends only on W_t: after many small updates the FP8 storage
    is exactly the quantization of the current master, and its distance to
    the master stays within half an E4M3 step of each element."""
    w0 = _master((128, 128), 6)
    rng = np.random.default_rng(7)
    w = w0
    for _ in range(20):
        w = orc.param_update(w, (rng.choice([-1.0, 1.0], w.shape) * 1e-4).astype(np.float32))
    c, s = orc.quant_block_128x128_f32(w)
    c_direct, s_direct = orc.quant_block_128x128_f32(w.copy())
    assert np.array_equal(c, c_direct) and np.array_equal(s, s_direct)
    deq = orc.dequant_block(c, s)
    v = np.abs(w.astype(np.float64)) / float(s[0, 0])
    step = np.exp2(np.floor(np.log2(np.maximum(v, 2.0 ** -6))) - 3) * float(s[0, 0])
    # the fp32 quotient adds at most half an fp32 ulp of v to the E4M3 rounding error
    assert np.all(np.abs(deq - w) <= 0.5 * step * (1 + 2.0 ** -20))


def test_scale_corner_cases(orc):
    w = np.zeros((128, 512), np.float32)
    w[:, 128:256] = np.float32(2.0 ** -146)             # amax / 448 underflows to 0 in fp32
    w[3, 256] = np.inf
    w[4, 257] = np.nan
    w[0:2, 384:512] = np.float32(1e-3)
    codes, scales = orc.quant_block_128x128_f32(w)
    assert scales[0, 0] == 1.0 and np.all(codes[:, :128] == 0)       # all-zero block
    assert scales[0, 1] == 1.0 and np.all(codes[:, 128:256] == 0)    # underflowing scale taken as 1
    assert scales[0, 2] == np.inf                                     # inf / 448
    # inf / inf and NaN give NaN codes; IEEE 754 leaves the sign of a NaN
    # produced by an invalid operation unspecified, so either NaN code
    assert codes[3, 256] & 0x7F == 0x7F and codes[4, 257] & 0x7F == 0x7F
    assert codes[5, 256] == 0x00
    assert np.all(codes[0:2, 384:512] == 0x7E)                       # the maximum maps to 448
    c2, s2 = orc.quant_block_128x128_f32(w, pow2=True)
    e_tiny = s2[orc.mx_scale_offset(0, 4, 512)]
    assert e_tiny == 0                                                 # 2^-127 (clamped)
    assert np.all(c2[:, 128:256] == 0)
    assert s2[orc.mx_scale_offset(0, 0, 512)] == 127                  # all-zero: e = 0


@pytest.mark.parametrize("pow2", [False, True])
def test_displacement_projection_is_near_one(orc, pow2):
    """[SkyRL] Figure 12, left, on the oracle: after many lr = 1e-6 sign
    updates the FP8 displacement projected on the master's equals the
    master's displacement on average (no update is systematically lost)."""
    w0 = _master((256, 256), 11)
    rng = np.random.default_rng(12)
    deq = (lambda c, s: orc.dequant_mx(c, s)) if pow2 else (lambda c, s: orc.dequant_block(c, s))
    d0 = deq(*orc.quant_block_128x128_f32(w0, pow2=pow2))
    w = w0
    for _ in range(300):
        w = orc.param_update(w, rng.choice(np.array([-1e-6, 1e-6], np.float32), w.shape))
    D = deq(*orc.quant_block_128x128_f32(w, pow2=pow2)) - d0
    M = w.astype(np.float64) - w0
    assert 0.85 < float((D * M).sum() / (M * M).sum()) < 1.15
