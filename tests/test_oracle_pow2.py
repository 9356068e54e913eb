"""Pins the oracle's blockwise recipe with power-of-two scales ("Deep dive:
FP8 quantization with FP32 and power-of-two block scales": on Blackwell the
block scales are powers of two).  The exponent is checked by its defining
property, the codes by an independent nearest-value search, and the layout
by the MX dequantization and by the transpose and cross-recipe identities."""
import numpy as np
import pytest
import torch

from block_scaled_fp8_e4m3_gb300 import synth
from test_oracle_e4m3 import _brute_force_encode


def _bits_of(values_f32):
    t = torch.tensor(np.asarray(values_f32, np.float32)).to(torch.bfloat16)
    return synth.bf16_bits(t)


def _bf16_values(bits):
    return (bits.astype(np.uint32) << 16).view(np.float32)


def test_exponent_is_the_smallest_power_of_two_not_below_the_fp32_scale(orc):
    rng = np.random.default_rng(5)
    # every positive finite bf16 value as a group maximum, plus zero
    amax = _bf16_values(np.arange(1, 0x7F80, dtype=np.uint16))
    for a in amax[rng.choice(amax.size, 4000, replace=False)].tolist() + [448.0, 449.0, 224.0, 1.0, 0.0]:
        e = orc.pow2_exponent(a)
        if a == 0.0:
            assert e == 0
            continue
        t = float(np.float32(a) / np.float32(448.0))  # the fp32 recipe's scale
        if -127 < e < 127:
            assert 2.0 ** e >= t and 2.0 ** (e - 1) < t, (a, e)
        elif e == -127:
            assert t <= 2.0 ** -127, (a, e)
        else:
            assert t > 2.0 ** 126, (a, e)


def test_codes_equal_the_fp32_recipe_when_its_scale_is_a_power_of_two(orc):
    # amax = 448 * 2^k makes amax/448 = 2^k exactly: both recipes divide by
    # the same scale (one by an IEEE division, the other by an exact product)
    rng = np.random.default_rng(6)
    for k in (-20, -3, 0, 5):
        x = (rng.standard_normal((4, 128)) * 2.0 ** k).astype(np.float32)
        x[:, 0] = 448.0 * 2.0 ** k
        bits = _bits_of(x)
        c_p2, s_p2 = orc.quant_group_1x128_pow2(bits)
        c_f32, s_f32 = orc.quant_group_1x128(bits)
        assert np.array_equal(c_p2, c_f32)
        assert np.all(s_f32 == np.float32(2.0 ** k))
        for r in range(4):
            assert s_p2[orc.mx_scale_offset(r, 0, 128)] == k + 127


def test_group_codes_brute_force(orc):
    rng = np.random.default_rng(7)
    x = rng.standard_normal((3, 256)).astype(np.float32) * np.array([[1e-3], [1.0], [300.0]], np.float32)
    x[1, 5] = 0.0
    x[2, 129] = -0.0
    bits = _bits_of(x)
    xv = _bf16_values(bits)
    codes, scales = orc.quant_group_1x128_pow2(bits)
    for r in range(3):
        for g in range(2):
            grp = xv[r, 128 * g:128 * (g + 1)].astype(np.float64)
            e = orc.pow2_exponent(float(np.abs(grp).max()))
            want = _brute_force_encode(grp * 2.0 ** -e)
            assert np.array_equal(codes[r, 128 * g:128 * (g + 1)], want), (r, g)
            # the group's exponent byte in all four 1x32 slots it covers
            for b in range(4):
                assert scales[orc.mx_scale_offset(r, 4 * g + b, 256)] == e + 127
            # no element saturates: max|x| / 2^e <= 448
            assert np.abs(grp).max() * 2.0 ** -e <= 448.0


def test_mx_dequantization_is_codes_times_the_power_of_two(orc):
    wl = synth.tiny()
    bits = synth.bf16_bits(wl.tensors["X"])
    codes, scales = orc.quant_group_1x128_pow2(bits)
    deq = orc.dequant_mx(codes, scales)
    xv = _bf16_values(bits).astype(np.float64)
    M, K = bits.shape
    for r in range(0, M, 17):
        for g in range(K // 128):
            e = orc.pow2_exponent(float(np.abs(xv[r, 128 * g:128 * (g + 1)]).max()))
            dec = orc.e4m3_decode(codes[r, 128 * g:128 * (g + 1)])
            assert np.array_equal(deq[r, 128 * g:128 * (g + 1)], dec * 2.0 ** e)
            # within half an E4M3 step of x (no fp32 rounding: the product is exact)
            step = np.exp2(np.floor(np.log2(np.maximum(np.abs(xv[r, 128 * g:128 * (g + 1)]) * 2.0 ** -e,
                                                       2.0 ** -6))) - 3)
            assert np.all(np.abs(dec * 2.0 ** e - xv[r, 128 * g:128 * (g + 1)]) <= 0.5 * step * 2.0 ** e)


def test_128x1_is_the_1x128_quantization_of_the_transpose(orc):
    x = synth.random_bf16((256, 384), seed=8)
    bits = synth.bf16_bits(x)
    ct, st = orc.quant_group_128x1_T_pow2(bits)
    c2, s2 = orc.quant_group_1x128_pow2(np.ascontiguousarray(bits.T))
    assert np.array_equal(ct, c2)
    assert np.array_equal(st, s2)


@pytest.mark.parametrize("shape", [(256, 256), (128, 384)])
def test_block_128x128(orc, shape):
    w = synth.random_bf16(shape, seed=9) * 0.02
    bits = synth.bf16_bits(w)
    N, K = shape
    codes, scales, codes_t, scales_t = orc.quant_block_128x128_pow2(bits, transposed=True)
    wv = _bf16_values(bits).astype(np.float64)
    assert np.array_equal(codes_t, codes.T)
    for nb in range(N // 128):
        for kb in range(K // 128):
            blk = wv[128 * nb:128 * (nb + 1), 128 * kb:128 * (kb + 1)]
            e = orc.pow2_exponent(float(np.abs(blk).max()))
            assert np.array_equal(codes[128 * nb:128 * (nb + 1), 128 * kb:128 * (kb + 1)],
                                  _brute_force_encode(blk * 2.0 ** -e))
            for i in range(0, 128, 31):
                for q in range(4):
                    assert scales[orc.mx_scale_offset(128 * nb + i, 4 * kb + q, K)] == e + 127
                    assert scales_t[orc.mx_scale_offset(128 * kb + i, 4 * nb + q, N)] == e + 127
    # the plain block quantizer without the transposed copy writes the same
    c1, s1 = orc.quant_block_128x128_pow2(bits)
    assert np.array_equal(c1, codes) and np.array_equal(s1, scales)


def test_gemm_reference_of_pow2_operands_is_the_blockwise_formula(orc):
    # Y = sum_kb sa(m,kb) sb(n,kb) sum_k qa qb with power-of-two scales, in
    # plain Python floats on a tiny case, against gemm_ref of the MX dequants
    x = synth.random_bf16((128, 256), seed=10)
    w = synth.random_bf16((128, 256), seed=11) * 0.02
    ca, sa = orc.quant_group_1x128_pow2(synth.bf16_bits(x))
    cb, sb = orc.quant_block_128x128_pow2(synth.bf16_bits(w))
    ref, _ = orc.gemm_ref(orc.dequant_mx(ca, sa), orc.dequant_mx(cb, sb))
    da, db = orc.e4m3_decode(ca), orc.e4m3_decode(cb)
    for m, n in ((0, 0), (5, 77), (127, 127)):
        total = 0.0
        for kb in range(2):
            ea = int(sa[orc.mx_scale_offset(m, 4 * kb, 256)]) - 127
            eb = int(sb[orc.mx_scale_offset(n, 4 * kb, 256)]) - 127
            part = sum(float(da[m, k]) * float(db[n, k]) for k in range(128 * kb, 128 * (kb + 1)))
            total += part * 2.0 ** (ea + eb)
        assert ref[m, n] == pytest.approx(total, rel=1e-12, abs=1e-30)
