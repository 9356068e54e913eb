"""Pins the oracle's re-quantization of a saved 1x128 FP8 activation into
the 128x1 WGrad operand ([Jet-RL] "Kwantisatieschema": saved activations in
FP8; WGrad operands in 128x1 groups): against the pinned bf16 128x1
quantizer where the dequantized values are exactly bf16, and against numpy
fp32 arithmetic plus a nearest-value search in general."""
import numpy as np
import torch

from block_scaled_fp8_e4m3_gb300 import synth
from test_oracle_e4m3 import _brute_force_encode


def test_equals_the_bf16_quantizer_when_scales_are_powers_of_two(orc):
    rng = np.random.default_rng(1)
    M, K = 256, 384
    codes = rng.integers(0, 256, (M, K), dtype=np.uint8)
    codes[(codes & 0x7F) == 0x7F] = 0x10                  # no NaN codes
    scales = np.exp2(rng.integers(-20, 5, (K // 128, M))).astype(np.float32)
    ct, st = orc.requant_1x128_to_128x1_T(codes, scales)
    # dec(q) * 2^k has at most 4 significant bits: exactly a bf16 value
    deq = orc.dequant_group(codes, scales)
    bits = torch.from_numpy(deq.astype(np.float32)).to(torch.bfloat16)
    assert np.array_equal(bits.double().numpy(), deq)
    c2, s2 = orc.quant_group_128x1_T(synth.bf16_bits(bits))
    assert np.array_equal(ct, c2) and np.array_equal(st, s2)


def test_general_scales_against_numpy_and_a_nearest_search(orc):
    x = synth.random_bf16((256, 256), seed=2, outliers=True)
    codes, scales = orc.quant_group_1x128(synth.bf16_bits(x))
    ct, st = orc.requant_1x128_to_128x1_T(codes, scales)
    dec = orc.e4m3_decode(codes)
    srow = np.repeat(scales.T, 128, axis=1)               # [M, K] row scales
    deq = (dec * srow.astype(np.float64)).astype(np.float32)   # one rounding to fp32
    for b in range(2):
        blk = deq[128 * b:128 * (b + 1)]                  # [128, K]
        s = np.abs(blk).max(axis=0).astype(np.float32) / np.float32(448.0)
        s = np.where(s == 0, np.float32(1.0), s).astype(np.float32)
        assert np.array_equal(st[b], s)
        q = (blk / s[None, :]).astype(np.float32)         # numpy's IEEE fp32 division
        want = _brute_force_encode(q.astype(np.float64)).T
        assert np.array_equal(ct[:, 128 * b:128 * (b + 1)], want), b


def test_second_quantization_moves_each_element_by_at_most_half_a_step(orc):
    x = synth.random_bf16((256, 128), seed=3, outliers=True)
    codes, scales = orc.quant_group_1x128(synth.bf16_bits(x))
    ct, st = orc.requant_1x128_to_128x1_T(codes, scales)
    d1 = orc.dequant_group(codes, scales)                 # [M, K], the saved activation
    d1f = d1.astype(np.float32).astype(np.float64)        # its fp32 rounding, the re-quantizer's input
    d2 = orc.dequant_group(ct, st).T                      # [M, K], the WGrad operand
    s2 = np.repeat(st, 128, axis=0).astype(np.float64)    # [M, K] scale of each element's 128x1 group
    v = np.abs(d1f) / s2
    step = np.exp2(np.floor(np.log2(np.maximum(v, 2.0 ** -6))) - 3)
    # half an E4M3 step of the scaled value, plus the fp32 rounding of the quotient
    assert np.all(np.abs(d2 - d1f) <= (0.5 * step + v * 2.0 ** -23) * s2)
    # each 128x1 group's maximum lands on +-448
    assert np.all(np.abs(orc.e4m3_decode(ct)).reshape(128, 2, 128).max(axis=2) == 448.0)
