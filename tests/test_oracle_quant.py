"""Pins the oracle quantizers: hand-worked groups, brute force on tiny
tensors (independent nearest-value search), and invariants that any slip in
grouping, indexing or scale handling breaks."""
import numpy as np
import pytest
import torch

from block_scaled_fp8_e4m3_gb300 import synth
from conftest import read_golden
from test_oracle_e4m3 import _brute_force_encode

E4M3_MAX = 448.0


def _bits_of(values_f32):
    t = torch.tensor(np.asarray(values_f32, np.float32)).to(torch.bfloat16)
    return synth.bf16_bits(t)


def _ulp_e4m3(v):
    """Spacing of the E4M3 grid at |v| (subnormal spacing 2^-9 below 2^-6)."""
    a = np.abs(v)
    e = np.floor(np.log2(np.maximum(a, 2.0 ** -6)))
    return np.exp2(e - 3)


def _half_ulp_checks(orc, codes, x, s_full):
    """Codes are E4M3(fl32(x / s)): the decoded code is within half an E4M3
    ulp of the fp32 quotient, and the dequantized value is within that plus
    the fp32 rounding of the quotient (2^-24 relative) of x.  The group
    maximum divided by the rounded scale can exceed 448 by an fp32 ulp or
    two, far below the 464 midpoint, so it still encodes to 448."""
    q32 = (x.astype(np.float32) / s_full.astype(np.float32)).astype(np.float64)
    assert np.all(np.abs(q32) <= 448.0 * (1 + 2.0 ** -21))
    dec = orc.e4m3_decode(codes)
    assert np.all(np.abs(dec - q32) <= 0.5 * _ulp_e4m3(q32))
    err = np.abs(dec * s_full - x)
    assert np.all(err <= (0.5 * _ulp_e4m3(x / s_full) + 2.0 ** -24 * np.abs(x / s_full)) * s_full)


# ---------------------------------------------------------------- worked cases
def test_hand_worked_groups(orc):
    for row in read_golden("quant_worked.txt"):
        kind, amax, elem, scale, code = row[0], float(row[1]), float(row[2]), float(row[3]), int(row[4], 16)
        if kind == "group":
            g = np.zeros((1, 128), np.float32)
            g[0, 0] = amax
            g[0, 1] = elem
            codes, scales = orc.quant_group_1x128(_bits_of(g))
            assert scales[0, 0] == np.float32(scale), row
            assert codes[0, 1] == code, row
        else:
            g = np.zeros((1, 32), np.float32)
            g[0, 0] = amax
            g[0, 1] = elem
            codes, scales = orc.quant_mx_1x32(_bits_of(g))
            assert scales[orc.mx_scale_offset(0, 0, 32)] == int(scale), row
            assert codes[0, 1] == code, row


# ---------------------------------------------------------------- brute force
def _brute_group(x_f32, axis_len, along_rows):
    """Independent restatement by loops: for each group find amax, s, codes."""
    M, K = x_f32.shape
    codes = np.zeros((M, K), np.uint8)
    if along_rows:  # 1x128 groups along K
        scales = np.zeros((K // axis_len, M), np.float32)
        for r in range(M):
            for g in range(K // axis_len):
                seg = x_f32[r, g * axis_len:(g + 1) * axis_len]
                amax = np.float32(max(abs(float(v)) for v in seg))
                s = np.float32(1.0) if amax == 0 else np.float32(amax / np.float32(E4M3_MAX))
                scales[g, r] = s
                codes[r, g * axis_len:(g + 1) * axis_len] = _brute_force_encode(
                    (seg / s).astype(np.float32))
    else:           # 128x1 groups along M
        scales = np.zeros((M // axis_len, K), np.float32)
        for c in range(K):
            for b in range(M // axis_len):
                seg = x_f32[b * axis_len:(b + 1) * axis_len, c]
                amax = np.float32(max(abs(float(v)) for v in seg))
                s = np.float32(1.0) if amax == 0 else np.float32(amax / np.float32(E4M3_MAX))
                scales[b, c] = s
                codes[b * axis_len:(b + 1) * axis_len, c] = _brute_force_encode(
                    (seg / s).astype(np.float32))
    return codes, scales


def test_group_1x128_brute_force(orc):
    x = synth.random_bf16((3, 256), seed=11, outliers=True)
    bits = synth.bf16_bits(x)
    xf = x.float().numpy()
    codes, scales = orc.quant_group_1x128(bits)
    bc, bs = _brute_group(xf, 128, along_rows=True)
    assert np.array_equal(scales, bs)
    assert np.array_equal(codes, bc)


def test_group_128x1_brute_force(orc):
    x = synth.random_bf16((256, 3), seed=12, outliers=True)
    bits = synth.bf16_bits(x)
    xf = x.float().numpy()
    codes_t, scales = orc.quant_group_128x1_T(bits)
    bc, bs = _brute_group(xf, 128, along_rows=False)
    assert np.array_equal(scales, bs)
    assert np.array_equal(codes_t, bc.T)


def test_block_128x128_brute_force(orc):
    w = synth.random_bf16((256, 256), seed=13, std=0.02)
    bits = synth.bf16_bits(w)
    wf = w.float().numpy()
    codes, scales, codes_t, scales_t = orc.quant_block_128x128(bits, transposed=True)
    for nb in range(2):
        for kb in range(2):
            blk = wf[nb * 128:(nb + 1) * 128, kb * 128:(kb + 1) * 128]
            amax = np.float32(np.abs(blk).max())
            s = np.float32(amax / np.float32(E4M3_MAX))
            assert scales[nb, kb] == s
            assert scales_t[kb, nb] == s
            exp = _brute_force_encode((blk / s).astype(np.float32))
            assert np.array_equal(codes[nb * 128:(nb + 1) * 128, kb * 128:(kb + 1) * 128], exp)
    assert np.array_equal(codes_t, codes.T)


def test_mx_brute_force(orc):
    x = synth.random_bf16((5, 96), seed=14, outliers=True)
    bits = synth.bf16_bits(x)
    xf = x.float().numpy().astype(np.float64)
    codes, scales = orc.quant_mx_1x32(bits)
    for r in range(5):
        for kb in range(3):
            seg = xf[r, kb * 32:(kb + 1) * 32]
            amax = np.abs(seg).max()
            # floor(log2 amax) by search over powers of two
            E = 0
            while 2.0 ** (E + 1) <= amax:
                E += 1
            while 2.0 ** E > amax:
                E -= 1
            e = max(-127, min(127, E - 8))
            assert scales[orc.mx_scale_offset(r, kb, 96)] == e + 127
            exp = _brute_force_encode((seg * 2.0 ** (-e)).astype(np.float32))
            assert np.array_equal(codes[r, kb * 32:(kb + 1) * 32], exp)


# ---------------------------------------------------------------- invariants
@pytest.fixture(scope="module")
def tiny():
    return synth.tiny()


def test_group_invariants(orc, tiny):
    X = tiny.tensors["X"]
    bits = synth.bf16_bits(X)
    x = X.float().numpy().astype(np.float64)
    codes, scales = orc.quant_group_1x128(bits)
    M, K = x.shape
    deq = orc.dequant_group(codes, scales)
    s_full = np.repeat(scales.T, 128, axis=1).astype(np.float64)           # [M, K]
    _half_ulp_checks(orc, codes, x, s_full)
    # the max element of every group encodes to +-448
    for r in range(M):
        for g in range(K // 128):
            seg = np.abs(x[r, g * 128:(g + 1) * 128])
            j = int(np.argmax(seg))
            assert codes[r, g * 128 + j] & 0x7F == 0x7E
    # re-quantizing the dequantized values with their own scales is identity
    back = (deq.astype(np.float32) / s_full.astype(np.float32)).astype(np.float32)
    assert np.array_equal(orc.e4m3_encode(back), codes)


def test_128x1_is_1x128_of_transpose(orc, tiny):
    X = tiny.tensors["X"]                                 # [128, 512]
    ct, st = orc.quant_group_128x1_T(synth.bf16_bits(X))
    c2, s2 = orc.quant_group_1x128(synth.bf16_bits(X.t().contiguous()))
    assert np.array_equal(ct, c2)
    assert np.array_equal(st, s2)


def test_block_invariants(orc, tiny):
    W = tiny.tensors["W"]
    w = W.float().numpy().astype(np.float64)
    codes, scales, codes_t, scales_t = orc.quant_block_128x128(synth.bf16_bits(W), transposed=True)
    deq = orc.dequant_block(codes, scales)
    s_full = np.kron(scales, np.ones((128, 128))).astype(np.float64)
    _half_ulp_checks(orc, codes, w, s_full)
    assert np.array_equal(codes_t, codes.T) and np.array_equal(scales_t, scales.T)
    assert np.array_equal(orc.dequant_block(codes_t, scales_t), deq.T)
    # block maxima
    for nb in range(4):
        for kb in range(4):
            blk = np.abs(w[nb * 128:(nb + 1) * 128, kb * 128:(kb + 1) * 128])
            i, j = np.unravel_index(int(np.argmax(blk)), blk.shape)
            assert codes[nb * 128 + i, kb * 128 + j] & 0x7F == 0x7E
    back = (deq.astype(np.float32) / s_full.astype(np.float32)).astype(np.float32)
    assert np.array_equal(orc.e4m3_encode(back), codes)


def test_mx_invariants(orc):
    X = synth.random_bf16((200, 160), seed=21, outliers=True)
    x = X.float().numpy().astype(np.float64)
    codes, scales = orc.quant_mx_1x32(synth.bf16_bits(X))
    deq = orc.dequant_mx(codes, scales)
    R, K = x.shape
    e = np.zeros((R, K))
    for r in range(R):
        for kb in range(K // 32):
            e[r, kb * 32:(kb + 1) * 32] = int(scales[orc.mx_scale_offset(r, kb, K)]) - 127
    v = x * np.exp2(-e)
    assert np.all(np.abs(v) < 512)
    sat = np.abs(v) > E4M3_MAX
    # saturated elements decode to +-448 * 2^e; the rest are within half an ulp
    assert np.all(np.abs(deq[sat]) == E4M3_MAX * np.exp2(e[sat]))
    ok = ~sat
    assert np.all(np.abs(deq[ok] - x[ok]) <= 0.5 * _ulp_e4m3(v[ok]) * np.exp2(e[ok]))
    # every block's max lies in [256, 512) after scaling (e = floor(log2 amax) - 8)
    for r in range(R):
        for kb in range(K // 32):
            amax = np.abs(v[r, kb * 32:(kb + 1) * 32]).max()
            assert 256 <= amax < 512
    # re-quantizing with the own scales is identity
    again = orc.e4m3_encode((deq * np.exp2(-e)).astype(np.float32))
    assert np.array_equal(again, codes)


def test_mx_scale_layout_is_a_bijection(orc):
    for R, K in [(128, 128), (256, 384), (200, 96), (1, 32)]:
        size = orc.mx_scale_bytes(R, K)
        seen = np.zeros(size, np.int32)
        for r in range(((R + 127) // 128) * 128):
            for kb in range(((K + 127) // 128) * 4):
                off = orc.mx_scale_offset(r, kb, K)
                assert 0 <= off < size
                seen[off] += 1
        assert np.all(seen == 1)
        # within a 128-row x 4-block atom the 512 bytes are contiguous
        offs = {orc.mx_scale_offset(r, kb, K) // 512 for r in range(128) for kb in range(4)}
        assert len(offs) == 1


def test_mx_zero_block_and_padding(orc):
    x = np.zeros((3, 64), np.float32)
    x[1, 40] = -2.0
    codes, scales = orc.quant_mx_1x32(_bits_of(x))
    assert scales[orc.mx_scale_offset(0, 0, 64)] == 0          # e = -127
    assert scales[orc.mx_scale_offset(1, 1, 64)] == 127 + (1 - 8)
    assert codes[1, 40] == 0xF8                                  # -2 * 2^7 = -256
    assert np.count_nonzero(codes) == 1


# ---------------------------------------------------------------- MX backward operands
def test_mx_32x1_transposed_is_the_1x32_quantization_of_the_transpose(orc):
    x = synth.random_bf16((256, 200), seed=21, outliers=True)
    bits = synth.bf16_bits(x)
    ct, st = orc.quant_mx_32x1_T(bits)
    c2, s2 = orc.quant_mx_1x32(np.ascontiguousarray(bits.T))
    assert ct.shape == (200, 256)
    assert np.array_equal(ct, c2)
    assert np.array_equal(st, s2)


def test_mx_32x1_block_exponent_brute_force(orc):
    # one column: 32-row blocks with known maxima; e = floor(log2 amax) - 8
    x = np.zeros((64, 32), np.float32)
    x[:32, 0] = np.linspace(-3.0, 3.0, 32)      # amax 3 -> e = 1 - 8 = -7
    x[32:, 0] = 1.0                              # amax 1 -> e = -8
    ct, st = orc.quant_mx_32x1_T(_bits_of(x))
    assert st[orc.mx_scale_offset(0, 0, 64)] == 127 - 7
    assert st[orc.mx_scale_offset(0, 1, 64)] == 127 - 8
    v = synth.bf16_bits(torch.tensor(x).to(torch.bfloat16))
    vals = (v.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    assert np.array_equal(ct[0, :32], _brute_force_encode(vals[:32, 0] * 2.0 ** 7))
    assert np.array_equal(ct[0, 32:], _brute_force_encode(vals[32:, 0] * 2.0 ** 8))
