"""Pins the oracle's fused producers ([Jet-RL] "Kwantisatieschema": saved
activations stored in FP8, fused with the previous operator; "Implementatie":
fused activation / RMSNorm kernels): the fp64 -> bf16 rounding against a
nearest-value search over every bf16 value and against torch's fp32 -> bf16
cast, RMSNorm and SwiGLU against torch's float64 functional ops rounded by
that search, and their invariants."""
import numpy as np
import pytest
import torch
import torch.nn.functional as Fn

from block_scaled_fp8_e4m3_gb300 import synth


def _bf16_table():
    """(values, codes) of every non-negative finite bf16, ascending, plus
    2^128 standing for +inf (the even neighbour of the largest finite)."""
    codes = np.arange(0, 0x7F80, dtype=np.uint16)
    vals = (codes.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    return np.append(vals, 2.0 ** 128), np.append(codes, np.uint16(0x7F80))


def _brute_force_bf16(v):
    vals, codes = _bf16_table()
    v = np.asarray(v, np.float64)
    a = np.abs(v)
    out = np.empty(v.shape, np.uint16)
    idx = np.searchsorted(vals, a)
    for i in range(a.size):
        x = a.flat[i]
        j = idx.flat[i]
        if j == 0:
            c = 0
        elif j >= vals.size:
            c = 0x7F80
        else:
            dlo, dhi = x - vals[j - 1], vals[j] - x
            if dlo < dhi:
                c = codes[j - 1]
            elif dhi < dlo:
                c = codes[j]
            else:
                c = codes[j - 1] if codes[j - 1] % 2 == 0 else codes[j]
        out.flat[i] = c | (0x8000 if np.signbit(v.flat[i]) else 0)
    return out


def _f64(bits):
    return (np.asarray(bits, np.uint16).astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def test_bf16_round_brute_force(orc):
    rng = np.random.default_rng(1)
    vals, _ = _bf16_table()
    fin = vals[:-1]
    mids = (fin[:-1] + fin[1:]) / 2                       # exact in fp64: ties
    pick = rng.choice(mids.size, 3000, replace=False)
    v = np.concatenate([fin[rng.choice(fin.size, 2000, replace=False)], mids[pick],
                        np.nextafter(mids[pick], 0), np.nextafter(mids[pick], np.inf),
                        rng.standard_normal(2000) * np.exp2(rng.uniform(-140, 128, 2000)),
                        [0.0, 2.0 ** -133, 2.0 ** -134, 1.5 * 2.0 ** -134, 3.0e38, 3.3961e38, 3.4e38, 1e300]])
    v = np.concatenate([v, -v])
    assert np.array_equal(orc.bf16_round(v), _brute_force_bf16(v))


def test_bf16_round_equals_torch_cast_of_fp32(orc):
    rng = np.random.default_rng(2)
    f = (rng.standard_normal(5000) * np.exp2(rng.uniform(-130, 120, 5000))).astype(np.float32)
    want = torch.from_numpy(f).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(orc.bf16_round(f.astype(np.float64)), want)


def test_rmsnorm_against_torch_float64(orc):
    x = synth.random_bf16((64, 512), seed=3, outliers=True)
    g = synth.random_bf16((512,), seed=4, std=0.5) + 1.0
    eps = 1e-6
    y, rstd = orc.rmsnorm(synth.bf16_bits(x), synth.bf16_bits(g.to(torch.bfloat16)), eps)
    x64, g64 = x.double(), g.to(torch.bfloat16).double()
    ref = Fn.rms_norm(x64, (512,), g64, eps=float(np.float32(eps))).numpy()
    assert np.array_equal(y, _brute_force_bf16(ref))
    r = torch.rsqrt(x64.pow(2).mean(-1) + float(np.float32(eps))).numpy()
    assert np.array_equal(rstd, r.astype(np.float32))


def test_rmsnorm_invariants(orc):
    x = synth.random_bf16((16, 256), seed=5)
    ones = np.full(256, 0x3F80, np.uint16)
    y1, _ = orc.rmsnorm(synth.bf16_bits(x), ones, 0.0)
    y2, _ = orc.rmsnorm(synth.bf16_bits(x * 8.0), ones, 0.0)   # scale invariance (exact powers of two)
    assert np.array_equal(y1, y2)
    ms = (_f64(y1) ** 2).mean(axis=1)
    assert np.all(np.abs(ms - 1.0) < 2 ** -7)                   # unit RMS up to the bf16 rounding
    yc, rc = orc.rmsnorm(np.full((1, 128), 0x4040, np.uint16), ones[:128], 0.0)   # x = 3: y = 1
    assert np.all(yc == 0x3F80) and rc[0] == np.float32(1.0 / 3.0)


def test_swiglu_against_torch_float64(orc):
    gu = synth.random_bf16((32, 2 * 384), seed=6, std=3.0)
    h = orc.swiglu(synth.bf16_bits(gu))
    g, u = gu[:, :384].double(), gu[:, 384:].double()
    assert np.array_equal(h, _brute_force_bf16((Fn.silu(g) * u).numpy()))


def test_swiglu_special_cases(orc):
    g = np.array([0.0, 100.0, -100.0, -0.0, 1.0], np.float32)
    u = np.array([5.0, 3.0, 7.0, 2.0, 1.0], np.float32)
    gu = torch.from_numpy(np.concatenate([g, u])[None, :]).to(torch.bfloat16)
    h = _f64(orc.swiglu(synth.bf16_bits(gu)))[0]
    assert h[0] == 0.0 and h[1] == 300.0 and h[3] == 0.0
    assert 0 < -h[2] < 1e-40 or h[2] == 0.0                     # silu(-100) * 7 ~ -2.6e-42: bf16 0 or subnormal
    assert h[4] == _f64(_brute_force_bf16([1.0 / (1.0 + np.exp(-1.0))]))[0]
