"""Pins the oracle's E4M3 codec to things other than itself: a library cast,
brute-force nearest-value search, hand-derived encodings and the softmax
worked example of the AIS explainer page."""
import math

import numpy as np
import pytest
import torch

from conftest import read_golden


def _torch_decode_all():
    codes = torch.arange(256, dtype=torch.uint8)
    return codes.view(torch.float8_e4m3fn).to(torch.float64).numpy()


def test_decode_matches_library_cast(orc):
    ours = orc.e4m3_decode(np.arange(256, dtype=np.uint8))
    ref = _torch_decode_all()
    nan = np.isnan(ref)
    assert list(np.nonzero(nan)[0]) == [0x7F, 0xFF]
    assert np.array_equal(np.isnan(ours), nan)
    assert np.array_equal(ours[~nan], ref[~nan])
    # sign of zero
    assert math.copysign(1.0, ours[0x80]) == -1.0


def test_round_trip_all_finite_codes(orc):
    codes = np.array([c for c in range(256) if c not in (0x7F, 0xFF)], dtype=np.uint8)
    vals = orc.e4m3_decode(codes).astype(np.float32)
    assert np.array_equal(orc.e4m3_encode(vals), codes)
    # NaN codes decode to NaN and re-encode to NaN
    assert orc.e4m3_encode(np.array([np.nan], np.float32))[0] == 0x7F


def _brute_force_encode(v: np.ndarray) -> np.ndarray:
    """Nearest finite E4M3 value by exhaustive search over the 127
    non-negative finite codes (decoded by the library cast), ties to the even
    code, magnitudes above 448 saturated, sign copied."""
    table = _torch_decode_all()[:0x7F]             # codes 0x00..0x7E, ascending
    a = np.abs(v.astype(np.float64))
    out = np.empty(v.shape, np.uint8)
    idx = np.searchsorted(table, a)                # table[idx-1] < a <= table[idx]
    for i in range(a.size):
        x = a.flat[i]
        if not np.isfinite(x) or x >= 448.0:
            code = 0x7E
        else:
            j = idx.flat[i]
            lo, hi = j - 1, j
            if hi <= 0:
                code = 0
            else:
                dlo, dhi = x - table[lo], table[hi] - x
                if dlo < dhi:
                    code = lo
                elif dhi < dlo:
                    code = hi
                else:
                    code = lo if lo % 2 == 0 else hi
        sign = 0x80 if math.copysign(1.0, float(v.flat[i])) < 0 else 0
        out.flat[i] = code | sign
    return out


def test_encode_brute_force_every_bf16_value(orc):
    bits = np.arange(65536, dtype=np.uint32) << 16
    vals = bits.view(np.float32)
    vals = vals[~np.isnan(vals)]
    assert np.array_equal(orc.e4m3_encode(vals), _brute_force_encode(vals))


def test_encode_brute_force_midpoints_and_neighbours(orc):
    table = _torch_decode_all()[:0x7F]
    mids = ((table[:-1] + table[1:]) / 2).astype(np.float32)
    extra = np.array([448.0, 464.0, 479.0, 480.0, 2.0 ** -10, 2.0 ** -11, 1e-45], np.float32)
    base = np.concatenate([mids, extra])
    nb = []
    for d in (-2, -1, 0, 1, 2):
        nb.append(np.nextafter(base, np.float32(np.inf) if d > 0 else np.float32(0))
                  if d != 0 else base)
        if abs(d) == 2:
            nb[-1] = np.nextafter(nb[-1], np.float32(np.inf) if d > 0 else np.float32(0))
    v = np.concatenate(nb).astype(np.float32)
    v = np.concatenate([v, -v])
    assert np.array_equal(orc.e4m3_encode(v), _brute_force_encode(v))


def test_encode_brute_force_random_fp32(orc):
    rng = np.random.default_rng(1234)
    v = (rng.standard_normal(20000) * np.exp2(rng.integers(-14, 11, 20000))).astype(np.float32)
    assert np.array_equal(orc.e4m3_encode(v), _brute_force_encode(v))


def test_encode_matches_library_cast_in_range(orc):
    rng = np.random.default_rng(7)
    v = (rng.standard_normal(200000) * 60).astype(np.float32)
    v = v[np.abs(v) <= 448]
    lib = torch.from_numpy(v).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(orc.e4m3_encode(v), lib)


def test_encode_hand_worked(orc):
    for row in read_golden("e4m3_worked.txt"):
        value, code = float(row[0]), int(row[1], 16)
        assert orc.e4m3_encode_exact(value) == code, row
        assert orc.e4m3_encode(np.array([value], np.float32))[0] == code, row


def test_softmax_worked_example(orc):
    """The explainer's FP8 logits are the round-to-nearest-even E4M3 codes of
    the BF16 logits at scale 1, and its probabilities are the softmax of the
    printed logits."""
    rows = read_golden("softmax_example.txt")
    bf16_logits = np.array([float(r[1]) for r in rows])
    bf16_pct = np.array([float(r[2]) for r in rows])
    fp8_logits = np.array([float(r[3]) for r in rows])
    fp8_pct = np.array([float(r[4]) for r in rows])
    # encoding of the logits (as decimals and as their bf16 roundings)
    for src in (bf16_logits.astype(np.float32),
                torch.tensor(bf16_logits, dtype=torch.float32).to(torch.bfloat16)
                .to(torch.float32).numpy()):
        codes = orc.e4m3_encode(src)
        assert np.array_equal(orc.e4m3_decode(codes), fp8_logits)

    def softmax(z):
        e = np.exp(z - z.max())
        return e / e.sum()

    assert np.array_equal(np.round(100 * softmax(bf16_logits), 2), bf16_pct)
    assert np.array_equal(np.round(100 * softmax(fp8_logits), 2), fp8_pct)
    # log-prob gap of token A between the two sides
    gap = math.log(softmax(fp8_logits)[0]) - math.log(softmax(bf16_logits)[0])
    assert gap == pytest.approx(math.log(0.3402 / 0.3535), abs=5e-4)


def test_sequence_probability_example():
    """Same page: 0.99 ** 1000 is about 4.3e-5."""
    assert round(0.99 ** 1000 / 1e-5, 1) == 4.3
