"""CPU check of the quantizer kernels' fast quotient path: where the kernel
keeps y = RN(x * RN(1/s)) instead of the IEEE quotient RN(x/s), both must
encode to the same E4M3 code.  The predicate below restates the kernels'
test (|y| in [2^-5, 512] and the 20 mantissa bits below the 3 kept ones outside
[-4, +3] ulps of the midpoint pattern 0x80000)."""
import numpy as np

import oracle


def needs_exact(y: np.ndarray) -> np.ndarray:
    a = (y.view(np.uint32) & np.uint32(0x7FFFFFFF)).astype(np.int64)
    out_of_range = (a < 0x3D000000) | (a > 0x44000000)
    low = a & 0xFFFFF
    return (a != 0) & (out_of_range | ((low >= 0x80000 - 4) & (low <= 0x80000 + 3)))


def test_fast_path_agrees_with_ieee_division():
    rng = np.random.default_rng(2024)
    bits = (np.arange(1 << 16, dtype=np.uint32) << 16)
    xs_all = bits.view(np.float32)
    xs_all = xs_all[np.isfinite(xs_all)]
    checked = kept = 0
    for _ in range(300):
        # a group maximum (any bf16 magnitude), its scale, and every bf16 value
        # within the group's range
        amax = np.float32(abs(xs_all[rng.integers(0, xs_all.size)]))
        if amax == 0:
            continue
        s = np.float32(amax / np.float32(448.0))
        r = np.float32(np.float32(1.0) / s)
        xs = xs_all[np.abs(xs_all) <= amax]
        with np.errstate(over="ignore", invalid="ignore"):
            q = (xs / s).astype(np.float32)
            y = (xs * r).astype(np.float32)
        fast = ~needs_exact(y)
        kept += int(fast.sum())
        checked += xs.size
        assert np.array_equal(oracle.e4m3_encode(y[fast]), oracle.e4m3_encode(q[fast]))
    assert kept > 0


def test_fast_path_is_the_common_case_for_gaussian_groups():
    rng = np.random.default_rng(7)
    x = rng.standard_normal((4096, 128)).astype(np.float32)
    amax = np.abs(x).max(axis=1, keepdims=True)
    s = (amax / np.float32(448.0)).astype(np.float32)
    r = (np.float32(1.0) / s).astype(np.float32)
    y = (x * r).astype(np.float32)
    q = (x / s).astype(np.float32)
    fast = ~needs_exact(y)
    assert fast.mean() > 0.99
    assert np.array_equal(oracle.e4m3_encode(y[fast]), oracle.e4m3_encode(q[fast]))


def test_fast_path_near_midpoints():
    """Quotients placed right at E4M3 midpoints: any y within 4 ulps of one
    must take the exact path."""
    mids = (oracle.e4m3_decode(np.arange(0x08, 0x7E, dtype=np.uint8)) +
            oracle.e4m3_decode(np.arange(0x09, 0x7F, dtype=np.uint8))) / 2
    mids = mids.astype(np.float32)
    for d in range(-4, 4):
        y = (mids.view(np.uint32).astype(np.int64) + d).astype(np.uint32).view(np.float32)
        big = np.abs(y) >= 2.0 ** -5
        assert needs_exact(y[big]).all()
