"""GPU parity of fp8_param ("Deep dive: FP8 quantization with FP32 and
power-of-two block scales": the FP8 storage recomputed from the FP32 master
after every optimizer step): the updated master bit for bit and the codes
and scales byte for byte against the oracle, for both scale recipes, with
and without the fused update, with the transposed copy, padded rows, special
values, a multi-step trajectory and the full 12288x4096 weight; then the
Figure 12 displacement measurements on the device."""
import numpy as np
import pytest
import torch

import block_scaled_fp8_e4m3_gb300 as fp8
import oracle
import param_drift
from block_scaled_fp8_e4m3_gb300 import synth
from gpu_util import DEV, assert_bytes_equal, to_np

pytestmark = pytest.mark.gpu


def _check(q, qt, w_ref, pow2, what=""):
    ref = oracle.quant_block_128x128_f32(w_ref, transposed=qt is not None, pow2=pow2)
    got = (q.codes, q.scales) + ((qt.codes, qt.scales) if qt is not None else ())
    for g, r, name in zip(got, ref, ("codes", "scales", "codes^T", "scales^T")):
        assert_bytes_equal(to_np(g), r, f"{what} {name}")


@pytest.mark.parametrize("N,K", [(128, 128), (256, 384), (384, 1024)])
@pytest.mark.parametrize("pow2", [False, True])
@pytest.mark.parametrize("with_delta", [False, True])
def test_parity(N, K, pow2, with_delta):
    w = synth.fp32_master((N, K), seed=N + K)
    d = synth.sign_updates((N, K), seed=N + K + 1, lr=1e-4) if with_delta else None
    m = w.to(DEV)
    q, qt = fp8.param_requantize(m, d.to(DEV) if with_delta else None, transposed=True, pow2=pow2)
    w_ref = oracle.param_update(w.numpy(), d.numpy()) if with_delta else w.numpy()
    assert_bytes_equal(to_np(m), w_ref, "master")
    _check(q, qt, w_ref, pow2, f"{N}x{K}")


@pytest.mark.parametrize("pow2", [False, True])
def test_padded_rows(pow2):
    N, K, ld = 256, 256, 320
    buf = synth.fp32_master((N, ld), seed=40)
    dbuf = synth.sign_updates((N, ld), seed=41, lr=1e-5)
    m, d = buf.to(DEV), dbuf.to(DEV)
    q = fp8.param_requantize(m[:, :K], d[:, :K], pow2=pow2)
    w_ref = oracle.param_update(np.ascontiguousarray(buf.numpy()[:, :K]), np.ascontiguousarray(dbuf.numpy()[:, :K]))
    assert_bytes_equal(to_np(m[:, :K]), w_ref, "master")
    assert_bytes_equal(to_np(m[:, K:]), buf.numpy()[:, K:], "padding columns untouched")
    _check(q, None, w_ref, pow2)


def test_special_values():
    w = torch.zeros((128, 640), dtype=torch.float32)
    w[:, 128:256] = 2.0 ** -146                 # amax / 448 underflows to 0: scale 1
    w[3, 256] = float("inf")
    w[4, 257] = float("nan")
    w[0:2, 384:512] = 1e-3
    w[7, 512:640] = -3.0e38                     # near the top of the fp32 range
    w[8, 520] = 1e-45                           # fp32 subnormal
    for pow2 in (False, True):
        q = fp8.param_requantize(w.to(DEV), pow2=pow2)
        c, s = oracle.quant_block_128x128_f32(w.numpy(), pow2=pow2)
        g = to_np(q.codes)
        # either NaN code for a NaN quotient (its sign is not specified by IEEE 754)
        nan_g, nan_r = (g & 0x7F) == 0x7F, (c & 0x7F) == 0x7F
        assert np.array_equal(nan_g, nan_r)
        assert_bytes_equal(np.where(nan_g, 0x7F, g).astype(np.uint8), np.where(nan_r, 0x7F, c).astype(np.uint8),
                           f"codes pow2={pow2}")
        assert_bytes_equal(to_np(q.scales), s, f"scales pow2={pow2}")


def _midpoint_band(s_target: float, ulps: int = 10) -> np.ndarray:
    """fp32 values at and within `ulps` representable steps of s_target times
    each of the 126 rounding midpoints between adjacent positive E4M3 values,
    with both signs."""
    v = oracle.e4m3_decode(np.arange(127, dtype=np.uint8))          # 0 .. 448, ascending
    base = ((v[:-1] + v[1:]) / 2 * s_target).astype(np.float32).view(np.int32)
    band = np.concatenate([base + k for k in range(-ulps, ulps + 1)]).view(np.float32)
    return np.concatenate([band, -band])


def test_quotients_at_rounding_midpoints():
    """fp32 elements whose quotient by a non-power-of-two block scale falls at
    or beside an E4M3 rounding midpoint: there the product with the reciprocal
    cannot decide the code, and the codes must still be those of the IEEE
    quotient (ties to even)."""
    targets = [1.37, 0.0071, 5.3e4, 3.1e-20, 2.9e15]
    w = np.zeros((128, 128 * len(targets)), np.float32)
    for b, st in enumerate(targets):
        blk = np.zeros(128 * 128, np.float32)
        band = _midpoint_band(st)
        blk[0] = np.float32(448.0 * st)            # the block maximum: s = RN(blk[0] / 448), near st
        blk[1:1 + band.size] = band
        w[:, 128 * b:128 * (b + 1)] = blk.reshape(128, 128)
    q, qt = fp8.param_requantize(torch.from_numpy(w).to(DEV), transposed=True)
    _check(q, qt, w, False, "midpoints")
    # the band reaches both sides of the midpoints, and it separates the IEEE
    # quotient from the plain product with RN(1/s)
    c, sc = oracle.quant_block_128x128_f32(w)
    assert len(np.unique(c)) > 200
    r = np.repeat(np.float32(1) / sc.astype(np.float32), 128, axis=1)
    naive = oracle.e4m3_encode((w * r).astype(np.float32))
    assert (naive != c).any()


@pytest.mark.parametrize("pow2", [False, True])
def test_trajectory(pow2):
    """30 optimizer steps: the master and Q(W_t) match the oracle after each."""
    w = synth.fp32_master((256, 256), seed=50)
    m = w.to(DEV)
    w_ref = w.numpy()
    q = None
    for t in range(30):
        d = synth.sign_updates((256, 256), seed=100 + t, lr=1e-5)
        q = fp8.param_requantize(m, d.to(DEV), out=q, pow2=pow2)
        w_ref = oracle.param_update(w_ref, d.numpy())
        if t % 10 == 9:
            assert_bytes_equal(to_np(m), w_ref, f"master step {t}")
            _check(q, None, w_ref, pow2, f"step {t}")


@pytest.mark.parametrize("pow2", [False, True])
def test_full_weight(pow2):
    wl = synth.fp8_param()
    W, dW = wl.tensors["W"], wl.tensors["dW"]
    m = W.to(DEV)
    q, qt = fp8.param_requantize(m, dW.to(DEV), transposed=True, pow2=pow2)
    w_ref = oracle.param_update(W.numpy(), dW.numpy())
    assert_bytes_equal(to_np(m), w_ref, "master 12288x4096")
    _check(q, qt, w_ref, pow2, "12288x4096")


def test_argument_errors():
    m = torch.zeros((128, 128), dtype=torch.float32, device=DEV)
    with pytest.raises(fp8.FP8Error):
        fp8.param_requantize(torch.zeros((100, 128), dtype=torch.float32, device=DEV))
    with pytest.raises(TypeError):
        fp8.param_requantize(m, torch.zeros((128, 256), dtype=torch.float32, device=DEV)[:, :128])


@pytest.mark.parametrize("pow2", [False, True])
def test_displacement_follows_the_master(pow2):
    """Figure 12, left: after many RL-sized steps the FP8 storage has moved,
    on average, as far as the master along the master's displacement."""
    w0 = synth.fp32_master((1024, 1024), seed=60).to(DEV)
    r = param_drift.cumulative_displacement(w0, steps=400, lr=1e-6, pow2=pow2, seed=61)[400]
    assert 0.9 < r["projection"] < 1.1, r
    assert 0.85 < r["l1"] < 1.35, r


def test_single_step_cosine_grows_with_the_update():
    """Figure 12, right: one RL-sized update barely correlates with the FP8
    change it causes; the correlation approaches 1 for large updates."""
    w = synth.fp32_master((1024, 1024), seed=70).to(DEV)
    for pow2 in (False, True):
        rows = param_drift.single_step_cosine(w, [1e-7, 1e-6, 1e-5, 1e-4, 1e-3, 1e-2], pow2=pow2, seed=71)
        cos = [r["cosine"] for r in rows]
        assert all(b > a for a, b in zip(cos, cos[1:])), cos
        assert cos[1] < 0.1 and cos[-1] > 0.95, cos
