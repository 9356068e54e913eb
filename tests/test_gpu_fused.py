"""GPU parity of the producers fused with the activation quantization
([Jet-RL] "Kwantisatieschema": saved activations stored in FP8, fused with
the previous operator): RMSNorm and SwiGLU.  The bf16 output is within one
bf16 step of the oracle's fp64 producer (the kernel computes in fp32); the
codes and scales are byte-equal to the oracle's quantization of the
kernel's own bf16 output (the quantization decision is taken on the same
bf16 values on both sides), for the three activation recipes."""
import numpy as np
import pytest
import torch

import block_scaled_fp8_e4m3_gb300 as fp8
import oracle
from block_scaled_fp8_e4m3_gb300 import synth
from gpu_util import DEV, assert_bytes_equal, to_np

pytestmark = pytest.mark.gpu

RECIPES = [fp8.RECIPE_BLOCKWISE, fp8.RECIPE_BLOCKWISE_POW2, fp8.RECIPE_MX]


def _oracle_quant(bits, recipe):
    if recipe == fp8.RECIPE_BLOCKWISE:
        return oracle.quant_group_1x128(bits)
    if recipe == fp8.RECIPE_BLOCKWISE_POW2:
        return oracle.quant_group_1x128_pow2(bits)
    return oracle.quant_mx_1x32(bits)


def _f64(bits):
    return (np.asarray(bits, np.uint16).astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def assert_within_one_bf16_step(got_bits, ref_bits, what, max_fraction=1e-3):
    g, r = _f64(got_bits), _f64(ref_bits)
    a = np.abs(r)
    step = np.where(a >= 2.0 ** -126, np.exp2(np.floor(np.log2(np.maximum(a, 2.0 ** -126))) - 7), 2.0 ** -133)
    both_nan = np.isnan(g) & np.isnan(r)
    ok = both_nan | (np.abs(g - r) <= step) | (g == r)
    assert ok.all(), f"{what}: {(~ok).sum()} values beyond one bf16 step, first {np.argwhere(~ok)[:4].tolist()}"
    frac = float((got_bits != ref_bits).mean())
    assert frac <= max_fraction, f"{what}: {frac:.2e} of the values differ by one step"


def _check_codes(q, y_bits, recipe, what):
    c, s = _oracle_quant(y_bits, recipe)
    assert_bytes_equal(to_np(q.codes), c, f"{what} codes")
    assert_bytes_equal(to_np(q.scales), s, f"{what} scales")


@pytest.mark.parametrize("M,K", [(1, 128), (37, 384), (130, 4096), (64, 8192), (9, 640)])
@pytest.mark.parametrize("recipe", RECIPES)
def test_rmsnorm(M, K, recipe):
    x = synth.random_bf16((M, K), seed=M + K, outliers=True)
    g = (synth.random_bf16((K,), seed=K + 1, std=0.2) + 1.0).to(torch.bfloat16)
    q, y, rstd = fp8.rmsnorm_quantize(x.to(DEV), g.to(DEV), 1e-6, recipe, want_y=True, want_rstd=True)
    y_ref, rstd_ref = oracle.rmsnorm(synth.bf16_bits(x), synth.bf16_bits(g), 1e-6)
    assert_within_one_bf16_step(to_np(y), y_ref, f"y {M}x{K}")
    assert np.allclose(to_np(rstd), rstd_ref, rtol=4e-6, atol=0)
    _check_codes(q, to_np(y), recipe, f"rmsnorm {M}x{K}")
    q2 = fp8.rmsnorm_quantize(x.to(DEV), g.to(DEV), 1e-6, recipe)      # no y / rstd outputs: same codes
    assert torch.equal(q2.codes, q.codes) and torch.equal(q2.scales, q.scales)


def test_rmsnorm_full_and_padded():
    M, K, ld = 8192, 4096, 4096 + 64
    x = synth.random_bf16((M, ld), seed=90, outliers=True)
    g = (synth.random_bf16((K,), seed=91, std=0.2) + 1.0).to(torch.bfloat16)
    xd = x.to(DEV)
    q, y = fp8.rmsnorm_quantize(xd[:, :K], g.to(DEV), 1e-6, fp8.RECIPE_BLOCKWISE, want_y=True)
    y_ref, _ = oracle.rmsnorm(synth.bf16_bits(x[:, :K].contiguous()), synth.bf16_bits(g), 1e-6)
    assert_within_one_bf16_step(to_np(y), y_ref, "y 8192x4096")
    _check_codes(q, to_np(y), fp8.RECIPE_BLOCKWISE, "rmsnorm 8192x4096")


def test_rmsnorm_special_rows():
    K = 256
    x = torch.zeros((6, K), dtype=torch.float32)
    x[1] = 1e15                                    # squares summed in fp32: |x| stays below ~1e19
    x[2, 0] = 1e18
    x[3] = torch.linspace(-1e-30, 1e-30, K)
    x[4, :128] = 2.0
    x[5, 7] = -5.0
    xb = x.to(torch.bfloat16)
    g = torch.ones((K,), dtype=torch.bfloat16)
    for recipe in RECIPES:
        q, y = fp8.rmsnorm_quantize(xb.to(DEV), g.to(DEV), 1e-6, recipe, want_y=True)
        y_ref, _ = oracle.rmsnorm(synth.bf16_bits(xb), synth.bf16_bits(g), 1e-6)
        assert_within_one_bf16_step(to_np(y), y_ref, "special y", max_fraction=0.02)
        _check_codes(q, to_np(y), recipe, f"special recipe {recipe}")


@pytest.mark.parametrize("M,F", [(1, 128), (33, 384), (300, 1024)])
@pytest.mark.parametrize("recipe", RECIPES)
def test_swiglu(M, F, recipe):
    gu = synth.random_bf16((M, 2 * F), seed=M * 7 + F, std=2.0, outliers=True)
    q, h = fp8.swiglu_quantize(gu.to(DEV), recipe, want_h=True)
    h_ref = oracle.swiglu(synth.bf16_bits(gu))
    assert_within_one_bf16_step(to_np(h), h_ref, f"h {M}x{F}")
    _check_codes(q, to_np(h), recipe, f"swiglu {M}x{F}")
    q2 = fp8.swiglu_quantize(gu.to(DEV), recipe)
    assert torch.equal(q2.codes, q.codes) and torch.equal(q2.scales, q.scales)


def test_swiglu_full_up_projection():
    """The dense MLP's up projection output 8192x12288 (gate | up) -> 8192x6144."""
    gu = synth.random_bf16((8192, 12288), seed=95, std=1.5)
    for recipe in (fp8.RECIPE_BLOCKWISE, fp8.RECIPE_MX):
        q, h = fp8.swiglu_quantize(gu.to(DEV), recipe, want_h=True)
        h_ref = oracle.swiglu(synth.bf16_bits(gu))
        assert_within_one_bf16_step(to_np(h), h_ref, "h 8192x6144")
        _check_codes(q, to_np(h), recipe, "swiglu 8192x6144")


def test_swiglu_special_values():
    g = torch.tensor([0.0, -0.0, 20.0, -20.0, 87.0, -87.0, 1e-30, -1e-30, 100.0, -3.0] + [0.5] * 118)
    u = torch.tensor([5.0, 2.0, 3.0, 7.0, 1.0, 1.0, 1.0, 1.0, -2.0, 4.0] + [-1.0] * 118)
    gu = torch.cat([g, u])[None, :].repeat(3, 1).to(torch.bfloat16)
    for recipe in RECIPES:
        q, h = fp8.swiglu_quantize(gu.to(DEV), recipe, want_h=True)
        h_ref = oracle.swiglu(synth.bf16_bits(gu))
        assert_within_one_bf16_step(to_np(h), h_ref, "special h", max_fraction=0.05)
        _check_codes(q, to_np(h), recipe, f"swiglu special recipe {recipe}")


def test_empty_and_errors():
    x = torch.empty((0, 256), dtype=torch.bfloat16, device=DEV)
    q = fp8.rmsnorm_quantize(x, torch.ones(256, dtype=torch.bfloat16, device=DEV))
    assert q.codes.numel() == 0
    q = fp8.swiglu_quantize(torch.empty((0, 512), dtype=torch.bfloat16, device=DEV), fp8.RECIPE_MX)
    assert q.codes.numel() == 0
    with pytest.raises(fp8.FP8Error):
        fp8.rmsnorm_quantize(torch.zeros((4, 200), dtype=torch.bfloat16, device=DEV),
                             torch.ones(200, dtype=torch.bfloat16, device=DEV))
    with pytest.raises(fp8.FP8Error):
        fp8.swiglu_quantize(torch.zeros((4, 200), dtype=torch.bfloat16, device=DEV))
    torch.cuda.synchronize()
