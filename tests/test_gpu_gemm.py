"""GPU parity of the block-scaled GEMMs against the oracle's fp64 product of
the dequantized operands, within |gpu - ref| <= 2e-3 sum|ab| + 2^-8 |ref|.
Operands are quantized on the GPU (byte-equal to the oracle, checked in
test_gpu_quant) and independently by the oracle from the same bf16 inputs."""
import numpy as np
import pytest
import torch

import block_scaled_fp8_e4m3_gb300 as fp8
import oracle
from block_scaled_fp8_e4m3_gb300 import synth
from gpu_util import (DEV, assert_bytes_equal, assert_gemm_close, bf16_dev_to_f64, oracle_block, oracle_group_k,
                      oracle_group_m, oracle_mx, sampled_gemm_check, to_np)

pytestmark = pytest.mark.gpu


def _fwd_case(M, N, K, seed):
    X = synth.random_bf16((M, K), seed=seed, outliers=True)
    W = synth.random_bf16((N, K), seed=seed + 1000, std=0.02)
    return X, W


@pytest.mark.parametrize("M,N,K", [(128, 256, 128), (300, 512, 512), (1, 128, 256), (257, 384, 1024),
                                   (640, 1280, 384)])
def test_blockwise_fwd(M, N, K):
    X, W = _fwd_case(M, N, K, seed=M + N + K)
    qx = fp8.quantize_group(X.to(DEV), "K")
    qw = fp8.quantize_block(W.to(DEV))
    Y = fp8.gemm(qx, qw, "fwd")
    cx, sx = oracle_group_k(X)
    cw, sw = oracle_block(W)
    ref, mag = oracle.gemm_ref(oracle.dequant_group(cx, sx), oracle.dequant_block(cw, sw))
    assert_gemm_close(bf16_dev_to_f64(Y), ref, mag, f"fwd {M}x{N}x{K}")


def test_blockwise_fwd_f32_out_and_fused_quant():
    M, N, K = 200, 512, 640
    X, W = _fwd_case(M, N, K, seed=77)
    qx = fp8.quantize_group(X.to(DEV), "K")
    qw = fp8.quantize_block(W.to(DEV))
    Y32 = fp8.gemm(qx, qw, "fwd", out_dtype=torch.float32)
    Y, qy = fp8.gemm(qx, qw, "fwd", quantize_output=True)
    cx, sx = oracle_group_k(X)
    cw, sw = oracle_block(W)
    ref, mag = oracle.gemm_ref(oracle.dequant_group(cx, sx), oracle.dequant_block(cw, sw))
    assert_gemm_close(Y32.double().cpu().numpy(), ref, mag, "fwd f32")
    assert_gemm_close(bf16_dev_to_f64(Y), ref, mag, "fwd bf16")
    # the fused quantization equals the standalone quantizer applied to Y
    q2 = fp8.quantize_group(Y, "K")
    assert_bytes_equal(to_np(qy.codes), to_np(q2.codes), "fused codes")
    assert_bytes_equal(to_np(qy.scales), to_np(q2.scales), "fused scales")
    # and the oracle's quantization of the returned bf16 Y
    c, s = oracle_group_k(Y.cpu())
    assert_bytes_equal(to_np(qy.codes), c, "fused codes vs oracle")


@pytest.mark.parametrize("M,Nw,Kw", [(256, 256, 384), (384, 512, 256)])
def test_dgrad_wgrad(M, Nw, Kw):
    """dX = dY W  (A = dY 1x128, B = W^T 128x128 transposed copy) and
    dW = dY^T X (A = dY^T, B = X^T, both from 128x1 groups)."""
    dY = synth.random_bf16((M, Nw), seed=M + 1, std=1e-3)
    W = synth.random_bf16((Nw, Kw), seed=M + 2, std=0.02)
    X = synth.random_bf16((M, Kw), seed=M + 3, outliers=True)
    q_dy = fp8.quantize_group(dY.to(DEV), "K")
    _, q_wt = fp8.quantize_block(W.to(DEV), transposed=True)
    dX = fp8.gemm(q_dy, q_wt, "dgrad")
    c_dy, s_dy = oracle_group_k(dY)
    _, _, c_wt, s_wt = oracle_block(W, transposed=True)
    ref, mag = oracle.gemm_ref(oracle.dequant_group(c_dy, s_dy), oracle.dequant_block(c_wt, s_wt))
    assert_gemm_close(bf16_dev_to_f64(dX), ref, mag, "dgrad")

    q_dyt = fp8.quantize_group(dY.to(DEV), "M")
    q_xt = fp8.quantize_group(X.to(DEV), "M")
    for dt in (torch.bfloat16, torch.float32):
        dW = fp8.gemm(q_dyt, q_xt, "wgrad", out_dtype=dt)
        c1, s1 = oracle_group_m(dY)
        c2, s2 = oracle_group_m(X)
        ref, mag = oracle.gemm_ref(oracle.dequant_group(c1, s1), oracle.dequant_group(c2, s2))
        assert_gemm_close(dW.double().cpu().numpy(), ref, mag, f"wgrad {dt}")


@pytest.mark.parametrize("M,N,K", [(128, 256, 128), (300, 512, 512), (1, 256, 256), (200, 400, 384),
                                   (513, 1024, 1024)])
def test_mx_fwd(M, N, K):
    X, W = _fwd_case(M, N, K, seed=M * 3 + N + K)
    qx = fp8.quantize_mx(X.to(DEV))
    qw = fp8.quantize_mx(W.to(DEV))
    Y = fp8.gemm(qx, qw, "fwd")
    cx, sx = oracle_mx(X)
    cw, sw = oracle_mx(W)
    ref, mag = oracle.gemm_ref(oracle.dequant_mx(cx, sx), oracle.dequant_mx(cw, sw))
    assert_gemm_close(bf16_dev_to_f64(Y), ref, mag, f"mx {M}x{N}x{K}")


def test_mx_fused_quant():
    M, N, K = 300, 512, 256
    X, W = _fwd_case(M, N, K, seed=91)
    qx = fp8.quantize_mx(X.to(DEV))
    qw = fp8.quantize_mx(W.to(DEV))
    Y, qy = fp8.gemm(qx, qw, "fwd", quantize_output=True)
    q2 = fp8.quantize_mx(Y)
    assert_bytes_equal(to_np(qy.codes), to_np(q2.codes), "fused codes")
    assert_bytes_equal(to_np(qy.scales), to_np(q2.scales), "fused scales")
    # and the oracle's MX 1x32 quantization of the returned bf16 Y
    c, s = oracle_mx(Y.cpu())
    assert_bytes_equal(to_np(qy.codes), c, "fused codes vs oracle")
    assert_bytes_equal(to_np(qy.scales), s, "fused scales vs oracle")


def _mx_row_scales(scales: np.ndarray, rows, K: int) -> np.ndarray:
    """E8M0 bytes [len(rows), K/32] of the given rows, read out of the MX
    scale-factor atom layout of a [R, K] tensor."""
    out = np.empty((len(rows), K // 32), np.uint8)
    for i, r in enumerate(rows):
        for j in range(K // 32):
            out[i, j] = scales[oracle.mx_scale_offset(int(r), j, K)]
    return out


@pytest.mark.parametrize("recipe", ["blockwise", "mx"])
def test_multi_tile_elementwise(recipe):
    """Every output of a GEMM large enough that each CTA pair of the
    persistent grid computes at least three 256x256 tiles (4096x4096: 256
    tiles on at most 76 pairs), against the oracle element by element: the
    TMEM set alternation and barrier phases across tiles are all checked."""
    M, N, K = 4096, 4096, 384 if recipe == "blockwise" else 256
    X, W = _fwd_case(M, N, K, seed=4096 + K)
    if recipe == "blockwise":
        Y = fp8.gemm(fp8.quantize_group(X.to(DEV), "K"), fp8.quantize_block(W.to(DEV)))
        cx, sx = oracle_group_k(X)
        cw, sw = oracle_block(W)
        a, b = oracle.dequant_group(cx, sx), oracle.dequant_block(cw, sw)
    else:
        Y = fp8.gemm(fp8.quantize_mx(X.to(DEV)), fp8.quantize_mx(W.to(DEV)))
        cx, sx = oracle_mx(X)
        cw, sw = oracle_mx(W)
        a, b = oracle.dequant_mx(cx, sx), oracle.dequant_mx(cw, sw)
    ref, mag = oracle.gemm_ref(a, b)
    assert_gemm_close(bf16_dev_to_f64(Y), ref, mag, f"{recipe} {M}x{N}x{K} all outputs")


def test_mx_scale_factors_are_applied_per_row_and_block():
    """Structured operands: A codes all 1.0 with scale 2^(r%7 - 3) varying by
    row and 32-block; B codes 1.0 with scale 2^(n%5 - 2).  D is then a
    closed form sum over blocks of products of powers of two."""
    M, N, K = 256, 256, 256
    a = torch.ones((M, K))
    for kb in range(K // 32):
        a[:, kb * 32:(kb + 1) * 32] *= torch.exp2(((torch.arange(M) + kb) % 7 - 3).float())[:, None]
    b = torch.ones((N, K))
    for kb in range(K // 32):
        b[:, kb * 32:(kb + 1) * 32] *= torch.exp2(((torch.arange(N) * 3 + kb) % 5 - 2).float())[:, None]
    A, B = a.to(torch.bfloat16), b.to(torch.bfloat16)
    Y = fp8.gemm(fp8.quantize_mx(A.to(DEV)), fp8.quantize_mx(B.to(DEV)))
    exact = a.double() @ b.double().T
    assert torch.equal(Y.double().cpu(), exact.to(torch.bfloat16).double())


def test_blockwise_scales_closed_form():
    """Blockwise: every group constant -> D exact: codes 448 at scale amax/448."""
    M, N, K = 256, 256, 512
    a = torch.ones((M, K))
    for g in range(K // 128):
        a[:, g * 128:(g + 1) * 128] *= torch.exp2(((torch.arange(M) + g) % 5 - 2).float())[:, None]
    b = torch.ones((N, K))
    for nb in range(N // 128):
        for kb in range(K // 128):
            b[nb * 128:(nb + 1) * 128, kb * 128:(kb + 1) * 128] *= 2.0 ** ((nb + 2 * kb) % 3 - 1)
    qa = fp8.quantize_group(a.to(torch.bfloat16).to(DEV), "K")
    qb = fp8.quantize_block(b.to(torch.bfloat16).to(DEV))
    Y = fp8.gemm(qa, qb, out_dtype=torch.float32)
    exact = a.double() @ b.double().T
    assert torch.allclose(Y.double().cpu(), exact, rtol=1e-6, atol=0)


# ---------------------------------------------------------------- full size, sampled
def _sampled_check(Y, A_deq, B_deq, what, seed=0):
    """Stratified: the four corners and 12 uniform positions of every 256x256
    output tile (the kernels' tile), against the oracle."""
    sampled_gemm_check(Y, A_deq, B_deq, what, seed=seed)


def test_full_mlp_forward_sampled():
    wl = synth.mlp()
    X, W = wl.tensors["X"], wl.tensors["W"]
    qx = fp8.quantize_group(X.to(DEV), "K")
    qw = fp8.quantize_block(W.to(DEV))
    Y, qy = fp8.gemm(qx, qw, "fwd", quantize_output=True)
    cx, sx = oracle_group_k(X)
    cw, sw = oracle_block(W)
    _sampled_check(Y, oracle.dequant_group(cx, sx), oracle.dequant_block(cw, sw), "mlp fwd 8192x4096x12288")
    q2 = fp8.quantize_group(Y, "K")
    assert torch.equal(qy.codes, q2.codes) and torch.equal(qy.scales, q2.scales)
    # the fused 1x128 quantization of Y against the oracle, on sampled rows
    rows = torch.from_numpy(np.random.default_rng(3).choice(Y.shape[0], 96, replace=False)).to(Y.device)
    c, s_ = oracle_group_k(Y[rows].cpu())
    assert_bytes_equal(to_np(qy.codes[rows]), c, "fused codes, sampled rows")
    assert_bytes_equal(to_np(qy.scales[:, rows].t().contiguous()), np.ascontiguousarray(s_.T), "fused scales, sampled rows")


def test_full_backward_sampled():
    wl = synth.backward()
    dY, W, X = wl.tensors["dY"], wl.tensors["W"], wl.tensors["X"]
    q_dy = fp8.quantize_group(dY.to(DEV), "K")
    _, q_wt = fp8.quantize_block(W.to(DEV), transposed=True)
    dX = fp8.gemm(q_dy, q_wt, "dgrad")
    c_dy, s_dy = oracle_group_k(dY)
    _, _, c_wt, s_wt = oracle_block(W, transposed=True)
    _sampled_check(dX, oracle.dequant_group(c_dy, s_dy), oracle.dequant_block(c_wt, s_wt), "dgrad full")
    q_dyt = fp8.quantize_group(dY.to(DEV), "M")
    q_xt = fp8.quantize_group(X.to(DEV), "M")
    dW = fp8.gemm(q_dyt, q_xt, "wgrad")
    c1, s1 = oracle_group_m(dY)
    c2, s2 = oracle_group_m(X)
    _sampled_check(dW, oracle.dequant_group(c1, s1), oracle.dequant_group(c2, s2), "wgrad full")


def test_full_mx_sampled():
    wl = synth.mx()
    X, W = wl.tensors["X"], wl.tensors["W"]
    Y, qy = fp8.gemm(fp8.quantize_mx(X.to(DEV)), fp8.quantize_mx(W.to(DEV)), quantize_output=True)
    cx, sx = oracle_mx(X)
    cw, sw = oracle_mx(W)
    _sampled_check(Y, oracle.dequant_mx(cx, sx), oracle.dequant_mx(cw, sw), "mx full")
    # the fused MX quantization of Y against the oracle, on sampled rows
    # (including the first and last row of the 128-row scale atoms)
    N = Y.shape[1]
    rows = np.unique(np.concatenate([np.random.default_rng(5).choice(Y.shape[0], 64, replace=False),
                                     [0, 127, 128, Y.shape[0] - 1]]))
    c, s = oracle_mx(Y[torch.from_numpy(rows).to(Y.device)].cpu())
    assert_bytes_equal(to_np(qy.codes)[rows], c, "fused MX codes, sampled rows")
    assert_bytes_equal(_mx_row_scales(to_np(qy.scales), rows, N), _mx_row_scales(s, range(len(rows)), N),
                       "fused MX scales, sampled rows")


def test_zero_rows_and_mismatched_operands():
    """A GEMM over zero rows returns an empty D (and an empty fused
    quantization) for both recipes; operands of different recipes, or a
    blockwise weight whose N is not a multiple of 128, are rejected before
    any launch and leave the device status clean."""
    K, N = 256, 256
    W = synth.random_bf16((N, K), seed=61, std=0.02).to(DEV)
    qw, mw = fp8.quantize_block(W), fp8.quantize_mx(W)
    x0 = torch.empty((0, K), dtype=torch.bfloat16, device=DEV)
    for qa, qb in ((fp8.quantize_group(x0, "K"), qw), (fp8.quantize_mx(x0), mw)):
        assert fp8.gemm(qa, qb).shape == (0, N)
        Y, qy = fp8.gemm(qa, qb, quantize_output=True)
        assert Y.shape == (0, N) and qy.codes.shape == (0, N)
    X = synth.random_bf16((128, K), seed=62).to(DEV)
    qx, mx = fp8.quantize_group(X, "K"), fp8.quantize_mx(X)
    for a, b in ((qx, mw), (mx, qw)):
        with pytest.raises(fp8.FP8Error) as err:
            fp8.gemm(a, b)
        assert err.value.status == 1
    w48 = fp8.quantize_mx(synth.random_bf16((48, K), seed=63, std=0.02).to(DEV))
    qw48 = fp8.QTensor(w48.codes, torch.ones((1, 2), dtype=torch.float32, device=DEV), 48, K,
                       fp8.RECIPE_BLOCKWISE, fp8.LAYOUT_BLOCK_128x128)
    with pytest.raises(fp8.FP8Error) as err:
        fp8.gemm(qx, qw48)
    assert err.value.status == 3
    fp8.status_poll()
    torch.testing.assert_close(fp8.gemm(qx, qw), fp8.gemm(qx, qw))    # still usable afterwards


@pytest.mark.parametrize("recipe", ["blockwise", "pow2", "mx"])
def test_strided_output(recipe):
    """D written into a view with a row pitch above N (912 bytes: 16-byte but
    not 32-byte aligned rows, so the 16-byte store path runs): the same
    values as a contiguous D, the fused quantization unchanged, and the
    padding columns untouched."""
    M, N, K = 300, 384, 512
    X, W = _fwd_case(M, N, K, seed=77)
    if recipe == "mx":
        qa, qb = fp8.quantize_mx(X.to(DEV)), fp8.quantize_mx(W.to(DEV))
    else:
        p2 = recipe == "pow2"
        qa, qb = fp8.quantize_group(X.to(DEV), "K", pow2=p2), fp8.quantize_block(W.to(DEV), pow2=p2)
    Y, qy = fp8.gemm(qa, qb, quantize_output=True)
    buf = torch.full((M, N + 72), 7.0, dtype=torch.bfloat16, device=DEV)
    Yv, qv = fp8.gemm(qa, qb, out=buf[:, :N], quantize_output=True)
    assert Yv.stride(0) == N + 72
    assert torch.equal(Yv, Y)
    assert torch.equal(qv.codes, qy.codes) and torch.equal(qv.scales, qy.scales)
    assert bool((buf[:, N:] == 7.0).all())
    if recipe == "blockwise":
        Yf = fp8.gemm(qa, qb, out_dtype=torch.float32)
        fbuf = torch.full((M, N + 40), 7.0, dtype=torch.float32, device=DEV)
        Yfv = fp8.gemm(qa, qb, out=fbuf[:, :N])
        assert torch.equal(Yfv, Yf) and bool((fbuf[:, N:] == 7.0).all())
