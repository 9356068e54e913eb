"""Pins the oracle GEMM reference: brute-force Python sums, a closed form,
the relation to the unquantized product, and the transpose identities that
tie forward, DGrad and WGrad together."""
import numpy as np

from block_scaled_fp8_e4m3_gb300 import synth


def test_gemm_ref_brute_force(orc):
    rng = np.random.default_rng(3)
    A = rng.standard_normal((3, 7))
    B = rng.standard_normal((5, 7))
    ref, mag = orc.gemm_ref(A, B)
    for m in range(3):
        for n in range(5):
            s = 0.0
            t = 0.0
            for k in range(7):
                s += A[m, k] * B[n, k]
                t += abs(A[m, k] * B[n, k])
            assert abs(ref[m, n] - s) <= 1e-12 * t
            assert abs(mag[m, n] - t) <= 1e-12 * t


def test_gemm_closed_form(orc):
    K = 384
    A = orc.dequant_group(np.full((4, K), 0x38, np.uint8), np.ones((K // 128, 4), np.float32))
    B = orc.dequant_block(np.full((128, K), 0x40, np.uint8), np.ones((1, K // 128), np.float32))
    ref, mag = orc.gemm_ref(A, B)
    assert np.all(ref == 2 * K) and np.all(mag == 2 * K)       # 1.0 * 2.0 summed K times


def test_sampled_equals_full(orc):
    rng = np.random.default_rng(4)
    A = rng.standard_normal((17, 64))
    B = rng.standard_normal((9, 64))
    ref, mag = orc.gemm_ref(A, B)
    ms = rng.integers(0, 17, 40)
    ns = rng.integers(0, 9, 40)
    r2, m2 = orc.gemm_ref_sampled(A, B, ms, ns)
    assert np.array_equal(r2, ref[ms, ns]) and np.array_equal(m2, mag[ms, ns])


def test_quantized_product_close_to_unquantized(orc):
    """|ref - X W^T| is bounded by the per-element quantization errors:
    sum_k |dx||w| + |x||dw| + |dx||dw| with |d| <= 2^-4 |v| (E4M3 half ulp,
    relative) plus the subnormal floor."""
    wl = synth.tiny()
    X, W = wl.tensors["X"], wl.tensors["W"]
    cx, sx = orc.quant_group_1x128(synth.bf16_bits(X))
    cw, sw = orc.quant_block_128x128(synth.bf16_bits(W))
    A, B = orc.dequant_group(cx, sx), orc.dequant_block(cw, sw)
    ref, _ = orc.gemm_ref(A, B)
    x = X.double().numpy()
    w = W.double().numpy()
    exact = x @ w.T
    sxf = np.repeat(sx.T, 128, axis=1)
    swf = np.kron(sw, np.ones((128, 128)))
    dx = 2.0 ** -4 * np.abs(x) + 2.0 ** -10 * sxf
    dw = 2.0 ** -4 * np.abs(w) + 2.0 ** -10 * swf
    bound = dx @ np.abs(w).T + np.abs(x) @ dw.T + dx @ dw.T
    assert np.all(np.abs(ref - exact) <= bound)


def test_dgrad_wgrad_transpose_identities(orc):
    """DGrad dX = dY W and WGrad dW = dY^T X computed as 'TN' products of the
    transposed operands equal the same products written out directly."""
    dY = synth.random_bf16((256, 128), seed=31, std=1e-3)
    W = synth.random_bf16((128, 256), seed=32, std=0.02)     # [N, K]
    X = synth.random_bf16((256, 256), seed=33, outliers=True)
    c_dy, s_dy = orc.quant_group_1x128(synth.bf16_bits(dY))          # [M, N]
    cw, sw, cwt, swt = orc.quant_block_128x128(synth.bf16_bits(W), transposed=True)
    dy_deq = orc.dequant_group(c_dy, s_dy)
    wt_deq = orc.dequant_block(cwt, swt)                              # [K, N]
    dx_ref, dx_mag = orc.gemm_ref(dy_deq, wt_deq)                     # [M, K]
    assert np.all(np.abs(dx_ref - dy_deq @ orc.dequant_block(cw, sw)) <= 1e-12 * dx_mag)
    c_dyt, s_dyt = orc.quant_group_128x1_T(synth.bf16_bits(dY))      # [N, M]
    c_xt, s_xt = orc.quant_group_128x1_T(synth.bf16_bits(X))         # [K, M]
    A = orc.dequant_group(c_dyt, s_dyt)
    B = orc.dequant_group(c_xt, s_xt)
    dw_ref, dw_mag = orc.gemm_ref(A, B)                               # [N, K]
    assert np.all(np.abs(dw_ref - A @ B.T) <= 1e-12 * dw_mag)
