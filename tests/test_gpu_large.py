"""Maximum sizes: tensors of more than 2^31 elements, so that every 64-bit
offset in the kernels is exercised.  Inputs are drawn on the device from a
seeded CUDA generator (only the sampled rows travel to the host); the
sampled rows -- including the last ones -- are checked against the oracle
byte for byte (quantizers) or within the GEMM tolerance."""
import numpy as np
import pytest
import torch

import block_scaled_fp8_e4m3_gb300 as fp8
import oracle
from block_scaled_fp8_e4m3_gb300 import synth
from gpu_util import DEV, assert_bytes_equal, assert_gemm_close, to_np

pytestmark = pytest.mark.gpu


def _device_bf16(shape, seed, std=1.0):
    g = torch.Generator(device=DEV)
    g.manual_seed(seed)
    return (torch.randn(shape, device=DEV, generator=g) * std).to(torch.bfloat16)


def _bits(t):
    return synth.bf16_bits(t.cpu())


@pytest.fixture(autouse=True)
def _free():
    yield
    torch.cuda.empty_cache()


def test_group_1x128_and_mx_beyond_2_31():
    M, K = 65552, 32768                                  # 2.148e9 elements
    x = _device_bf16((M, K), 1)
    rows = torch.tensor([0, 1, 40000, M - 2, M - 1], device=DEV)
    q = fp8.quantize_group(x, "K")
    c, s = oracle.quant_group_1x128(_bits(x[rows]))
    assert_bytes_equal(to_np(q.codes[rows]), c, "1x128 codes, sampled rows")
    assert_bytes_equal(to_np(q.scales[:, rows].t().contiguous()), np.ascontiguousarray(s.T), "1x128 scales")
    del q
    qm = fp8.quantize_mx(x)
    c, s = oracle.quant_mx_1x32(_bits(x[rows]))
    assert_bytes_equal(to_np(qm.codes[rows]), c, "MX codes, sampled rows")
    sc = to_np(qm.scales)
    for i, r in enumerate(rows.tolist()):
        got = np.array([sc[oracle.mx_scale_offset(r, kb, K)] for kb in range(0, K // 32, 97)])
        want = np.array([s[oracle.mx_scale_offset(i, kb, K)] for kb in range(0, K // 32, 97)])
        assert np.array_equal(got, want), r


def test_group_128x1_transposed_beyond_2_31():
    M, K = 65536, 32784                                  # codes^T [32784][65536]: offsets past 2^31
    x = _device_bf16((M, K), 2)
    q = fp8.quantize_group(x, "M")
    cols = torch.tensor([0, 7, 20000, K - 1], device=DEV)
    for mb in (0, M // 128 - 1):
        blk = x[128 * mb:128 * (mb + 1)][:, cols].contiguous()
        c, s = oracle.quant_group_128x1_T(_bits(blk))    # codes^T [len(cols)][128]
        assert_bytes_equal(to_np(q.codes[cols, 128 * mb:128 * (mb + 1)]), c, f"128x1 codes, block {mb}")
        assert_bytes_equal(to_np(q.scales[mb, cols]), s[0], f"128x1 scales, block {mb}")


def test_block_128x128_beyond_2_31():
    N, K = 65536, 32896
    w = _device_bf16((N, K), 3, std=0.02)
    q = fp8.quantize_block(w)
    for nb in (0, N // 128 - 1):
        blk = w[128 * nb:128 * (nb + 1)]
        c, s = oracle.quant_block_128x128(_bits(blk))
        assert_bytes_equal(to_np(q.codes[128 * nb:128 * (nb + 1)]), c, f"block row {nb} codes")
        assert_bytes_equal(to_np(q.scales[nb]), s[0], f"block row {nb} scales")


def test_blockwise_gemm_with_a_beyond_2_31():
    M, K, N = 524416, 4096, 256                          # A codes: 2.148e9 bytes
    x = _device_bf16((M, K), 4)
    w = _device_bf16((N, K), 5, std=0.02)
    qx = fp8.quantize_group(x, "K")
    del x
    qw = fp8.quantize_block(w)
    Y = fp8.gemm(qx, qw, "fwd")
    rows = torch.tensor([0, 300000, M - 1], device=DEV)
    a = oracle.dequant_group(to_np(qx.codes[rows]), to_np(qx.scales[:, rows].contiguous()))
    cw, sw = oracle.quant_block_128x128(_bits(w))
    ref, mag = oracle.gemm_ref(a, oracle.dequant_block(cw, sw))
    assert_gemm_close(Y[rows].double().cpu().numpy(), ref, mag, "rows of a 524416x4096x256 GEMM")
