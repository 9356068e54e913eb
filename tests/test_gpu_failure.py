"""Failure detection without a GPU fault: a bounded on-device wait whose
peer never signals gives up after its limit, records FP8_ERR_TIMEOUT in the
status block, and leaves the context usable."""
import pytest
import torch

import block_scaled_fp8_e4m3_gb300 as fp8
import oracle
from block_scaled_fp8_e4m3_gb300 import synth
from gpu_util import DEV, assert_bytes_equal, to_np

pytestmark = pytest.mark.gpu


def test_expired_wait_is_reported_and_the_context_stays_usable():
    fp8.status_poll()                                    # start clean
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    fp8.check_wait_expiry(20_000_000)                    # 20 ms
    e1.record()
    with pytest.raises(fp8.FP8Error) as ei:
        fp8.status_poll()
    assert ei.value.status == 6                          # FP8_ERR_TIMEOUT
    assert e0.elapsed_time(e1) >= 19.0                   # it really waited for its limit
    fp8.status_poll()                                    # the error was reported once and cleared
    # the context still computes correctly
    x = synth.random_bf16((256, 384), seed=12, outliers=True)
    q = fp8.quantize_group(x.to(DEV), "K")
    c, s = oracle.quant_group_1x128(synth.bf16_bits(x))
    assert_bytes_equal(to_np(q.codes), c, "codes after the expired wait")
    w = synth.random_bf16((256, 384), seed=13, std=0.02)
    y = fp8.gemm(q, fp8.quantize_block(w.to(DEV)))
    assert torch.isfinite(y.float()).all()
    fp8.status_poll()


def test_limit_is_checked_on_the_host():
    with pytest.raises(fp8.FP8Error):
        fp8.check_wait_expiry(10)
