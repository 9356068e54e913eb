"""The whole hot path as one CUDA graph: quantize X (1x128), quantize W
(128x128), the blockwise GEMM with the fused quantization of Y, sync pack
and sync install are captured once and replayed on new inputs.  Every call
is device work only (the pack writes the payload header from a kernel
parameter), so the replay must give, byte for byte, what the eager calls
give on the same inputs, and the installed weights must equal the
trainer's."""
import pytest
import torch

import block_scaled_fp8_e4m3_gb300 as fp8
from block_scaled_fp8_e4m3_gb300 import synth
from gpu_util import DEV

pytestmark = pytest.mark.gpu


def _zeros_like(q):
    return fp8.QTensor(torch.zeros_like(q.codes), torch.zeros_like(q.scales), q.rows, q.cols, q.recipe, q.layout)


def test_tiny_step_replays_as_one_graph():
    wl = synth.tiny()
    X, W = wl.tensors["X"].to(DEV), wl.tensors["W"].to(DEV)
    X2 = synth.random_bf16(tuple(X.shape), seed=91, outliers=True).to(DEV)
    W2 = synth.random_bf16(tuple(W.shape), seed=92, std=0.02).to(DEV)

    # eager reference on the second inputs
    rx, rw = fp8.quantize_group(X2, "K"), fp8.quantize_block(W2)
    rY, rq = fp8.gemm(rx, rw, quantize_output=True)
    rpay = fp8.sync_pack([fp8.SyncEntry(5, rw)])

    # buffers owned by the graph, warmed up eagerly once
    qx, qw = fp8.quantize_group(X, "K"), fp8.quantize_block(W)
    Y, qy = fp8.gemm(qx, qw, quantize_output=True)
    payload = fp8.sync_pack([fp8.SyncEntry(5, qw)]).clone()
    dst = _zeros_like(qw)
    fp8.sync_install(payload, [fp8.SyncEntry(5, dst)])
    torch.cuda.synchronize()

    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        fp8.quantize_group(X, "K", out=qx)
        fp8.quantize_block(W, out=qw)
        fp8.gemm(qx, qw, out=Y, out_q=qy, quantize_output=True)
        fp8.sync_pack([fp8.SyncEntry(5, qw)], payload=payload)
        fp8.sync_install(payload, [fp8.SyncEntry(5, dst)], check=False)

    X.copy_(X2)
    W.copy_(W2)
    dst.codes.zero_()
    dst.scales.zero_()
    payload.zero_()
    for _ in range(3):
        g.replay()
    torch.cuda.synchronize()
    fp8.status_poll()
    assert torch.equal(qx.codes, rx.codes) and torch.equal(qx.scales, rx.scales)
    assert torch.equal(qw.codes, rw.codes) and torch.equal(qw.scales, rw.scales)
    assert torch.equal(Y, rY)
    assert torch.equal(qy.codes, rq.codes) and torch.equal(qy.scales, rq.scales)
    assert torch.equal(payload, rpay)
    assert torch.equal(dst.codes, rw.codes) and torch.equal(dst.scales, rw.scales)


def test_packed_header_written_on_the_device_matches_a_host_copy():
    """Payloads whose header and table fit a kernel parameter (written by the
    pack kernel) and ones that do not (copied from the host) carry the same
    bytes for the same tensors: the first entries of a 30-entry payload are
    laid out as a 2-entry payload's, apart from the entry count and offsets,
    so both are checked by a round trip through install."""
    ws = [synth.random_bf16((128, 256), seed=300 + i, std=0.02).to(DEV) for i in range(30)]
    qs = [fp8.quantize_block(w) for w in ws]
    for n in (1, 2, 30):
        entries = [fp8.SyncEntry(40 + i, q) for i, q in enumerate(qs[:n])]
        payload = fp8.sync_pack(entries)
        dst = [fp8.SyncEntry(40 + i, _zeros_like(q)) for i, q in enumerate(qs[:n])]
        fp8.sync_install(payload, dst)
        for q, d in zip(qs[:n], dst):
            assert torch.equal(q.codes, d.tensor.codes) and torch.equal(q.scales, d.tensor.scales)
