"""GPU parity of the weight-sync path: the device payload is byte-identical to
the oracle's, the installed rollout tensors are bit-identical to the
trainer's, and corruption is caught before anything is written."""
import numpy as np
import pytest
import torch

import block_scaled_fp8_e4m3_gb300 as fp8
import oracle
from block_scaled_fp8_e4m3_gb300 import synth
from gpu_util import DEV, assert_bytes_equal, oracle_block, oracle_group_k, oracle_mx, to_np

pytestmark = pytest.mark.gpu


def _trainer_tensors(seed=0, n=384, k=512):
    W = synth.random_bf16((n, k), seed=seed + 1, std=0.02)
    X = synth.random_bf16((130, 256), seed=seed + 2, outliers=True)
    M = synth.random_bf16((100, 96), seed=seed + 3)
    N = synth.random_bf16((3, 72), seed=seed + 4)
    return W, X, M, N


def _entries(W, X, M, N):
    qw = fp8.quantize_block(W.to(DEV))
    qx = fp8.quantize_group(X.to(DEV), "K")
    qm = fp8.quantize_mx(M.to(DEV))
    nd = N.to(DEV)
    return [fp8.SyncEntry(0x1111, qw), fp8.SyncEntry(0x2222, qx), fp8.SyncEntry(0x3333, qm),
            fp8.SyncEntry(0x4444, nd)]


def _oracle_specs(W, X, M, N):
    cw, sw = oracle_block(W)
    cx, sx = oracle_group_k(X)
    cm, sm = oracle_mx(M)
    return [
        dict(tag=0x1111, kind=oracle.KIND_FP8, recipe=oracle.RECIPE_BLOCKWISE, rows=W.shape[0], cols=W.shape[1],
             layout=oracle.LAYOUT_BLOCK_128x128, data=cw, scales=sw),
        dict(tag=0x2222, kind=oracle.KIND_FP8, recipe=oracle.RECIPE_BLOCKWISE, rows=130, cols=256,
             layout=oracle.LAYOUT_GROUP_1x128, data=cx, scales=sx),
        dict(tag=0x3333, kind=oracle.KIND_FP8, recipe=oracle.RECIPE_MX, rows=100, cols=96,
             layout=oracle.LAYOUT_MX_1x32, data=cm, scales=sm),
        dict(tag=0x4444, kind=oracle.KIND_BF16, recipe=oracle.RECIPE_NONE, rows=3, cols=72,
             layout=oracle.LAYOUT_NONE, data=synth.bf16_bits(N), scales=None),
    ]


def _empty_like(entries):
    out = []
    for e in entries:
        t = e.tensor
        if isinstance(t, fp8.QTensor):
            t2 = fp8.QTensor(torch.zeros_like(t.codes), torch.zeros_like(t.scales), t.rows, t.cols, t.recipe,
                             t.layout)
        else:
            t2 = torch.zeros_like(t)
        out.append(fp8.SyncEntry(e.tag, t2))
    return out


def test_payload_matches_oracle_and_round_trip():
    W, X, M, N = _trainer_tensors()
    entries = _entries(W, X, M, N)
    payload = fp8.sync_pack(entries)
    ref = oracle.sync_pack(_oracle_specs(W, X, M, N))
    assert_bytes_equal(payload.cpu().numpy(), ref, "payload")
    dst = _empty_like(entries)
    fp8.sync_install(payload, dst)
    for s, d in zip(entries, dst):
        if isinstance(s.tensor, fp8.QTensor):
            assert torch.equal(s.tensor.codes, d.tensor.codes)
            assert torch.equal(s.tensor.scales.view(torch.uint8), d.tensor.scales.view(torch.uint8))
        else:
            assert torch.equal(s.tensor.view(torch.int16), d.tensor.view(torch.int16))


def test_corrupted_payload_writes_nothing():
    W, X, M, N = _trainer_tensors(seed=10)
    entries = _entries(W, X, M, N)
    payload = fp8.sync_pack(entries).clone()
    payload[payload.numel() // 2] ^= 0x40                     # a data byte
    dst = _empty_like(entries)
    with pytest.raises(fp8.FP8Error) as ei:
        fp8.sync_install(payload, dst)
    assert ei.value.status == 5                               # FP8_ERR_CHECKSUM
    for d in dst:
        t = d.tensor.codes if isinstance(d.tensor, fp8.QTensor) else d.tensor
        assert int(t.view(torch.uint8).count_nonzero()) == 0
    # a clean install afterwards works (the status block was cleared)
    good = fp8.sync_pack(entries)
    fp8.sync_install(good, dst)


def test_installs_on_two_streams_are_ordered():
    """Installs of a clean and a corrupted payload issued back to back on two
    streams, ten rounds in both orders: the library orders them on the
    device, so the clean one lands bit for bit, the corrupted one writes
    nothing, and the checksum verdicts do not mix."""
    W, X, M, N = _trainer_tensors(seed=30)
    entries = _entries(W, X, M, N)
    good = fp8.sync_pack(entries)
    bad = good.clone()
    bad[bad.numel() // 2] ^= 0x40
    s1, s2 = torch.cuda.Stream(), torch.cuda.Stream()
    for r in range(10):
        d_good, d_bad = _empty_like(entries), _empty_like(entries)
        torch.cuda.synchronize()
        order = [(s1, good, d_good), (s2, bad, d_bad)]
        for s, payload, dst in (order if r % 2 == 0 else order[::-1]):
            fp8.sync_install(payload, dst, stream=s, check=False)
        torch.cuda.synchronize()
        with pytest.raises(fp8.FP8Error) as ei:
            fp8.status_poll()
        assert ei.value.status == 5                           # FP8_ERR_CHECKSUM, from the corrupted one
        for src, d in zip(entries, d_good):
            a, b = (src.tensor, d.tensor)
            if isinstance(a, fp8.QTensor):
                assert torch.equal(a.codes, b.codes) and torch.equal(a.scales, b.scales)
            else:
                assert torch.equal(a, b)
        for d in d_bad:
            t = d.tensor.codes if isinstance(d.tensor, fp8.QTensor) else d.tensor
            assert int(t.view(torch.uint8).count_nonzero()) == 0
    fp8.status_poll()


def test_header_mismatch_rejected():
    W, X, M, N = _trainer_tensors(seed=20)
    entries = _entries(W, X, M, N)
    payload = fp8.sync_pack(entries)
    dst = _empty_like(entries)
    dst[1] = fp8.SyncEntry(0x9999, dst[1].tensor)              # wrong tag
    with pytest.raises(fp8.FP8Error) as ei:
        fp8.sync_install(payload, dst)
    assert ei.value.status == 4                               # FP8_ERR_BAD_PAYLOAD
    with pytest.raises(fp8.FP8Error) as ei:
        fp8.sync_install(payload, _empty_like(entries)[:3])   # wrong count
    assert ei.value.status in (4,)


def test_full_mlp_weight_round_trip():
    """The dense-MLP weight (12288x4096, 128x128 blocks): pack -> install is
    bit-identical, and the payload equals the oracle's byte for byte."""
    W = synth.mlp().tensors["W"]
    qw = fp8.quantize_block(W.to(DEV))
    entries = [fp8.SyncEntry(7, qw)]
    payload = fp8.sync_pack(entries)
    cw, sw = oracle_block(W)
    ref = oracle.sync_pack([dict(tag=7, kind=oracle.KIND_FP8, recipe=oracle.RECIPE_BLOCKWISE, rows=12288,
                                 cols=4096, layout=oracle.LAYOUT_BLOCK_128x128, data=cw, scales=sw)])
    assert_bytes_equal(payload.cpu().numpy(), ref, "payload")
    dst = _empty_like(entries)
    fp8.sync_install(payload, dst)
    assert torch.equal(dst[0].tensor.codes, qw.codes)
    assert torch.equal(dst[0].tensor.scales, qw.scales)


def test_many_entries_use_the_two_kernel_path():
    """30 quantized entries (60 segments, more than one cooperative launch's
    table of 32, and more than the 23 entries whose header the device checks):
    the verify + scatter path and the host header check.  The payload equals
    the oracle's, the round trip is bit-identical, and a corrupted payload
    writes nothing."""
    ws = [synth.random_bf16((128, 256), seed=100 + i, std=0.02) for i in range(30)]
    qs = [fp8.quantize_block(w.to(DEV)) for w in ws]
    entries = [fp8.SyncEntry(1000 + i, q) for i, q in enumerate(qs)]
    payload = fp8.sync_pack(entries)
    specs = []
    for i, w in enumerate(ws):
        c, s = oracle_block(w)
        specs.append(dict(tag=1000 + i, kind=oracle.KIND_FP8, recipe=oracle.RECIPE_BLOCKWISE, rows=128, cols=256,
                          layout=oracle.LAYOUT_BLOCK_128x128, data=c, scales=s))
    assert_bytes_equal(payload.cpu().numpy(), oracle.sync_pack(specs), "30-entry payload")
    dst = _empty_like(entries)
    fp8.sync_install(payload, dst)
    for q, d in zip(qs, dst):
        assert torch.equal(d.tensor.codes, q.codes) and torch.equal(d.tensor.scales, q.scales)
    bad = payload.clone()
    bad[bad.numel() - 300] ^= 0x01
    dst2 = _empty_like(entries)
    with pytest.raises(fp8.FP8Error) as ei:
        fp8.sync_install(bad, dst2)
    assert ei.value.status == 5
    for d in dst2:
        assert int(d.tensor.codes.count_nonzero()) == 0
