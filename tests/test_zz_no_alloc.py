"""The allocation-free install entry point, for callers that cannot call
cudaMalloc (e.g. a rollout engine whose memory pool already owns the device).
It must leave the destinations byte-identical to what fp8_sync_install
writes, on two calls in a row, and reject more entries than its fixed
scratch array holds.  This file is collected last on purpose."""
import ctypes as C

import pytest
import torch

import block_scaled_fp8_e4m3_gb300 as fp8
from block_scaled_fp8_e4m3_gb300 import synth

pytestmark = pytest.mark.gpu

DEV = "cuda:0"


def _trainer_entries(seed):
    W = synth.random_bf16((384, 512), seed=seed + 1, std=0.02).to(DEV)
    X = synth.random_bf16((130, 256), seed=seed + 2, outliers=True).to(DEV)
    M = synth.random_bf16((100, 96), seed=seed + 3).to(DEV)
    N = synth.random_bf16((3, 72), seed=seed + 4).to(DEV)
    return [fp8.SyncEntry(0x11, fp8.quantize_block(W)), fp8.SyncEntry(0x22, fp8.quantize_group(X, "K")),
            fp8.SyncEntry(0x33, fp8.quantize_mx(M)), fp8.SyncEntry(0x44, N)]


def _blank(entries, fill=0):
    out = []
    for e in entries:
        t = e.tensor
        if isinstance(t, fp8.QTensor):
            t2 = fp8.QTensor(torch.full_like(t.codes, fill), torch.full_like(t.scales.view(torch.uint8), fill)
                             .view(t.scales.dtype), t.rows, t.cols, t.recipe, t.layout)
        else:
            t2 = torch.full_like(t.view(torch.int16), fill).view(t.dtype)
        out.append(fp8.SyncEntry(e.tag, t2))
    return out


def _bytes(entry):
    t = entry.tensor
    if isinstance(t, fp8.QTensor):
        return [t.codes.view(torch.uint8).cpu(), t.scales.view(torch.uint8).cpu()]
    return [t.view(torch.uint8).cpu()]


def _install_noalloc(payload, dst):
    lib = fp8.library()
    arr = fp8._entries(dst)
    st = lib.fp8_sync_install_noalloc(C.c_void_p(payload.data_ptr()), C.c_uint64(payload.numel()), arr,
                                      C.c_int32(len(dst)), C.c_void_p(torch.cuda.current_stream().cuda_stream))
    return st, lib.fp8_last_error().decode()


def test_matches_sync_install_on_two_calls():
    for call, seed in enumerate((100, 200)):
        entries = _trainer_entries(seed)
        payload = fp8.sync_pack(entries)
        ref = _blank(entries)
        fp8.sync_install(payload, ref)                       # the existing entry point
        got = _blank(entries, fill=0x5A)                      # stale bytes must be overwritten
        st, msg = _install_noalloc(payload, got)
        assert st == 0, f"call {call}: {msg}"
        torch.cuda.synchronize()
        for r, g in zip(ref, got):
            for a, b in zip(_bytes(r), _bytes(g)):
                assert torch.equal(a, b), f"call {call}: tag {r.tag:#x} differs"


def test_checksum_mismatch_and_capacity():
    entries = _trainer_entries(300)
    payload = fp8.sync_pack(entries).clone()
    payload[payload.numel() - 300] ^= 0x01
    dst = _blank(entries)
    st, msg = _install_noalloc(payload, dst)
    assert st == 5, msg                                       # FP8_ERR_CHECKSUM
    for d in dst:
        for a in _bytes(d):
            assert int(a.count_nonzero()) == 0
    # a clean payload right after a failed one installs correctly
    good = fp8.sync_pack(entries)
    st, msg = _install_noalloc(good, dst)
    assert st == 0, msg
    # more entries than the fixed scratch array holds
    many = [fp8.SyncEntry(i, entries[3].tensor) for i in range(129)]
    st, msg = _install_noalloc(fp8.sync_pack(many[:1]), many)
    assert st == 8 and "128" in msg                           # FP8_ERR_CAPACITY
