"""Pins the oracle's on-policy weight-sync model: round trip is bit-identical,
corruption is detected, the layout is as specified, and the naive off-policy
path (dequantize -> bf16 -> per-tensor re-quantize) does NOT reproduce the
trainer's FP8 weights while the sync path does."""
import numpy as np
import pytest

from block_scaled_fp8_e4m3_gb300 import synth
from conftest import read_golden


def _specs(orc, seed=0):
    W = synth.random_bf16((256, 384), seed=seed + 1, std=0.02)
    cw, sw = orc.quant_block_128x128(synth.bf16_bits(W))
    X = synth.random_bf16((130, 256), seed=seed + 2, outliers=True)
    cx, sx = orc.quant_group_1x128(synth.bf16_bits(X))
    M = synth.random_bf16((100, 96), seed=seed + 3)
    cm, sm = orc.quant_mx_1x32(synth.bf16_bits(M))
    N = synth.random_bf16((3, 70), seed=seed + 4)
    return [
        dict(tag=0x1111, kind=orc.KIND_FP8, recipe=orc.RECIPE_BLOCKWISE, rows=256, cols=384,
             layout=orc.LAYOUT_BLOCK_128x128, data=cw, scales=sw),
        dict(tag=0x2222, kind=orc.KIND_FP8, recipe=orc.RECIPE_BLOCKWISE, rows=130, cols=256,
             layout=orc.LAYOUT_GROUP_1x128, data=cx, scales=sx),
        dict(tag=0x3333, kind=orc.KIND_FP8, recipe=orc.RECIPE_MX, rows=100, cols=96,
             layout=orc.LAYOUT_MX_1x32, data=cm, scales=sm),
        dict(tag=0x4444, kind=orc.KIND_BF16, recipe=orc.RECIPE_NONE, rows=3, cols=70,
             layout=orc.LAYOUT_NONE, data=synth.bf16_bits(N), scales=None),
    ]


def _empty_like(specs):
    out = []
    for s in specs:
        d = dict(s)
        d["data"] = np.zeros_like(s["data"])
        d["scales"] = None if s["scales"] is None else np.zeros_like(s["scales"])
        out.append(d)
    return out


def _rd(p, off, n):
    return int.from_bytes(bytes(p[off:off + n]), "little")


def test_round_trip_bit_identical(orc):
    specs = _specs(orc)
    payload = orc.sync_pack(specs)
    dst = _empty_like(specs)
    assert orc.sync_install(payload, dst) == 0
    for s, d in zip(specs, dst):
        assert np.array_equal(s["data"], d["data"])
        if s["scales"] is not None:
            assert s["scales"].tobytes() == d["scales"].tobytes()


def test_layout(orc):
    specs = _specs(orc)
    p = orc.sync_pack(specs)
    assert bytes(p[:8]) == b"FP8SYNC1"
    assert _rd(p, 8, 4) == 2 and _rd(p, 12, 4) == len(specs)
    total = _rd(p, 16, 8)
    assert total == p.size and total % 256 == 0
    assert _rd(p, 24, 8) == 768                       # roundup(64 + 4*128, 256)
    prev_end = 768
    for i, s in enumerate(specs):
        t = 64 + 128 * i
        doff, dbytes = _rd(p, t + 40, 8), _rd(p, t + 48, 8)
        soff, sbytes = _rd(p, t + 56, 8), _rd(p, t + 64, 8)
        assert doff % 256 == 0 and doff >= prev_end
        assert dbytes == s["data"].nbytes
        assert bytes(p[doff:doff + dbytes]) == s["data"].tobytes()
        prev_end = doff + dbytes
        if s["scales"] is not None:
            assert soff % 256 == 0 and soff >= prev_end and sbytes == s["scales"].nbytes
            assert bytes(p[soff:soff + sbytes]) == s["scales"].tobytes()
            prev_end = soff + sbytes
        else:
            assert soff == 0 and sbytes == 0
        assert not np.any(p[t + 72:t + 128])
    # padding is zero
    assert _rd(p, 40, 24) == 0


def test_checksum_is_the_sum_of_word_terms(orc):
    """The checksum field equals the sum mod 2^64 of the per-word terms over
    the words at byte offsets >= 64 (the header's own words excluded), with
    the checksum field itself counted as zero when the sum was formed."""
    specs = _specs(orc)
    p = orc.sync_pack(specs)
    q = p.copy()
    q[32:40] = 0
    words = q.view("<u8")
    total = sum(orc.sync_word_term(int(w), i) for i, w in enumerate(words) if i >= 8) % 2 ** 64
    assert total == _rd(p, 32, 8) == orc.sync_checksum(p)


def test_word_term_is_bilinear_in_the_keyed_halves(orc):
    """t(w, i) = ((lo + i K1) mod 2^32) ((hi + i K2) mod 2^32): with the key
    sums a, b of a word, adding d to lo (no wrap of a) changes t by exactly
    d * b, adding d to hi changes it by d * a, and t is the product a * b --
    checked against keys recovered from words whose halves are zero, so a
    swapped pair of halves, a wrong key or a dropped key fails."""
    rng = np.random.default_rng(11)
    K1, K2 = 0x9E3779B9, 0x85EBCA6B
    for _ in range(200):
        i = int(rng.integers(8, 2 ** 40))
        ka = (i * K1) % 2 ** 32                         # key sums of the zero word
        kb = (i * K2) % 2 ** 32
        assert orc.sync_word_term(0, i) == ka * kb
        lo, hi = int(rng.integers(0, 2 ** 32)), int(rng.integers(0, 2 ** 32))
        a, b = (lo + ka) % 2 ** 32, (hi + kb) % 2 ** 32
        w = lo | (hi << 32)
        t = orc.sync_word_term(w, i)
        assert t == a * b
        d = int(rng.integers(1, 2 ** 16))
        if a + d < 2 ** 32 and (lo + d) < 2 ** 32:
            assert orc.sync_word_term(w + d, i) == t + d * b
        if b + d < 2 ** 32 and (hi + d) < 2 ** 32:
            assert orc.sync_word_term(w + (d << 32), i) == t + d * a
    # keys depend on the index modulo 2^32 words only
    assert orc.sync_word_term(12345, 7) == orc.sync_word_term(12345, 7 + 2 ** 32)


def test_checksum_detects_every_single_bit_flip(orc):
    """Flipping any one of the 64 bits of a word changes its term by
    +-2^b times the other keyed half, which is nonzero whenever that half is
    (true for every word of this payload), so every single-bit flip of the
    covered region is detected: all 64 bits of 40 words spread over the
    header tail, the table, data, padding and scales."""
    specs = _specs(orc)
    p = orc.sync_pack(specs)
    base = orc.sync_checksum(p)
    nwords = p.size // 8
    for wi in np.linspace(8, nwords - 1, 40).astype(int):
        for bit in range(64):
            q = p.copy()
            q[8 * wi + bit // 8] ^= 1 << (bit % 8)
            assert orc.sync_checksum(q) != base, (wi, bit)


def test_checksum_detects_any_single_word_change(orc):
    specs = _specs(orc)
    p = orc.sync_pack(specs)
    base = orc.sync_checksum(p)
    assert base == _rd(p, 32, 8)
    rng = np.random.default_rng(5)
    for off in list(range(64, p.size, 8))[::7]:
        q = p.copy()
        q[off + rng.integers(0, 8)] ^= 1 << int(rng.integers(0, 8))
        assert orc.sync_checksum(q) != base
    # header words (bytes 0..63) are not covered by the sum
    q = p.copy()
    q[40] = 1
    assert orc.sync_checksum(q) == base


@pytest.mark.parametrize("where", ["data", "table", "magic", "count", "shape", "tag"])
def test_install_rejects_corruption(orc, where):
    specs = _specs(orc)
    p = orc.sync_pack(specs)
    dst = _empty_like(specs)
    expect = 2
    if where == "data":
        p[_rd(p, 64 + 40, 8) + 5] ^= 0x10
    elif where == "table":
        p[64 + 72] = 1                                  # reserved byte, covered by checksum
    elif where == "magic":
        p[0] ^= 1
        expect = 1
    elif where == "count":
        dst = dst[:3]
        expect = 1
    elif where == "shape":
        dst[0]["rows"] = 128
        dst[0]["data"] = dst[0]["data"][:128].copy()
        dst[0]["scales"] = dst[0]["scales"][:1].copy()
        expect = 1
    elif where == "tag":
        dst[1]["tag"] = 0x9999
        expect = 1
    assert orc.sync_install(p, dst) == expect
    for d in dst:
        assert not np.any(d["data"])                    # nothing written


def test_naive_off_policy_differs_sync_does_not(orc):
    """The per-tensor re-quantization of the dequantized BF16 weights does not
    reproduce the trainer's FP8 representation; the sync payload does."""
    W = synth.tiny().tensors["W"]
    w = W.double().numpy()
    cw, sw = orc.quant_block_128x128(synth.bf16_bits(W))
    naive_codes, s_naive = orc.naive_requant_per_tensor(cw, sw)
    # the block holding the tensor maximum round-trips exactly (its max code
    # is 448 * s and the product is bf16-representable), so the per-tensor
    # scale equals the largest block scale; every other block gets a scale
    # that is not its own, and its codes change
    assert s_naive == sw.max()
    trainer = orc.dequant_block(cw, sw)
    rollout = orc.e4m3_decode(naive_codes) * s_naive
    nb, kb = np.unravel_index(int(np.argmax(sw)), sw.shape)
    same = np.zeros_like(trainer, dtype=bool)
    same[nb * 128:(nb + 1) * 128, kb * 128:(kb + 1) * 128] = True
    assert np.array_equal(trainer[same], rollout[same])
    assert np.count_nonzero(trainer[~same] != rollout[~same]) > 0.5 * np.count_nonzero(~same)
    # the synthetic analogue of the mismatch figure (reported, not pinned)
    rel = np.abs(rollout - trainer).mean() / np.abs(trainer).mean()
    q_err = np.abs(trainer - w).mean() / np.abs(w).mean()
    assert rel > 0 and q_err > 0
    # sync path: identical
    spec = [dict(tag=1, kind=orc.KIND_FP8, recipe=orc.RECIPE_BLOCKWISE, rows=512, cols=512,
                 layout=orc.LAYOUT_BLOCK_128x128, data=cw, scales=sw)]
    dst = _empty_like(spec)
    assert orc.sync_install(orc.sync_pack(spec), dst) == 0
    assert np.array_equal(orc.dequant_block(dst[0]["data"], dst[0]["scales"]), trainer)


def test_naive_mismatch_figure_on_the_mlp_weight(orc):
    """[SkyRL] "独立した量子化がポリシーの一貫性を崩す場合": the synthetic analogue of
    the trainer-vs-rollout mismatch of the naive (BF16 bridge, per-tensor
    re-quantization) sync, on the dense-MLP weight 12288x4096 ~N(0, 0.02).
    Reported, not pinned: the pages' 0.038 and 1.4x come from a trained 4B
    model."""
    W = synth.mlp().tensors["W"]
    w = W.double().numpy()
    cw, sw = orc.quant_block_128x128(synth.bf16_bits(W))
    naive_codes, s_naive = orc.naive_requant_per_tensor(cw, sw)
    trainer = orc.dequant_block(cw, sw)
    rollout = orc.e4m3_decode(naive_codes) * s_naive
    rel = np.abs(rollout - trainer).mean() / np.abs(trainer).mean()
    q_err = np.abs(trainer - w).mean() / np.abs(w).mean()
    print(f"naive sync: mean relative mismatch {rel:.4f}, {rel / q_err:.2f}x the trainer's quantization error, "
          f"{np.count_nonzero(naive_codes != cw) / cw.size:.4f} of the codes differ")
    assert 0.01 < rel < 0.05 and 0.5 < rel / q_err < 2.0
    assert np.count_nonzero(naive_codes != cw) > 0.9 * cw.size
