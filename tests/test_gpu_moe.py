"""GPU parity of the MoE path: quantize once, gather rows into expert groups
(bit-exact: equals quantizing the gathered rows), grouped MXFP8 GEMM within
tolerance per expert segment."""
import numpy as np
import pytest
import torch

import block_scaled_fp8_e4m3_gb300 as fp8
import oracle
from block_scaled_fp8_e4m3_gb300 import synth
from gpu_util import DEV, assert_bytes_equal, assert_gemm_close, oracle_mx, stratified_positions, to_np

pytestmark = pytest.mark.gpu


def _grouped_oracle_scales(codes_src, scales_src, gather, offsets, K):
    """Expected grouped-layout scale bytes, by definition: dst row i of group
    g sits at atom row P_g + (i - off_g)/128, P_g = sum_{h<g} ceil(M_h/128)."""
    G = len(offsets) - 1
    P = np.zeros(G + 1, np.int64)
    for g in range(G):
        P[g + 1] = P[g] + (offsets[g + 1] - offsets[g] + 127) // 128
    total = offsets[-1]
    out = np.zeros(((total + 127) // 128 + G) * (K // 128) * 512, np.uint8)
    for g in range(G):
        for i in range(offsets[g], offsets[g + 1]):
            src = gather[i]
            l = i - offsets[g]
            for kb in range(K // 32):
                out[oracle.mx_scale_offset(P[g] * 128 + l, kb, K)] = scales_src[oracle.mx_scale_offset(src, kb, K)]
    return out


def _moe_case(tokens, experts, top_k, hidden, ffn, seed):
    wl = synth.moe(tokens=tokens, experts=experts, top_k=top_k, hidden=hidden, ffn=ffn, seed=seed)
    return wl.tensors["X"], wl.tensors["W"], wl.tensors["gather"], wl.tensors["offsets"]


def _run(X, W, gather, offsets):
    G, N, K = W.shape
    qx = fp8.quantize_mx(X.to(DEV))
    qa = fp8.permute_rows_mx(qx, gather.to(DEV), offsets.to(DEV))
    qw = fp8.quantize_mx(W.reshape(G * N, K).to(DEV))
    Y = fp8.grouped_gemm(qa, qw, offsets.to(DEV), N)
    return qa, Y


@pytest.mark.parametrize("tokens,experts,top_k,hidden,ffn,seed", [(200, 8, 2, 256, 256, 5),
                                                                  (700, 16, 4, 512, 512, 6)])
def test_moe_small(tokens, experts, top_k, hidden, ffn, seed):
    X, W, gather, offsets = _moe_case(tokens, experts, top_k, hidden, ffn, seed)
    qa, Y = _run(X, W, gather, offsets)
    g_np, off_np = gather.numpy(), offsets.numpy().astype(np.int64)
    cx, sx = oracle_mx(X)
    # permutation: codes and scales exactly as defined
    assert_bytes_equal(to_np(qa.codes), cx[g_np], "permuted codes")
    assert_bytes_equal(to_np(qa.scales), _grouped_oracle_scales(cx, sx, g_np, off_np, hidden), "grouped scales")
    # quantize-then-permute == permute-then-quantize
    cp, sp = oracle_mx(X[torch.from_numpy(g_np.astype(np.int64))])
    assert np.array_equal(cp, cx[g_np])
    # grouped GEMM per expert segment
    A_deq = oracle.dequant_mx(cx, sx)[g_np]
    G, N, K = W.shape
    cw, sw = oracle_mx(W.reshape(G * N, K))
    W_deq = oracle.dequant_mx(cw, sw).reshape(G, N, K)
    Yh = Y.double().cpu().numpy()
    for g in range(G):
        a, b = off_np[g], off_np[g + 1]
        if b == a:
            continue
        ref, mag = oracle.gemm_ref(A_deq[a:b], W_deq[g])
        assert_gemm_close(Yh[a:b], ref, mag, f"expert {g} ({b - a} rows)")


def test_moe_empty_and_single_row_groups():
    """Groups with 0 and 1 rows, and a group that is an exact multiple of 128."""
    K, N, G = 256, 256, 4
    counts = [0, 1, 128, 77]
    offsets = torch.tensor(np.concatenate([[0], np.cumsum(counts)]), dtype=torch.int32)
    total = int(offsets[-1])
    X = synth.random_bf16((50, K), seed=3, outliers=True)
    gather = torch.randint(0, 50, (total,), generator=torch.Generator().manual_seed(4), dtype=torch.int64).to(torch.int32)
    W = synth.random_bf16((G, N, K), seed=5, std=0.02)
    qa, Y = _run(X, W, gather, offsets)
    cx, sx = oracle_mx(X)
    A_deq = oracle.dequant_mx(cx, sx)[gather.numpy()]
    cw, sw = oracle_mx(W.reshape(G * N, K))
    W_deq = oracle.dequant_mx(cw, sw).reshape(G, N, K)
    off = offsets.numpy()
    for g in range(G):
        a, b = off[g], off[g + 1]
        if b > a:
            ref, mag = oracle.gemm_ref(A_deq[a:b], W_deq[g])
            assert_gemm_close(Y[a:b].double().cpu().numpy(), ref, mag, f"group {g}")


@pytest.mark.parametrize("bad", [[0, 100, 450, 300], [0, 150, 100, 300], [-5, 100, 200, 300], [0, 100, 200, 340]])
def test_bad_group_offsets_are_reported_and_contained(bad):
    """Group offsets past the rows of A, decreasing, or negative: the grouped
    GEMM reports FP8_ERR_INVALID_ARG at the next status poll, writes nothing
    outside D's rows, and later calls with valid offsets are exact again."""
    K, N, G = 256, 256, 3
    offsets = torch.tensor([0, 100, 200, 300], dtype=torch.int32)
    X = synth.random_bf16((300, K), seed=21, outliers=True)
    gather = torch.arange(300, dtype=torch.int32)
    W = synth.random_bf16((G, N, K), seed=22, std=0.02)
    qa, Y = _run(X, W, gather, offsets)
    qw = fp8.quantize_mx(W.reshape(G * N, K).to(DEV))
    buf = torch.full((300 + 64, N), 7.0, dtype=torch.bfloat16, device=DEV)
    fp8.grouped_gemm(qa, qw, torch.tensor(bad, dtype=torch.int32, device=DEV), N, out=buf[:300])
    with pytest.raises(fp8.FP8Error) as ei:
        fp8.status_poll()
    assert ei.value.status == 1
    assert bool((buf[300:] == 7.0).all())
    Y2 = fp8.grouped_gemm(qa, qw, offsets.to(DEV), N)
    fp8.status_poll()
    assert torch.equal(Y2, Y)


@pytest.mark.parametrize("bad", [[0, 150, 100, 300], [10, 100, 200, 300], [0, 100, 200, 290], [-128, 100, 200, 300]])
def test_permute_and_dispatch_reject_bad_offsets(bad):
    """Group offsets that decrease, do not start at 0 or do not end at the
    row count: the row gather and the fused dispatch report
    FP8_ERR_INVALID_ARG and write nothing outside the destination buffers
    (the dispatch writes no codes at all)."""
    rows, K, G = 300, 256, 3
    X = synth.random_bf16((rows, K), seed=31, outliers=True).to(DEV)
    qx = fp8.quantize_mx(X)
    sb = fp8.mx_grouped_scale_bytes(rows, K, G)
    codes_buf = torch.full((rows + 8, K), 0x5A, dtype=torch.uint8, device=DEV)
    scales_buf = torch.full((sb + 4096,), 0x5A, dtype=torch.uint8, device=DEV)
    out = fp8.QTensor(codes_buf[:rows], scales_buf[:sb], rows, K, fp8.RECIPE_MX, fp8.LAYOUT_MX_1x32_GROUPED)
    off = torch.tensor(bad, dtype=torch.int32, device=DEV)
    fp8.permute_rows_mx(qx, torch.arange(rows, dtype=torch.int32, device=DEV), off, out=out)
    with pytest.raises(fp8.FP8Error) as ei:
        fp8.status_poll()
    assert ei.value.status == 1
    assert bool((codes_buf[rows:] == 0x5A).all()) and bool((scales_buf[sb:] == 0x5A).all())
    codes_buf.fill_(0x5A)
    scales_buf.fill_(0x5A)
    dst_index = torch.arange(rows, dtype=torch.int32, device=DEV).reshape(rows, 1)
    fp8.dispatch_quantize_mx(X, dst_index, off, rows, out=out)
    with pytest.raises(fp8.FP8Error) as ei:
        fp8.status_poll()
    assert ei.value.status == 1
    assert bool((codes_buf == 0x5A).all()) and bool((scales_buf[sb:] == 0x5A).all())


def test_full_moe_sampled():
    X, W, gather, offsets = _moe_case(16384, 64, 8, 2048, 1024, 4)
    qa, Y = _run(X, W, gather, offsets)
    g_np, off_np = gather.numpy(), offsets.numpy().astype(np.int64)
    cx, sx = oracle_mx(X)
    assert_bytes_equal(to_np(qa.codes), cx[g_np], "permuted codes")
    G, N, K = W.shape
    cw, sw = oracle_mx(W.reshape(G * N, K))
    A_deq_src = oracle.dequant_mx(cx, sx)
    W_deq = oracle.dequant_mx(cw, sw)
    # stratified over the kernel's tiles: 256-row tiles from each expert's
    # first row, 256-column tiles
    segs = [(int(off_np[e]), int(off_np[e + 1])) for e in range(G) if off_np[e + 1] > off_np[e]]
    rows, cols = stratified_positions(int(off_np[-1]), N, seed=1, row_segments=segs)
    grp = np.searchsorted(off_np, rows, side="right") - 1
    ref, mag = oracle.gemm_ref_sampled(A_deq_src, W_deq, g_np[rows].astype(np.int64), grp * N + cols)
    got = Y[torch.from_numpy(rows).to(DEV), torch.from_numpy(cols).to(DEV)].double().cpu().numpy()
    assert_gemm_close(got, ref, mag, "moe full sampled")


def _moe_dispatch_case(tokens, experts, top_k, hidden, seed):
    wl = synth.moe(tokens=tokens, experts=experts, top_k=top_k, hidden=hidden, ffn=256, seed=seed)
    return wl.tensors["X"], wl.tensors["gather"], wl.tensors["offsets"], wl.tensors["dst_index"]


@pytest.mark.parametrize("tokens,experts,top_k,hidden,seed", [(200, 8, 2, 256, 5), (700, 16, 4, 384, 6),
                                                             (300, 4, 2, 128, 7), (90, 6, 3, 2304, 8)])
def test_fused_dispatch_quantization(tokens, experts, top_k, hidden, seed):
    """dispatch_quantize_mx: the oracle's 1x32 quantization of the gathered
    rows in the grouped layout, and the same bytes as quantize-then-permute
    (hidden 384 and 128 leave a half round of 256 columns; 2304 takes two
    passes of 2048 columns)."""
    X, gather, offsets, dst_index = _moe_dispatch_case(tokens, experts, top_k, hidden, seed)
    g_np, off_np = gather.numpy(), offsets.numpy().astype(np.int64)
    assert np.array_equal(g_np[dst_index.numpy()], np.repeat(np.arange(tokens), top_k).reshape(tokens, top_k))
    q = fp8.dispatch_quantize_mx(X.to(DEV), dst_index.to(DEV), offsets.to(DEV), gather.numel())
    cx, sx = oracle_mx(X)
    assert_bytes_equal(to_np(q.codes), cx[g_np], "fused dispatch codes")
    assert_bytes_equal(to_np(q.scales), _grouped_oracle_scales(cx, sx, g_np, off_np, hidden), "fused dispatch scales")
    q2 = fp8.permute_rows_mx(fp8.quantize_mx(X.to(DEV)), gather.to(DEV), offsets.to(DEV))
    assert torch.equal(q.codes, q2.codes) and torch.equal(q.scales, q2.scales)
    assert fp8.status_poll() is None


def test_fused_dispatch_full_size():
    wl = synth.moe()
    X, gather, offsets, dst_index = (wl.tensors[k] for k in ("X", "gather", "offsets", "dst_index"))
    q = fp8.dispatch_quantize_mx(X.to(DEV), dst_index.to(DEV), offsets.to(DEV), gather.numel())
    q2 = fp8.permute_rows_mx(fp8.quantize_mx(X.to(DEV)), gather.to(DEV), offsets.to(DEV))
    assert torch.equal(q.codes, q2.codes) and torch.equal(q.scales, q2.scales)
    cx, _ = oracle_mx(X)
    assert_bytes_equal(to_np(q.codes), cx[gather.numpy()], "fused dispatch codes 131072x2048")


def test_fused_dispatch_dropped_and_bad_slots():
    """-1 drops a slot (its row keeps its codes); an index past the end is
    skipped and reported."""
    X = synth.random_bf16((4, 128), seed=9)
    offsets = torch.tensor([0, 2, 4], dtype=torch.int32)
    dst_index = torch.tensor([[0], [-1], [3], [1]], dtype=torch.int32)
    out = fp8.QTensor(torch.full((4, 128), 0x5A, dtype=torch.uint8, device=DEV),
                      torch.empty((fp8.mx_grouped_scale_bytes(4, 128, 2),), dtype=torch.uint8, device=DEV),
                      4, 128, fp8.RECIPE_MX, fp8.LAYOUT_MX_1x32_GROUPED)
    fp8.dispatch_quantize_mx(X.to(DEV), dst_index.to(DEV), offsets.to(DEV), 4, out=out)
    cx, _ = oracle_mx(X)
    got = to_np(out.codes)
    assert_bytes_equal(got[[0, 3, 1]], cx[[0, 2, 3]], "dispatched rows")
    assert np.all(got[2] == 0x5A)                                  # named by no slot
    assert fp8.status_poll() is None
    bad = torch.tensor([[0], [7], [3], [1]], dtype=torch.int32)   # 7 >= 4 rows
    fp8.dispatch_quantize_mx(X.to(DEV), bad.to(DEV), offsets.to(DEV), 4, out=out)
    with pytest.raises(fp8.FP8Error):
        fp8.status_poll()
