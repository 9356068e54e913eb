"""Out-of-bounds write check for every kernel output (the substitute for a
memory sanitizer on this pool): each output buffer -- D, codes, scales, MX
scale atoms, transposed copies, grouped outputs, fused-producer outputs,
sync destinations -- is the interior of a larger allocation whose leading
and trailing 4 KB are filled with 0xA5.  After the call the bands must be
intact and the interior must equal the same call's result into a plain
allocation.  Shapes are the ragged ones: M = 1, 257, 300, 513 rows; MoE
groups of 0, 1 and 77 rows."""
import math

import numpy as np
import pytest
import torch

import block_scaled_fp8_e4m3_gb300 as fp8
from block_scaled_fp8_e4m3_gb300 import synth
from gpu_util import DEV

pytestmark = pytest.mark.gpu

BAND = 4096
FILL = 0xA5


class Guarded:
    """An output tensor of `shape`/`dtype` inside a 0xA5-banded allocation."""

    def __init__(self, shape, dtype):
        itemsize = torch.empty((), dtype=dtype).element_size()
        self.nbytes = int(math.prod(shape)) * itemsize
        self.buf = torch.full((2 * BAND + self.nbytes,), FILL, dtype=torch.uint8, device=DEV)
        self.t = self.buf[BAND:BAND + self.nbytes].view(dtype).view(shape)

    def check(self, what):
        torch.cuda.synchronize()
        head = self.buf[:BAND]
        tail = self.buf[BAND + self.nbytes:]
        bad_h = int((head != FILL).sum())
        bad_t = int((tail != FILL).sum())
        assert bad_h == 0 and bad_t == 0, f"{what}: {bad_h} bytes before and {bad_t} bytes after the buffer written"


def _gq(rows, cols, scales_shape, scales_dtype, recipe, layout):
    codes = Guarded((rows, cols), torch.uint8)
    scales = Guarded(scales_shape, scales_dtype)
    return codes, scales, fp8.QTensor(codes.t, scales.t, rows, cols, recipe, layout)


def _act_out(rows, cols, recipe):
    if recipe == fp8.RECIPE_BLOCKWISE:
        return _gq(rows, cols, (cols // 128, rows), torch.float32, recipe, fp8.LAYOUT_GROUP_1x128)
    return _gq(rows, cols, (fp8.mx_scale_bytes(rows, cols),), torch.uint8, recipe, fp8.LAYOUT_MX_1x32)


def _check_all(items, what):
    for i, g in enumerate(items):
        g.check(f"{what} [{i}]")


def _eq(a, b, what):
    assert torch.equal(a, b), what


@pytest.mark.parametrize("M", [1, 257, 300, 513])
def test_row_quantizers(M):
    K = 384
    X = synth.random_bf16((M, K), seed=M, outliers=True).to(DEV)
    for recipe in (fp8.RECIPE_BLOCKWISE, fp8.RECIPE_BLOCKWISE_POW2, fp8.RECIPE_MX):
        c, s, q = _act_out(M, K, recipe)
        if recipe == fp8.RECIPE_MX:
            fp8.quantize_mx(X, out=q)
            ref = fp8.quantize_mx(X)
        else:
            p2 = recipe == fp8.RECIPE_BLOCKWISE_POW2
            fp8.quantize_group(X, "K", out=q, pow2=p2)
            ref = fp8.quantize_group(X, "K", pow2=p2)
        _check_all([c, s], f"row quantizer recipe {recipe} M={M}")
        _eq(q.codes, ref.codes, "codes")
        _eq(q.scales, ref.scales, "scales")


def test_transposing_quantizers():
    M, K = 384, 200
    X = synth.random_bf16((M, K), seed=5, outliers=True).to(DEV)
    # 128x1 groups along M, codes transposed [K, M]
    for p2 in (False, True):
        if p2:
            c, s, q = _gq(K, M, (fp8.mx_scale_bytes(K, M),), torch.uint8, fp8.RECIPE_BLOCKWISE_POW2,
                          fp8.LAYOUT_MX_1x32)
        else:
            c, s, q = _gq(K, M, (M // 128, K), torch.float32, fp8.RECIPE_BLOCKWISE, fp8.LAYOUT_GROUP_1x128)
        fp8.quantize_group(X, "M", out=q, pow2=p2)
        ref = fp8.quantize_group(X, "M", pow2=p2)
        _check_all([c, s], f"128x1 pow2={p2}")
        _eq(q.codes, ref.codes, "128x1 codes")
        _eq(q.scales, ref.scales, "128x1 scales")
    # MX 32x1, codes transposed
    c, s, q = _gq(K, M, (fp8.mx_scale_bytes(K, M),), torch.uint8, fp8.RECIPE_MX, fp8.LAYOUT_MX_1x32)
    fp8.quantize_mx(X, out=q, transposed=True)
    ref = fp8.quantize_mx(X, transposed=True)
    _check_all([c, s], "MX 32x1")
    _eq(q.codes, ref.codes, "MX 32x1 codes")
    _eq(q.scales, ref.scales, "MX 32x1 scales")
    # saved 1x128 activation -> 128x1 transposed
    q1 = fp8.quantize_group(synth.random_bf16((M, 256), seed=6, outliers=True).to(DEV), "K")
    c, s, q = _gq(256, M, (M // 128, 256), torch.float32, fp8.RECIPE_BLOCKWISE, fp8.LAYOUT_GROUP_1x128)
    fp8.requantize_transposed(q1, out=q)
    ref = fp8.requantize_transposed(q1)
    _check_all([c, s], "requantize_transposed")
    _eq(q.codes, ref.codes, "requant codes")
    _eq(q.scales, ref.scales, "requant scales")


def test_block_quantizer_and_param_requant():
    N, K = 384, 640
    W = synth.random_bf16((N, K), seed=8, std=0.02).to(DEV)
    for p2 in (False, True):
        if p2:
            shp, st = (fp8.mx_scale_bytes(N, K),), torch.uint8
            shp_t = (fp8.mx_scale_bytes(K, N),)
            rec, lay = fp8.RECIPE_BLOCKWISE_POW2, fp8.LAYOUT_MX_1x32
        else:
            shp, st, shp_t = (N // 128, K // 128), torch.float32, (K // 128, N // 128)
            rec, lay = fp8.RECIPE_BLOCKWISE, fp8.LAYOUT_BLOCK_128x128
        c, s, q = _gq(N, K, shp, st, rec, lay)
        ct, stt, qt = _gq(K, N, shp_t, st, rec, lay)
        fp8.quantize_block(W, transposed=True, out=q, out_t=qt, pow2=p2)
        ref, ref_t = fp8.quantize_block(W, transposed=True, pow2=p2)
        _check_all([c, s, ct, stt], f"128x128 with transposed copy pow2={p2}")
        _eq(q.codes, ref.codes, "block codes")
        _eq(qt.codes, ref_t.codes, "block codes T")
        _eq(q.scales, ref.scales, "block scales")
        _eq(qt.scales, ref_t.scales, "block scales T")
        # fp8_param: W += dW then Q(W), Q(W)^T, from an fp32 master
        master = W.float().contiguous()
        delta = torch.full_like(master, 1e-6)
        m1, m2 = master.clone(), master.clone()
        c, s, q = _gq(N, K, shp, st, rec, lay)
        ct, stt, qt = _gq(K, N, shp_t, st, rec, lay)
        fp8.param_requantize(m1, delta, True, out=q, out_t=qt, pow2=p2)
        ref, ref_t = fp8.param_requantize(m2, delta, True, pow2=p2)
        _check_all([c, s, ct, stt], f"param_requantize pow2={p2}")
        _eq(m1, m2, "master")
        _eq(q.codes, ref.codes, "param codes")
        _eq(qt.codes, ref_t.codes, "param codes T")


@pytest.mark.parametrize("M", [1, 257, 513])
@pytest.mark.parametrize("recipe", ["blockwise", "pow2", "mx"])
def test_gemm_outputs(recipe, M):
    N, K = 384, 384
    X = synth.random_bf16((M, K), seed=M + 11, outliers=True).to(DEV)
    W = synth.random_bf16((N, K), seed=M + 12, std=0.02).to(DEV)
    if recipe == "mx":
        qa, qb = fp8.quantize_mx(X), fp8.quantize_mx(W)
        rq = fp8.RECIPE_MX
    else:
        p2 = recipe == "pow2"
        qa, qb = fp8.quantize_group(X, "K", pow2=p2), fp8.quantize_block(W, pow2=p2)
        rq = fp8.RECIPE_BLOCKWISE_POW2 if p2 else fp8.RECIPE_BLOCKWISE
    ref, ref_q = fp8.gemm(qa, qb, quantize_output=True)
    D = Guarded((M, N), torch.bfloat16)
    if rq == fp8.RECIPE_BLOCKWISE:
        c, s, q = _gq(M, N, (N // 128, M), torch.float32, rq, fp8.LAYOUT_GROUP_1x128)
    else:
        c, s, q = _gq(M, N, (fp8.mx_scale_bytes(M, N),), torch.uint8, rq, fp8.LAYOUT_MX_1x32)
    fp8.gemm(qa, qb, out=D.t, quantize_output=True, out_q=q)
    _check_all([D, c, s], f"gemm {recipe} M={M}")
    _eq(D.t, ref, "D")
    _eq(q.codes, ref_q.codes, "fused codes")
    _eq(q.scales, ref_q.scales, "fused scales")
    if recipe == "blockwise":
        D32 = Guarded((M, N), torch.float32)
        fp8.gemm(qa, qb, out=D32.t)
        D32.check(f"gemm f32 M={M}")
        _eq(D32.t, fp8.gemm(qa, qb, out_dtype=torch.float32), "D f32")


def test_backward_gemm_outputs():
    M, Nw, Kw = 384, 384, 256
    dY = synth.random_bf16((M, Nw), seed=21, std=1e-3).to(DEV)
    W = synth.random_bf16((Nw, Kw), seed=22, std=0.02).to(DEV)
    X = synth.random_bf16((M, Kw), seed=23, outliers=True).to(DEV)
    q_dy = fp8.quantize_group(dY, "K")
    _, q_wt = fp8.quantize_block(W, transposed=True)
    dX = Guarded((M, Kw), torch.bfloat16)
    fp8.gemm(q_dy, q_wt, "dgrad", out=dX.t)
    dX.check("dgrad")
    _eq(dX.t, fp8.gemm(q_dy, q_wt, "dgrad"), "dgrad D")
    q_dyt, q_xt = fp8.quantize_group(dY, "M"), fp8.quantize_group(X, "M")
    for dt in (torch.bfloat16, torch.float32):
        dW = Guarded((Nw, Kw), dt)
        fp8.gemm(q_dyt, q_xt, "wgrad", out=dW.t)
        dW.check(f"wgrad {dt}")
        _eq(dW.t, fp8.gemm(q_dyt, q_xt, "wgrad", out_dtype=dt), "wgrad D")


def test_moe_outputs():
    """Gather into expert groups of 0, 1, 77, 300 and 0 rows, fused dispatch,
    grouped GEMM: every output banded."""
    K, N = 256, 256
    sizes = [0, 1, 77, 300, 0]
    G = len(sizes)
    total = sum(sizes)
    T = 200
    X = synth.random_bf16((T, K), seed=31, outliers=True).to(DEV)
    rng = np.random.default_rng(31)
    gather = torch.from_numpy(rng.integers(0, T, total).astype(np.int32)).to(DEV)
    offsets = torch.from_numpy(np.concatenate([[0], np.cumsum(sizes)]).astype(np.int32)).to(DEV)
    gsb = fp8.mx_grouped_scale_bytes(total, K, G)
    qx = fp8.quantize_mx(X)
    c, s, q = _gq(total, K, (gsb,), torch.uint8, fp8.RECIPE_MX, fp8.LAYOUT_MX_1x32_GROUPED)
    fp8.permute_rows_mx(qx, gather, offsets, out=q)
    ref = fp8.permute_rows_mx(qx, gather, offsets)
    _check_all([c, s], "permute_rows_mx")
    _eq(q.codes, ref.codes, "permuted codes")
    _eq(q.scales, ref.scales, "permuted scales")
    # fused dispatch: token t goes to rows dst_index[t, :]; the inverse of gather
    g_np = gather.cpu().numpy()
    top_k = int(np.bincount(g_np, minlength=T).max())
    dst = torch.full((T, top_k), -1, dtype=torch.int32)
    fill = np.zeros(T, np.int64)
    for i, t in enumerate(g_np):
        dst[t, fill[t]] = i
        fill[t] += 1
    dst = dst.to(DEV)
    c2, s2, q2 = _gq(total, K, (gsb,), torch.uint8, fp8.RECIPE_MX, fp8.LAYOUT_MX_1x32_GROUPED)
    fp8.dispatch_quantize_mx(X, dst, offsets, total, out=q2)
    ref2 = fp8.dispatch_quantize_mx(X, dst, offsets, total)
    _check_all([c2, s2], "dispatch_quantize_mx")
    _eq(q2.codes, ref2.codes, "dispatch codes")
    _eq(q2.scales, ref2.scales, "dispatch scales")
    # grouped GEMM
    Wst = synth.random_bf16((G * N, K), seed=32, std=0.02).to(DEV)
    qw = fp8.quantize_mx(Wst)
    D = Guarded((total, N), torch.bfloat16)
    fp8.grouped_gemm(ref, qw, offsets, N, out=D.t)
    D.check("grouped gemm")
    _eq(D.t, fp8.grouped_gemm(ref, qw, offsets, N), "grouped D")


@pytest.mark.parametrize("recipe", [fp8.RECIPE_BLOCKWISE, fp8.RECIPE_BLOCKWISE_POW2, fp8.RECIPE_MX])
def test_fused_producer_outputs(recipe):
    M, K = 257, 384
    X = synth.random_bf16((M, K), seed=41, outliers=True).to(DEV)
    gam = synth.random_bf16((K,), seed=42).to(DEV)
    c, s, q = _act_out(M, K, recipe)
    y = Guarded((M, K), torch.bfloat16)
    rstd = Guarded((M,), torch.float32)
    fp8.rmsnorm_quantize(X, gam, 1e-6, recipe, want_y=True, want_rstd=True, out=q, y=y.t, rstd=rstd.t)
    ref, ref_y, ref_r = fp8.rmsnorm_quantize(X, gam, 1e-6, recipe, want_y=True, want_rstd=True)
    _check_all([c, s, y, rstd], f"rmsnorm recipe {recipe}")
    _eq(q.codes, ref.codes, "rmsnorm codes")
    _eq(y.t, ref_y, "rmsnorm y")
    _eq(rstd.t, ref_r, "rmsnorm rstd")
    F = 384
    GU = synth.random_bf16((M, 2 * F), seed=43).to(DEV)
    c, s, q = _act_out(M, F, recipe)
    h = Guarded((M, F), torch.bfloat16)
    fp8.swiglu_quantize(GU, recipe, want_h=True, out=q, h=h.t)
    ref, ref_h = fp8.swiglu_quantize(GU, recipe, want_h=True)
    _check_all([c, s, h], f"swiglu recipe {recipe}")
    _eq(q.codes, ref.codes, "swiglu codes")
    _eq(h.t, ref_h, "swiglu h")


def test_sync_install_destinations():
    W = synth.random_bf16((384, 512), seed=51, std=0.02).to(DEV)
    X = synth.random_bf16((257, 256), seed=52, outliers=True).to(DEV)
    qw, qx, qm = fp8.quantize_block(W), fp8.quantize_group(X, "K"), fp8.quantize_mx(X)
    entries = [fp8.SyncEntry(1, qw), fp8.SyncEntry(2, qx), fp8.SyncEntry(3, qm)]
    payload = fp8.sync_pack(entries)
    outs, dst = [], []
    for tag, t in ((1, qw), (2, qx), (3, qm)):
        c = Guarded(tuple(t.codes.shape), t.codes.dtype)
        s = Guarded(tuple(t.scales.shape), t.scales.dtype)
        outs += [c, s]
        dst.append(fp8.SyncEntry(tag, fp8.QTensor(c.t, s.t, t.rows, t.cols, t.recipe, t.layout)))
    fp8.sync_install(payload, dst)
    _check_all(outs, "sync install")
    for e, t in zip(dst, (qw, qx, qm)):
        _eq(e.tensor.codes, t.codes, "installed codes")
        _eq(e.tensor.scales, t.scales, "installed scales")
