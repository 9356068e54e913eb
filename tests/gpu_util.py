"""Helpers for the GPU parity tests: run the CUDA path through the Python
binding (which calls the C ABI) and compare with the CPU oracle on the same
seeded inputs."""
import numpy as np
import torch

import oracle
from block_scaled_fp8_e4m3_gb300 import synth

DEV = "cuda:0"


def to_np(t: torch.Tensor) -> np.ndarray:
    t = t.detach().cpu().contiguous()
    if t.dtype == torch.bfloat16:
        return t.view(torch.int16).numpy().view(np.uint16)
    return t.numpy()


def bf16_dev_to_f64(t: torch.Tensor) -> np.ndarray:
    return t.detach().float().cpu().numpy().astype(np.float64)


def assert_bytes_equal(gpu, ref, what):
    g = np.ascontiguousarray(gpu)
    r = np.ascontiguousarray(ref)
    assert g.shape == r.shape, f"{what}: shape {g.shape} vs {r.shape}"
    if g.dtype != r.dtype:
        g = g.view(np.uint8)
        r = r.view(np.uint8)
    bad = np.nonzero(g.view(np.uint8).ravel() != r.view(np.uint8).ravel())[0]
    assert bad.size == 0, (f"{what}: {bad.size} of {g.nbytes} bytes differ; first at byte {bad[:8].tolist()}: "
                           f"gpu {g.view(np.uint8).ravel()[bad[:8]].tolist()} "
                           f"oracle {r.view(np.uint8).ravel()[bad[:8]].tolist()}")


def assert_gemm_close(gpu, ref, mag, what):
    """|gpu - ref| <= 2e-3 * sum_k |a b| + 2^-8 * |ref| per element."""
    gpu = np.asarray(gpu, np.float64)
    tol = oracle.gemm_tolerance(ref, mag)
    err = np.abs(gpu - ref)
    bad = np.nonzero(~(err <= tol))
    assert bad[0].size == 0, (f"{what}: {bad[0].size} of {gpu.size} outside tolerance; worst "
                              f"err/tol {float(np.max(err / np.maximum(tol, 1e-300))):.3g} at "
                              f"{[int(b[0]) for b in bad]}: gpu {gpu[tuple(b[0] for b in bad)]} "
                              f"ref {ref[tuple(b[0] for b in bad)]}")


def oracle_group_k(x: torch.Tensor):
    return oracle.quant_group_1x128(synth.bf16_bits(x))


def oracle_group_m(x: torch.Tensor):
    return oracle.quant_group_128x1_T(synth.bf16_bits(x))


def oracle_block(w: torch.Tensor, transposed=False):
    return oracle.quant_block_128x128(synth.bf16_bits(w), transposed=transposed)


def oracle_mx(x: torch.Tensor):
    return oracle.quant_mx_1x32(synth.bf16_bits(x))


def stratified_positions(M: int, N: int, per_tile: int = 16, tile: int = 256, seed: int = 0,
                         row_segments=None):
    """Output positions for a sampled GEMM check: every tile x tile block of
    the output (tiles start at each row segment's first row when
    row_segments = [(start, end), ...] is given, as the grouped GEMM tiles
    each expert's rows) contributes its four corners and per_tile - 4
    uniform positions.  A wrong tile cannot escape the check."""
    rng = np.random.default_rng(seed)
    segs = row_segments if row_segments is not None else [(0, M)]
    ms, ns = [], []
    extra = max(per_tile - 4, 0)
    for s0, s1 in segs:
        for t0 in range(s0, s1, tile):
            t1 = min(s1, t0 + tile)
            for u0 in range(0, N, tile):
                u1 = min(N, u0 + tile)
                ms.extend([t0, t0, t1 - 1, t1 - 1])
                ns.extend([u0, u1 - 1, u0, u1 - 1])
                ms.extend(rng.integers(t0, t1, extra).tolist())
                ns.extend(rng.integers(u0, u1, extra).tolist())
    return np.asarray(ms, np.int64), np.asarray(ns, np.int64)


def sampled_gemm_check(Y: torch.Tensor, A_deq, B_deq, what: str, seed: int = 0, per_tile: int = 16):
    """Y = A B^T checked at stratified positions against the oracle's fp64
    reference of those outputs."""
    M, N = Y.shape
    ms, ns = stratified_positions(M, N, per_tile=per_tile, seed=seed)
    ref, mag = oracle.gemm_ref_sampled(A_deq, B_deq, ms, ns)
    got = Y[torch.from_numpy(ms).to(Y.device), torch.from_numpy(ns).to(Y.device)].double().cpu().numpy()
    assert_gemm_close(got, ref, mag, what)
