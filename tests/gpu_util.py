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
