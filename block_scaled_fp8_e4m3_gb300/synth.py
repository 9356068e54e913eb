"""Seeded synthetic inputs shaped like the linear layers the pages discuss.

This module only draws random numbers; it holds none of the quantization or
GEMM arithmetic, and it is the one piece shared by the CPU oracle's tests and
the CUDA path's tests and benchmark.  Every tensor is drawn on the host with
``torch.Generator().manual_seed(seed)`` in fp32, in the order listed for each
workload, then rounded to bf16 (round to nearest even).

Workloads (matrices follow torch ``nn.Linear``: X [M,K], W [N,K], Y = X W^T):

* ``tiny``      seed 0: X [128,512] ~N(0,1) + outliers, W [512,512] ~N(0,0.02)
* ``mx``        seed 1: X [2048,4096] + outliers, W [4096,4096] ~N(0,0.02)
* ``mlp``       seed 2: X [8192,4096] + outliers, W [12288,4096] ~N(0,0.02)
* ``backward``  seed 3: dY [8192,4096] ~N(0,1e-3), W [4096,4096] ~N(0,0.02),
                X [8192,4096] ~N(0,1) + outliers
* ``moe``       seed 4: top-8 routing of 16384 tokens over 64 experts with
                Zipf(1.1) expert popularity, then X [16384,2048] ~N(0,1),
                W [64,1024,2048] ~N(0,0.02)
* ``fp8_param`` seed 5: fp32 master W [12288,4096] ~N(0,0.02) (kept in
                fp32), then one optimizer update dW = 1e-6 * (+-1) with
                independent fair signs: an Adam-like step whose magnitude is
                the learning rate (the pages report max |dW| = 1.01e-6 and a
                mean relative update of 0.6-0.9e-4; 1e-6 / E|W| = 0.63e-4)

"Outliers": exactly round(0.001 * numel) distinct positions, drawn uniformly
without replacement (``randperm``), are multiplied by 50 before the bf16
rounding.
"""
from __future__ import annotations

import hashlib
from dataclasses import dataclass, field

import torch

OUTLIER_FRACTION = 0.001
OUTLIER_FACTOR = 50.0


def _gen(seed: int) -> torch.Generator:
    g = torch.Generator()
    g.manual_seed(seed)
    return g


def normal_bf16(shape, std: float, gen: torch.Generator, outliers: bool = False) -> torch.Tensor:
    x = torch.randn(*shape, generator=gen, dtype=torch.float32)
    if std != 1.0:
        x.mul_(std)
    if outliers:
        n = x.numel()
        count = int(round(OUTLIER_FRACTION * n))
        pos = torch.randperm(n, generator=gen)[:count]
        x.view(-1)[pos] *= OUTLIER_FACTOR
    return x.to(torch.bfloat16)


@dataclass
class Workload:
    name: str
    seed: int
    tensors: dict = field(default_factory=dict)
    meta: dict = field(default_factory=dict)

    def sha256(self) -> str:
        h = hashlib.sha256()
        for k in sorted(self.tensors):
            t = self.tensors[k].contiguous()
            h.update(k.encode())
            h.update(t.view(torch.uint8).numpy().tobytes() if t.dtype != torch.bfloat16
                     else t.view(torch.int16).numpy().tobytes())
        return h.hexdigest()


def tiny() -> Workload:
    g = _gen(0)
    X = normal_bf16((128, 512), 1.0, g, outliers=True)
    W = normal_bf16((512, 512), 0.02, g)
    return Workload("tiny blockwise 128x512x512", 0, {"X": X, "W": W})


def mx() -> Workload:
    g = _gen(1)
    X = normal_bf16((2048, 4096), 1.0, g, outliers=True)
    W = normal_bf16((4096, 4096), 0.02, g)
    return Workload("MXFP8 forward 2048x4096x4096", 1, {"X": X, "W": W})


def mlp() -> Workload:
    g = _gen(2)
    X = normal_bf16((8192, 4096), 1.0, g, outliers=True)
    W = normal_bf16((12288, 4096), 0.02, g)
    return Workload("dense MLP forward + sync 8192x4096x12288", 2, {"X": X, "W": W})


def backward() -> Workload:
    g = _gen(3)
    dY = normal_bf16((8192, 4096), 1e-3, g)
    W = normal_bf16((4096, 4096), 0.02, g)
    X = normal_bf16((8192, 4096), 1.0, g, outliers=True)
    return Workload("blockwise backward DGrad+WGrad 8192x4096x4096", 3,
                    {"dY": dY, "W": W, "X": X})


def moe_routing(gen: torch.Generator, tokens: int, experts: int, top_k: int, zipf_s: float):
    """Top-k routing with Zipf expert popularity.  Returns (gather index into
    the token rows, int32 group offsets [experts+1], per-(token,slot) expert
    ids, int32 [tokens, top_k] destination row of every (token, slot) -- the
    inverse of gather).  Rows are ordered by expert, then token (a stable
    sort)."""
    ranks = torch.arange(1, experts + 1, dtype=torch.float64)
    p_rank = ranks.pow(-zipf_s)
    p_rank = p_rank / p_rank.sum()
    expert_of_rank = torch.randperm(experts, generator=gen)
    p = torch.empty(experts, dtype=torch.float64)
    p[expert_of_rank] = p_rank
    choice = torch.multinomial(p.to(torch.float32).expand(tokens, experts).contiguous(), top_k,
                               replacement=False, generator=gen)          # [tokens, top_k]
    flat_expert = choice.reshape(-1)
    flat_token = torch.arange(tokens).repeat_interleave(top_k)
    # stable sort by expert, then token (flat order is token-major already)
    order = torch.argsort(flat_expert, stable=True)
    gather = flat_token[order].to(torch.int32)
    counts = torch.bincount(flat_expert, minlength=experts)
    offsets = torch.zeros(experts + 1, dtype=torch.int32)
    offsets[1:] = torch.cumsum(counts, 0).to(torch.int32)
    dst_index = torch.empty_like(order)
    dst_index[order] = torch.arange(order.numel())
    return gather, offsets, choice, dst_index.reshape(tokens, top_k).to(torch.int32)


def moe(tokens: int = 16384, experts: int = 64, top_k: int = 8, hidden: int = 2048,
        ffn: int = 1024, seed: int = 4) -> Workload:
    g = _gen(seed)
    gather, offsets, choice, dst_index = moe_routing(g, tokens, experts, top_k, 1.1)
    X = normal_bf16((tokens, hidden), 1.0, g)
    W = normal_bf16((experts, ffn, hidden), 0.02, g)
    return Workload(f"MoE grouped MXFP8 {tokens}x{top_k} tokens, {experts} experts, "
                    f"{ffn}x{hidden}", seed,
                    {"X": X, "W": W, "gather": gather, "offsets": offsets, "dst_index": dst_index},
                    {"tokens": tokens, "experts": experts, "top_k": top_k})


def fp32_master(shape, seed: int, std: float = 0.02) -> torch.Tensor:
    """fp32 master weights ~N(0, std), not rounded to bf16."""
    x = torch.randn(*shape, generator=_gen(seed), dtype=torch.float32)
    return x.mul_(std)


def sign_updates(shape, seed: int, lr: float = 1e-6, gen: torch.Generator = None, device=None) -> torch.Tensor:
    """lr * (+-1) with independent fair signs, fp32 (on `device` with `gen`
    when given, for long update sequences drawn where they are used)."""
    g = gen if gen is not None else _gen(seed)
    b = torch.randint(0, 2, tuple(shape), generator=g, dtype=torch.int32, device=device)
    return (b.to(torch.float32) * 2.0 - 1.0).mul_(lr)


def fp8_param(N: int = 12288, K: int = 4096, seed: int = 5, lr: float = 1e-6) -> Workload:
    g = _gen(seed)
    W = torch.randn(N, K, generator=g, dtype=torch.float32).mul_(0.02)
    dW = sign_updates((N, K), seed, lr, gen=g)
    return Workload(f"fp8_param {N}x{K}", seed, {"W": W, "dW": dW}, {"lr": lr})


def random_bf16(shape, seed: int, std: float = 1.0, outliers: bool = False) -> torch.Tensor:
    """Small seeded tensor for parity cases at arbitrary shapes."""
    return normal_bf16(shape, std, _gen(seed), outliers=outliers)


def bf16_bits(t: torch.Tensor):
    """bf16 tensor -> numpy uint16 bit patterns (for the oracle)."""
    import numpy as np
    return t.contiguous().view(torch.int16).numpy().view(np.uint16)
