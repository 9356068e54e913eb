"""Displacement diagnostics for fp8_param: does re-quantizing the fp32
master after every optimizer step lose the small RL updates?

[SkyRL] "Deep dive: FP8 quantization with FP32 and power-of-two block
scales", Figure 12.  Left: the cumulative displacement of the FP8 storage
over many steps, in units of the master's own displacement; right: the
cosine similarity between one master update and the change it causes in the
FP8 storage, against the update's size.  The steps run through
``param_requantize`` (the fused W += dW and Q(W) kernel); the analysis below
(dequantization, sums) is plain torch on the device: an experiment run by
``bench.py --experiment fp8_param_drift``, kept outside the library package.

Readings: the updates are Adam-like, lr * (+-1) with independent fair signs;
"displacement normalized by the master's" is taken as the projection
<D, M> / <M, M> of the FP8 displacement D = deq(Q(W_T)) - deq(Q(W_0)) on the
master's M = W_T - W_0, which is 1 when the storage follows the master on
average (an update that the quantization dropped would pull it below 1).
The L1 and L2 ratios are reported beside it.
"""
from __future__ import annotations

import torch

from block_scaled_fp8_e4m3_gb300 import LAYOUT_MX_1x32, QTensor, param_requantize, synth


def dequantize_block(q: QTensor) -> torch.Tensor:
    """fp64 values of a 128x128-block FP8 weight (fp32 or power-of-two scales)."""
    R, K = q.rows, q.cols
    v = q.codes.view(torch.float8_e4m3fn).to(torch.float64)
    if q.layout == LAYOUT_MX_1x32:   # power-of-two exponents: every byte of a block's atom holds it
        e = q.scales.view(-1, 512)[:, 0].to(torch.int32).view(R // 128, K // 128) - 127
        s = torch.pow(torch.tensor(2.0, dtype=torch.float64, device=v.device), e.to(torch.float64))
    else:
        s = q.scales.view(R // 128, K // 128).to(torch.float64)
    return v * s.repeat_interleave(128, 0).repeat_interleave(128, 1)


def _ratios(D: torch.Tensor, M: torch.Tensor) -> dict:
    mm = float((M * M).sum())
    return {"projection": float((D * M).sum()) / mm,
            "l1": float(D.abs().sum()) / float(M.abs().sum()),
            "l2": float(torch.linalg.vector_norm(D)) / mm ** 0.5,
            "changed_fraction": float((D != 0).double().mean())}


def cumulative_displacement(master0: torch.Tensor, steps: int, lr: float = 1e-6, pow2: bool = False,
                            seed: int = 0, checkpoints=()) -> dict:
    """Runs `steps` updates W += lr * (+-1) with re-quantization after each
    and returns the displacement ratios at the end (and at `checkpoints`)."""
    W = master0.clone()
    q = param_requantize(W, pow2=pow2)
    D0 = dequantize_block(q)
    W0 = master0.to(torch.float64)
    gen = torch.Generator(device=W.device)
    gen.manual_seed(seed)
    dW = torch.empty_like(W)
    out = {}
    for t in range(1, steps + 1):
        dW.copy_(synth.sign_updates(W.shape, seed, lr, gen=gen, device=W.device))
        param_requantize(W, dW, out=q, pow2=pow2)
        if t == steps or t in checkpoints:
            out[t] = _ratios(dequantize_block(q) - D0, W.to(torch.float64) - W0)
    return out


def single_step_cosine(master: torch.Tensor, magnitudes, pow2: bool = False, seed: int = 0) -> list:
    """cos(deq(Q(W + dW)) - deq(Q(W)), dW) for one update of each size."""
    D0 = dequantize_block(param_requantize(master.clone(), pow2=pow2))
    gen = torch.Generator(device=master.device)
    gen.manual_seed(seed)
    rows = []
    for m in magnitudes:
        W = master.clone()
        dW = synth.sign_updates(W.shape, seed, float(m), gen=gen, device=W.device)
        D = dequantize_block(param_requantize(W, dW, pow2=pow2)) - D0
        M = W.to(torch.float64) - master.to(torch.float64)
        nd = float(torch.linalg.vector_norm(D))
        cos = float((D * M).sum()) / (nd * float(torch.linalg.vector_norm(M))) if nd > 0 else 0.0
        rows.append({"magnitude": float(m), "cosine": cos, **{k: v for k, v in _ratios(D, M).items()
                                                               if k in ("projection", "changed_fraction")}})
    return rows
