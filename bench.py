#!/usr/bin/env python3
"""Benchmark of the block-scaled FP8 hot path on GB300.

One step = one pass of the dense-MLP workload (X [8192,4096] bf16 with 0.1%
x50 outliers, W [12288,4096] ~N(0,0.02), seed 2):
  1x128 quantize X -> 128x128 quantize W -> blockwise FP8 GEMM Y = X W^T
  (fp32 accumulate, bf16 out, 1x128 quantization of Y fused in the epilogue)
  -> weight-sync pack of W -> install into the rollout copy.
value = GEMM FLOPs (2 M N K) per step / device time per step, inputs resident
in HBM; L2 (129 MB) is flushed between steps by writing 256 MB.

Also reported: the dominant kernel's roofline (GEMM against the FP8 dense
peak = 2 x measured bf16 peak), every kernel's own roofline over all
workloads ("kernels"), an end-to-end number through the public API with
host buffers ("e2e"), the CPU oracle on a bounded sample ("cpu_baseline"),
SM clocks sampled during the timed region, and the kernel launch count.

--impl reference times the CPU oracle (the only reference this project
has) on a bounded sample of the same workload per step.
Multi-GPU: replicas only (each rank runs the same independent workload;
no data-path collective); value sums over ranks.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import time

import numpy as np
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "block-scaled FP8 GEMM TFLOP/s + quantize GB/s, % of GB300 roofline"
WORKLOAD = "dense MLP forward + weight sync: X 8192x4096 (1x128), W 12288x4096 (128x128), GEMM 8192x4096x12288"
M, K, N = 8192, 4096, 12288
L2_FLUSH_BYTES = 256 << 20


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return {"hbm_gbs": float(d["hbm_gbs"]), "bf16_tflops": float(d["bf16_tflops"]),
                "bf16_tflops_sustained": float(d.get("bf16_tflops_sustained", d["bf16_tflops"])),
                "source": "measured"}
    except Exception:
        return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0, "source": "fallback"}


# ------------------------------------------------------------------ ranks
def max_over_ranks(x: float, world: int, device) -> float:
    """The largest of the ranks' values (the slowest rank's time); x as is
    for one rank."""
    if world <= 1:
        return x
    t = torch.tensor([x], device=device, dtype=torch.float64)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return float(t.item())


def whole_job_tflops(flops_per_rank_step: float, ms_per_step: float, world: int) -> float:
    """Throughput of the whole job: every rank processes its own step, the
    job's step time is the slowest rank's."""
    return world * flops_per_rank_step / (ms_per_step * 1e-3) / 1e12


# ------------------------------------------------------------------ clocks
class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.proc = None
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits", "-lms", "50",
                 "-i", str(gpu_index)], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except Exception:
            self.proc.kill()
            out, _ = self.proc.communicate()
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in out.strip().splitlines():
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                mx.append(float(parts[2]))
            except ValueError:
                continue
            for nm, v in zip(names, parts[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(nm)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "samples": len(sm),
                "reasons": sorted(reasons)}


# ------------------------------------------------------------------ timing helpers
class Flusher:
    """Writes a buffer larger than L2, then reads another one, so that the
    timed kernel starts with no data of its own and no dirty lines in L2
    (the write-backs of the flush itself stay outside the timed region)."""

    def __init__(self, dev):
        self.buf = torch.empty(L2_FLUSH_BYTES // 4, dtype=torch.float32, device=dev)
        self.rbuf = torch.ones(L2_FLUSH_BYTES // 4, dtype=torch.float32, device=dev)
        self.sink = torch.empty((), dtype=torch.float32, device=dev)

    def __call__(self):
        self.buf.fill_(1.0)
        torch.sum(self.rbuf, dim=0, out=self.sink)


def time_kernel(fn, flush, reps, warmup=3):
    """Device time (ms) of fn(), L2 flushed before each launch: the mean of
    reps CUDA-event pairs with the lowest and highest 10 % dropped.  The
    events' clock ticks in steps of about 2 us on this GPU, so a median of
    ~20 us launches would sit on that grid; the mean of many pairs, whose
    start falls at random within a tick, does not."""
    for _ in range(warmup):
        flush()
        fn()
    ts = []
    for _ in range(reps):
        flush()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        fn()
        e1.record()
        ts.append((e0, e1))
    torch.cuda.synchronize()
    d = np.sort([a.elapsed_time(b) for a, b in ts])
    k = len(d) // 10
    return float(np.mean(d[k:len(d) - k]))


def gemm_traffic():
    """DRAM bytes (read + write) per launch of the step's GEMM, from the
    machine-readable ncu record under profiles/, or None when the kernel
    source has changed since those counters were taken (the record holds the
    sha256 of gemm_blockwise.cu)."""
    import hashlib
    here = os.path.dirname(os.path.abspath(__file__))
    record = os.path.join(here, "profiles", "k_gemm_blockwise_traffic.json")
    src = os.path.join(here, "block_scaled_fp8_e4m3_gb300", "csrc", "gemm_blockwise.cu")
    try:
        with open(record) as f:
            d = json.load(f)
        digest = hashlib.sha256(open(src, "rb").read()).hexdigest()
    except (OSError, ValueError):
        return None
    if d.get("gemm_blockwise_cu_sha256") != digest or "traffic_bytes_per_launch" not in d:
        return None
    return int(d["traffic_bytes_per_launch"])


# ------------------------------------------------------------------ our arm
def make_step(fp8, X, W, dev):
    qx = fp8.quantize_group(X, "K")
    qw = fp8.quantize_block(W)
    Y, qy = fp8.gemm(qx, qw, "fwd", quantize_output=True)
    payload = fp8.sync_pack([fp8.SyncEntry(1, qw)])
    rollout = fp8.QTensor(torch.empty_like(qw.codes), torch.empty_like(qw.scales), qw.rows, qw.cols, qw.recipe,
                          qw.layout)
    torch.cuda.synchronize()

    def step(events=None):
        rec = (lambda i: events[i].record()) if events is not None else (lambda i: None)
        rec(0)
        fp8.quantize_group(X, "K", out=qx)
        rec(1)
        fp8.quantize_block(W, out=qw)
        rec(2)
        fp8.gemm(qx, qw, "fwd", quantize_output=True, out=Y, out_q=qy)
        rec(3)
        fp8.sync_pack([fp8.SyncEntry(1, qw)], payload=payload)
        rec(4)
        fp8.sync_install(payload, [fp8.SyncEntry(1, rollout)], check=False)
        rec(5)
        return Y

    return step, payload.numel(), (qx, qw, Y, qy, rollout)


KERNELS_PER_STEP = 5   # quant X, quant W, GEMM, pack, install (one cooperative launch)


def breakdown(fp8, synth, dev, flush, pk, reps):
    """Every kernel of the hot path on its own workload, against its roofline."""
    hbm = pk["hbm_gbs"]
    fp8_peak = 2.0 * pk["bf16_tflops"]
    out = {}
    copy_ms = {}

    def same_size_copy_ms(nbytes):
        """Device time of a plain tensor copy moving the same bytes (half read,
        half written): what a launch of this size reaches in practice, as
        context beside the fraction of the sustained copy bandwidth."""
        half = (int(nbytes) // 2 + 15) // 16 * 16
        if half not in copy_ms:
            src = torch.empty(half, dtype=torch.uint8, device=dev).fill_(3)
            dst = torch.empty_like(src)
            copy_ms[half] = time_kernel(lambda: dst.copy_(src), flush, reps)
            del src, dst
        return copy_ms[half]

    def rec(name, ms, bytes_=None, flops=None, workload=""):
        d = {"ms": round(ms, 5), "workload": workload}
        if bytes_ is not None:
            gbs = bytes_ / (ms * 1e-3) / 1e9
            cms = same_size_copy_ms(bytes_)
            d.update(bound="hbm", achieved=round(gbs, 1), unit="GB/s", peak=hbm, frac=round(gbs / hbm, 4),
                     frac_of_8tbs=round(gbs / 8000.0, 4), algorithmic_bytes=int(bytes_),
                     same_size_copy_ms=round(cms, 5), frac_of_same_size_copy=round(cms / ms, 4))
        else:
            tf = flops / (ms * 1e-3) / 1e12
            d.update(bound="tensor", achieved=round(tf, 1), unit="TFLOP/s", peak=round(fp8_peak, 1),
                     frac=round(tf / fp8_peak, 4), algorithmic_flops=int(flops))
        out[name] = d

    # tiny blockwise configuration (X 128x512, W 512x512): launch-latency bound,
    # reported without a roofline; eager, and replayed as one CUDA graph (the
    # quantize + GEMM part, and the whole step with pack and install)
    wl = synth.tiny()
    Xt, Wt = wl.tensors["X"].to(dev), wl.tensors["W"].to(dev)
    qxt, qwt = fp8.quantize_group(Xt, "K"), fp8.quantize_block(Wt)
    Yt = fp8.gemm(qxt, qwt)
    pt = fp8.sync_pack([fp8.SyncEntry(1, qwt)])
    rt = fp8.QTensor(torch.empty_like(qwt.codes), torch.empty_like(qwt.scales), qwt.rows, qwt.cols, qwt.recipe,
                     qwt.layout)

    def tiny_compute():
        fp8.quantize_group(Xt, "K", out=qxt)
        fp8.quantize_block(Wt, out=qwt)
        fp8.gemm(qxt, qwt, out=Yt)

    def tiny_step():
        tiny_compute()
        fp8.sync_pack([fp8.SyncEntry(1, qwt)], payload=pt)
        fp8.sync_install(pt, [fp8.SyncEntry(1, rt)], check=False)

    out["tiny_step_eager"] = {"ms": round(time_kernel(tiny_step, flush, reps), 5), "bound": "launch",
                              "workload": "X 128x512 1x128, W 512x512 128x128, GEMM 128x512x512, pack + install W"}
    out["tiny_quant_gemm_eager"] = {"ms": round(time_kernel(tiny_compute, flush, reps), 5), "bound": "launch",
                                    "workload": "quantize X and W, GEMM 128x512x512"}
    try:
        side = torch.cuda.Stream(device=dev)
        side.wait_stream(torch.cuda.current_stream(dev))
        with torch.cuda.stream(side):
            tiny_compute()
        torch.cuda.current_stream(dev).wait_stream(side)
        torch.cuda.synchronize()
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph):
            tiny_compute()
        out["tiny_quant_gemm_graph"] = {"ms": round(time_kernel(graph.replay, flush, reps), 5), "bound": "launch",
                                        "workload": "the same three kernels replayed as one CUDA graph"}
        del graph
    except Exception as e:  # noqa: BLE001 - reported, the rest of the breakdown still runs
        out["tiny_quant_gemm_graph"] = {"error": str(e).splitlines()[0][:200]}
    try:
        torch.cuda.synchronize()
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph):
            tiny_step()
        out["tiny_step_graph"] = {"ms": round(time_kernel(graph.replay, flush, reps), 5), "bound": "launch",
                                  "workload": "the five-kernel step (with pack and install) replayed as one CUDA graph"}
        del graph
    except Exception as e:  # noqa: BLE001
        out["tiny_step_graph"] = {"error": str(e).splitlines()[0][:200]}
    del Xt, Wt, qxt, qwt, Yt, pt, rt

    # dense MLP forward + sync
    wl = synth.mlp()
    X, W = wl.tensors["X"].to(dev), wl.tensors["W"].to(dev)
    qx = fp8.quantize_group(X, "K")
    qw = fp8.quantize_block(W)
    rec("quant_group_1x128", time_kernel(lambda: fp8.quantize_group(X, "K", out=qx), flush, reps),
        bytes_=M * K * (3 + 4 / 128), workload="X 8192x4096")
    rec("quant_block_128x128", time_kernel(lambda: fp8.quantize_block(W, out=qw), flush, reps),
        bytes_=N * K * (3 + 4 / 16384), workload="W 12288x4096")
    Y = torch.empty((M, N), dtype=torch.bfloat16, device=dev)
    rec("gemm_blockwise_fwd", time_kernel(lambda: fp8.gemm(qx, qw, out=Y), flush, reps),
        flops=2.0 * M * N * K, workload="8192x4096x12288")
    Y2, qy = fp8.gemm(qx, qw, quantize_output=True)
    rec("gemm_blockwise_fwd_fused_quant",
        time_kernel(lambda: fp8.gemm(qx, qw, quantize_output=True, out=Y2, out_q=qy), flush, reps),
        flops=2.0 * M * N * K, workload="8192x4096x12288 + 1x128 quant of Y")
    payload = fp8.sync_pack([fp8.SyncEntry(1, qw)])
    rollout = fp8.QTensor(torch.empty_like(qw.codes), torch.empty_like(qw.scales), qw.rows, qw.cols, qw.recipe,
                          qw.layout)
    pb = payload.numel()
    rec("sync_pack", time_kernel(lambda: fp8.sync_pack([fp8.SyncEntry(1, qw)], payload=payload), flush, reps),
        bytes_=2 * pb, workload=f"W 12288x4096 payload {pb} B")
    rec("sync_install", time_kernel(lambda: fp8.sync_install(payload, [fp8.SyncEntry(1, rollout)], check=False),
                                    flush, reps),
        bytes_=2 * pb, workload=f"W 12288x4096 payload {pb} B")
    # the same forward with power-of-two block scales: the GEMM runs on the
    # block-scaled MMA (no promotion)
    px = fp8.quantize_group(X, "K", pow2=True)
    pw = fp8.quantize_block(W, pow2=True)
    rec("quant_group_1x128_pow2", time_kernel(lambda: fp8.quantize_group(X, "K", out=px, pow2=True), flush, reps),
        bytes_=M * K * (3 + 4 / 128), workload="X 8192x4096, power-of-two scales")
    rec("quant_block_128x128_pow2", time_kernel(lambda: fp8.quantize_block(W, out=pw, pow2=True), flush, reps),
        bytes_=N * K * (3 + 1 / 32), workload="W 12288x4096, power-of-two scales")
    rec("gemm_blockwise_pow2_fwd", time_kernel(lambda: fp8.gemm(px, pw, out=Y), flush, reps),
        flops=2.0 * M * N * K, workload="8192x4096x12288, power-of-two scales")
    Y3, qy3 = fp8.gemm(px, pw, quantize_output=True)
    rec("gemm_blockwise_pow2_fwd_fused_quant",
        time_kernel(lambda: fp8.gemm(px, pw, quantize_output=True, out=Y3, out_q=qy3), flush, reps),
        flops=2.0 * M * N * K, workload="8192x4096x12288 + 1x128 power-of-two quant of Y")
    del X, W, qx, qw, Y, Y2, qy, payload, rollout, px, pw, Y3, qy3
    torch.cuda.empty_cache()

    # fp8_param: Q(W) of the fp32 master, alone and fused with the update
    wl = synth.fp8_param()
    Wm, dW = wl.tensors["W"].to(dev), wl.tensors["dW"].to(dev)
    for p2 in (False, True):
        sfx = "_pow2" if p2 else ""
        qm, qmt = fp8.param_requantize(Wm, transposed=True, pow2=p2)
        sb = N * K / 16384 * (512 if p2 else 4)
        rec("param_requant" + sfx, time_kernel(lambda: fp8.param_requantize(Wm, out=qm, pow2=p2), flush, reps),
            bytes_=N * K * 5 + sb, workload="fp32 master W 12288x4096 -> FP8" + (", power-of-two scales" if p2 else ""))
        rec("param_update_requant_with_T" + sfx,
            time_kernel(lambda: fp8.param_requantize(Wm, dW, True, out=qm, out_t=qmt, pow2=p2), flush, reps),
            bytes_=N * K * 14 + 2 * sb,
            workload="W += dW (fp32) then FP8 W and W^T, 12288x4096" + (", power-of-two scales" if p2 else ""))
    del Wm, dW, qm, qmt
    torch.cuda.empty_cache()

    # producers fused with the activation quantization
    X = synth.mlp().tensors["X"].to(dev)
    gam = torch.ones((K,), dtype=torch.bfloat16, device=dev)
    for rc, nm in ((fp8.RECIPE_BLOCKWISE, ""), (fp8.RECIPE_MX, "_mx")):
        qn = fp8.rmsnorm_quantize(X, gam, 1e-6, rc)
        sbytes = 4 / 128 if rc == fp8.RECIPE_BLOCKWISE else 1 / 32
        rec("rmsnorm_quant" + nm, time_kernel(lambda: fp8.rmsnorm_quantize(X, gam, 1e-6, rc, out=qn), flush, reps),
            bytes_=M * K * (3 + sbytes), workload="RMSNorm of X 8192x4096 -> FP8" + (" MX" if nm else " 1x128"))
    GU = torch.empty((M, N), dtype=torch.bfloat16, device=dev).normal_(0.0, 1.5)
    for rc, nm in ((fp8.RECIPE_BLOCKWISE, ""), (fp8.RECIPE_MX, "_mx")):
        qs = fp8.swiglu_quantize(GU, rc)
        sbytes = 4 / 128 if rc == fp8.RECIPE_BLOCKWISE else 1 / 32
        rec("swiglu_quant" + nm, time_kernel(lambda: fp8.swiglu_quantize(GU, rc, out=qs), flush, reps),
            bytes_=M * (N // 2) * (5 + sbytes),
            workload="SwiGLU of the 8192x12288 up projection -> FP8 8192x6144" + (" MX" if nm else " 1x128"))
    del X, gam, qn, GU, qs
    torch.cuda.empty_cache()

    # backward
    wl = synth.backward()
    dY, Wb, Xb = (wl.tensors[k].to(dev) for k in ("dY", "W", "X"))
    q_dy = fp8.quantize_group(dY, "K")
    q_w, q_wt = fp8.quantize_block(Wb, transposed=True)
    q_dyt = fp8.quantize_group(dY, "M")
    q_xt = fp8.quantize_group(Xb, "M")
    Mb, Nb, Kb = 8192, 4096, 4096
    rec("quant_group_128x1_T", time_kernel(lambda: fp8.quantize_group(Xb, "M", out=q_xt), flush, reps),
        bytes_=Mb * Kb * (3 + 4 / 128), workload="X 8192x4096 -> X^T")
    q_x1 = fp8.quantize_group(Xb, "K")
    q_xr = fp8.requantize_transposed(q_x1)
    rec("requant_1x128_to_128x1_T", time_kernel(lambda: fp8.requantize_transposed(q_x1, out=q_xr), flush, reps),
        bytes_=Mb * Kb * (2 + 8 / 128), workload="saved FP8 X 8192x4096 (1x128) -> X^T 128x1")
    del q_x1, q_xr
    rec("quant_block_128x128_with_T", time_kernel(lambda: fp8.quantize_block(Wb, True, out=q_w, out_t=q_wt),
                                                  flush, reps),
        bytes_=Nb * Kb * (4 + 8 / 16384), workload="W 4096x4096 + transposed copy")
    dX = torch.empty((Mb, Kb), dtype=torch.bfloat16, device=dev)
    rec("gemm_blockwise_dgrad", time_kernel(lambda: fp8.gemm(q_dy, q_wt, "dgrad", out=dX), flush, reps),
        flops=2.0 * Mb * Nb * Kb, workload="dX = dY W, 8192x4096(N)x4096")
    dW = torch.empty((Nb, Kb), dtype=torch.bfloat16, device=dev)
    rec("gemm_blockwise_wgrad", time_kernel(lambda: fp8.gemm(q_dyt, q_xt, "wgrad", out=dW), flush, reps),
        flops=2.0 * Mb * Nb * Kb, workload="dW = dY^T X, 4096x8192(M)x4096")
    # the same backward in MXFP8: 32x1 blocks for the transposed operands
    m_dy = fp8.quantize_mx(dY)
    m_wt = fp8.quantize_mx(Wb, transposed=True)
    m_dyt = fp8.quantize_mx(dY, transposed=True)
    m_xt = fp8.quantize_mx(Xb, transposed=True)
    rec("quant_mx_32x1_T", time_kernel(lambda: fp8.quantize_mx(Xb, out=m_xt, transposed=True), flush, reps),
        bytes_=Mb * Kb * (3 + 1 / 32), workload="X 8192x4096 -> X^T, 32x1 blocks")
    rec("gemm_mx_dgrad", time_kernel(lambda: fp8.gemm(m_dy, m_wt, "dgrad", out=dX), flush, reps),
        flops=2.0 * Mb * Nb * Kb, workload="MXFP8 dX = dY W, 8192x4096(N)x4096")
    rec("gemm_mx_wgrad", time_kernel(lambda: fp8.gemm(m_dyt, m_xt, "wgrad", out=dW), flush, reps),
        flops=2.0 * Mb * Nb * Kb, workload="MXFP8 dW = dY^T X, 4096x8192(M)x4096")
    del dY, Wb, Xb, q_dy, q_w, q_wt, q_dyt, q_xt, dX, dW, m_dy, m_wt, m_dyt, m_xt
    torch.cuda.empty_cache()

    # MXFP8 forward
    wl = synth.mx()
    Xm, Wm = wl.tensors["X"].to(dev), wl.tensors["W"].to(dev)
    qxm, qwm = fp8.quantize_mx(Xm), fp8.quantize_mx(Wm)
    rec("quant_mx_1x32", time_kernel(lambda: fp8.quantize_mx(Wm, out=qwm), flush, reps),
        bytes_=4096 * 4096 * (3 + 1 / 32), workload="W 4096x4096")
    Ym = torch.empty((2048, 4096), dtype=torch.bfloat16, device=dev)
    rec("gemm_mx_fwd", time_kernel(lambda: fp8.gemm(qxm, qwm, out=Ym), flush, reps),
        flops=2.0 * 2048 * 4096 * 4096, workload="2048x4096x4096")
    del Xm, Wm, qxm, qwm, Ym
    torch.cuda.empty_cache()

    # MoE
    wl = synth.moe()
    Xe, We = wl.tensors["X"].to(dev), wl.tensors["W"]
    G, Ne, Ke = We.shape
    We = We.reshape(G * Ne, Ke).to(dev)
    gather, offsets = wl.tensors["gather"].to(dev), wl.tensors["offsets"].to(dev)
    qxe = fp8.quantize_mx(Xe)
    qa = fp8.permute_rows_mx(qxe, gather, offsets)
    qwe = fp8.quantize_mx(We)
    rows = gather.numel()
    rec("quant_mx_1x32_moe_x", time_kernel(lambda: fp8.quantize_mx(Xe, out=qxe), flush, reps),
        bytes_=Xe.numel() * (3 + 1 / 32), workload=f"MoE tokens X {Xe.shape[0]}x{Ke}")
    rec("quant_mx_1x32_moe_w", time_kernel(lambda: fp8.quantize_mx(We, out=qwe), flush, reps),
        bytes_=We.numel() * (3 + 1 / 32), workload=f"64 expert weights {G}x{Ne}x{Ke}")
    rec("permute_rows_mx", time_kernel(lambda: fp8.permute_rows_mx(qxe, gather, offsets, out=qa), flush, reps),
        bytes_=2 * rows * Ke + 4 * rows + 2 * rows * Ke / 32, workload=f"{rows} rows x {Ke}")
    dsti = wl.tensors["dst_index"].to(dev)
    qd = fp8.dispatch_quantize_mx(Xe, dsti, offsets, rows)
    rec("dispatch_quantize_mx", time_kernel(lambda: fp8.dispatch_quantize_mx(Xe, dsti, offsets, rows, out=qd), flush,
                                            reps),
        bytes_=Xe.numel() * 2 + rows * Ke * (1 + 1 / 32) + 4 * rows,
        workload=f"MoE dispatch of X {Xe.shape[0]}x{Ke} to {rows} rows (top-8) fused with the MX quantization")
    del qd
    Ye = torch.empty((rows, Ne), dtype=torch.bfloat16, device=dev)
    rec("gemm_mx_grouped", time_kernel(lambda: fp8.grouped_gemm(qa, qwe, offsets, Ne, out=Ye), flush, reps),
        flops=2.0 * rows * Ne * Ke, workload=f"64 experts, {rows} rows, {Ne}x{Ke}")
    del Xe, We, qxe, qa, qwe, Ye
    torch.cuda.empty_cache()
    return out


def _case_gemm(kind):
    def setup(fp8, synth, dev):
        if kind in ("fwd", "fwd_fused", "pow2", "pow2_fused"):
            wl = synth.mlp()
            X, W = wl.tensors["X"].to(dev), wl.tensors["W"].to(dev)
            p2 = kind.startswith("pow2")
            qx, qw = fp8.quantize_group(X, "K", pow2=p2), fp8.quantize_block(W, pow2=p2)
            Y, qy = fp8.gemm(qx, qw, quantize_output=True)
            if kind in ("fwd", "pow2"):
                return lambda: fp8.gemm(qx, qw, out=Y), 2.0 * M * N * K
            return lambda: fp8.gemm(qx, qw, quantize_output=True, out=Y, out_q=qy), 2.0 * M * N * K
        if kind in ("dgrad", "wgrad", "mx_dgrad", "mx_wgrad"):
            wl = synth.backward()
            dY, W, X = (wl.tensors[k].to(dev) for k in ("dY", "W", "X"))
            if kind == "mx_dgrad":
                a, b = fp8.quantize_mx(dY), fp8.quantize_mx(W, transposed=True)
            elif kind == "mx_wgrad":
                a, b = fp8.quantize_mx(dY, transposed=True), fp8.quantize_mx(X, transposed=True)
            elif kind == "dgrad":
                a, (_, b) = fp8.quantize_group(dY, "K"), fp8.quantize_block(W, True)
            else:
                a, b = fp8.quantize_group(dY, "M"), fp8.quantize_group(X, "M")
            D = torch.empty((a.rows, b.rows), dtype=torch.bfloat16, device=dev)
            return lambda: fp8.gemm(a, b, kind.replace("mx_", ""), out=D), 2.0 * 8192 * 4096 * 4096
        if kind == "mx":
            wl = synth.mx()
            a, b = fp8.quantize_mx(wl.tensors["X"].to(dev)), fp8.quantize_mx(wl.tensors["W"].to(dev))
            D = torch.empty((a.rows, b.rows), dtype=torch.bfloat16, device=dev)
            return lambda: fp8.gemm(a, b, out=D), 2.0 * 2048 * 4096 * 4096
        wl = synth.moe()
        We = wl.tensors["W"]
        G, Ne, Ke = We.shape
        off = wl.tensors["offsets"].to(dev)
        qa = fp8.permute_rows_mx(fp8.quantize_mx(wl.tensors["X"].to(dev)), wl.tensors["gather"].to(dev), off)
        qw = fp8.quantize_mx(We.reshape(G * Ne, Ke).to(dev))
        D = torch.empty((qa.rows, Ne), dtype=torch.bfloat16, device=dev)
        return lambda: fp8.grouped_gemm(qa, qw, off, Ne, out=D), 2.0 * qa.rows * Ne * Ke
    return setup


def _case_quant(kind):
    def setup(fp8, synth, dev):
        if kind == "group_k":
            X = synth.mlp().tensors["X"].to(dev)
            q = fp8.quantize_group(X, "K")
            return lambda: fp8.quantize_group(X, "K", out=q), None
        if kind == "block":
            W = synth.mlp().tensors["W"].to(dev)
            q = fp8.quantize_block(W)
            return lambda: fp8.quantize_block(W, out=q), None
        if kind == "requant":
            X = synth.backward().tensors["X"].to(dev)
            q1 = fp8.quantize_group(X, "K")
            qr = fp8.requantize_transposed(q1)
            return lambda: fp8.requantize_transposed(q1, out=qr), None
        if kind == "block_t":
            W = synth.backward().tensors["W"].to(dev)
            q, qt = fp8.quantize_block(W, True)
            return lambda: fp8.quantize_block(W, True, out=q, out_t=qt), None
        if kind == "group_m":
            X = synth.backward().tensors["X"].to(dev)
            q = fp8.quantize_group(X, "M")
            return lambda: fp8.quantize_group(X, "M", out=q), None
        if kind == "permute_quant":
            wl = synth.moe()
            Xe = wl.tensors["X"].to(dev)
            dsti, offsets = wl.tensors["dst_index"].to(dev), wl.tensors["offsets"].to(dev)
            rows = wl.tensors["gather"].numel()
            qd = fp8.dispatch_quantize_mx(Xe, dsti, offsets, rows)
            return lambda: fp8.dispatch_quantize_mx(Xe, dsti, offsets, rows, out=qd), None
        if kind == "permute":
            wl = synth.moe()
            Xe = wl.tensors["X"].to(dev)
            gather, offsets = wl.tensors["gather"].to(dev), wl.tensors["offsets"].to(dev)
            qxe = fp8.quantize_mx(Xe)
            qa = fp8.permute_rows_mx(qxe, gather, offsets)
            return lambda: fp8.permute_rows_mx(qxe, gather, offsets, out=qa), None
        if kind in ("sync_split", "sync_noalloc"):
            # the same W as 48 entries of 256 rows: 96 segments, more than one
            # copy table holds, so the install takes the two-kernel path
            # (verify, then copy); or the whole W through the allocation-free
            # entry point (verify, then a table-driven copy)
            W = synth.mlp().tensors["W"].to(dev)
            qw = fp8.quantize_block(W)
            parts = 48 if kind == "sync_split" else 1
            rows = qw.rows // parts
            ents = [fp8.SyncEntry(i + 1, fp8.QTensor(qw.codes[i * rows:(i + 1) * rows],
                                                     qw.scales[i * rows // 128:(i + 1) * rows // 128], rows, qw.cols,
                                                     qw.recipe, qw.layout)) for i in range(parts)]
            payload = fp8.sync_pack(ents)
            dst = [fp8.SyncEntry(e.tag, fp8.QTensor(torch.empty_like(e.tensor.codes), torch.empty_like(e.tensor.scales),
                                                   e.tensor.rows, e.tensor.cols, e.tensor.recipe, e.tensor.layout))
                   for e in ents]
            if kind == "sync_noalloc":
                return lambda: fp8.sync_install_noalloc(payload, dst), None
            return lambda: fp8.sync_install(payload, dst, check=False), None
        if kind in ("sync_pack", "sync_install"):
            W = synth.mlp().tensors["W"].to(dev)
            qw = fp8.quantize_block(W)
            payload = fp8.sync_pack([fp8.SyncEntry(1, qw)])
            if kind == "sync_pack":
                return lambda: fp8.sync_pack([fp8.SyncEntry(1, qw)], payload=payload), None
            dst = fp8.QTensor(torch.empty_like(qw.codes), torch.empty_like(qw.scales), qw.rows, qw.cols, qw.recipe,
                              qw.layout)
            return lambda: fp8.sync_install(payload, [fp8.SyncEntry(1, dst)], check=False), None
        if kind in ("rmsnorm", "swiglu"):
            if kind == "rmsnorm":
                X = synth.mlp().tensors["X"].to(dev)
                gam = torch.ones((X.shape[1],), dtype=torch.bfloat16, device=dev)
                q = fp8.rmsnorm_quantize(X, gam)
                return lambda: fp8.rmsnorm_quantize(X, gam, out=q), None
            GU = torch.empty((M, N), dtype=torch.bfloat16, device=dev).normal_(0.0, 1.5)
            q = fp8.swiglu_quantize(GU)
            return lambda: fp8.swiglu_quantize(GU, out=q), None
        if kind in ("param", "param_update"):
            wl = synth.fp8_param()
            Wm, dW = wl.tensors["W"].to(dev), wl.tensors["dW"].to(dev)
            q, qt = fp8.param_requantize(Wm, transposed=True)
            if kind == "param":
                return lambda: fp8.param_requantize(Wm, out=q), None
            return lambda: fp8.param_requantize(Wm, dW, True, out=q, out_t=qt), None
        if kind == "mx_t":
            X = synth.backward().tensors["X"].to(dev)
            q = fp8.quantize_mx(X, transposed=True)
            return lambda: fp8.quantize_mx(X, out=q, transposed=True), None
        W = synth.mx().tensors["W"].to(dev)
        q = fp8.quantize_mx(W)
        return lambda: fp8.quantize_mx(W, out=q), None
    return setup


KERNEL_CASES = {
    "gemm_blockwise_fwd": _case_gemm("fwd"), "gemm_blockwise_fwd_fused": _case_gemm("fwd_fused"),
    "gemm_blockwise_dgrad": _case_gemm("dgrad"), "gemm_blockwise_wgrad": _case_gemm("wgrad"),
    "gemm_mx_fwd": _case_gemm("mx"), "gemm_mx_grouped": _case_gemm("grouped"),
    "gemm_blockwise_pow2_fwd": _case_gemm("pow2"), "gemm_blockwise_pow2_fwd_fused": _case_gemm("pow2_fused"),
    "quant_group_1x128": _case_quant("group_k"), "quant_block_128x128": _case_quant("block"),
    "quant_group_128x1_T": _case_quant("group_m"), "quant_mx_1x32": _case_quant("mx"),
    "gemm_mx_dgrad": _case_gemm("mx_dgrad"), "gemm_mx_wgrad": _case_gemm("mx_wgrad"),
    "quant_mx_32x1_T": _case_quant("mx_t"), "requant_1x128_to_128x1_T": _case_quant("requant"), "quant_block_128x128_with_T": _case_quant("block_t"),
    "param_requant": _case_quant("param"), "param_update_requant_with_T": _case_quant("param_update"),
    "rmsnorm_quant": _case_quant("rmsnorm"), "swiglu_quant": _case_quant("swiglu"),
    "sync_pack": _case_quant("sync_pack"), "sync_install": _case_quant("sync_install"), "permute_rows_mx": _case_quant("permute"),
    "sync_install_split": _case_quant("sync_split"), "sync_install_noalloc": _case_quant("sync_noalloc"),
    "dispatch_quantize_mx": _case_quant("permute_quant"),
}


def run_fp8_param_drift(args, dev):
    """Figure 12 of the SkyRL page on synthetic weights: the cumulative FP8
    displacement over many lr = 1e-6 sign updates, and the single-step
    cosine against the update size, for fp32 and power-of-two scales."""
    import param_drift
    from block_scaled_fp8_e4m3_gb300 import synth
    n = args.drift_size
    w0 = synth.fp32_master((n, n), seed=80).to(dev)
    steps = args.drift_steps
    marks = tuple(sorted({steps // 10, steps // 2, steps}))
    out = {"experiment": "fp8_param_drift", "config": {
        "master": f"{n}x{n} fp32 ~N(0,0.02), seed 80", "update": "1e-6 * (+-1), fair signs, per element and step",
        "steps": steps, "displacement": "projection <D,M>/<M,M> (also L1, L2 ratios)"}}
    for p2 in (False, True):
        key = "pow2" if p2 else "fp32"
        out[f"cumulative_{key}"] = {str(t): v for t, v in param_drift.cumulative_displacement(
            w0, steps, 1e-6, p2, seed=81, checkpoints=marks).items()}
        out[f"single_step_{key}"] = param_drift.single_step_cosine(
            w0, [1e-7, 3e-7, 1e-6, 3e-6, 1e-5, 1e-4, 1e-3, 1e-2], p2, seed=82)
    print(json.dumps(out), flush=True)


def run_single_kernel(args, fp8, synth, dev):
    fn, flops = KERNEL_CASES[args.kernel](fp8, synth, dev)
    flush = Flusher(dev)
    ms = time_kernel(fn, flush, args.steps, warmup=args.warmup)
    d = {"kernel": args.kernel, "ms": ms, "steps": args.steps, "warmup": args.warmup}
    if flops:
        d["TFLOP/s"] = flops / (ms * 1e-3) / 1e12
    print(json.dumps(d), flush=True)


def cpu_baseline_sample(X, W, rows_x, rows_w):
    """The CPU oracle, as it stands, on rows_x rows of X and rows_w rows of W
    (full K): quantize both, fp64 GEMM reference of that block, pack and
    install the W slice.  Returns (seconds, flops, sample description)."""
    import oracle
    from block_scaled_fp8_e4m3_gb300 import synth
    xs = synth.bf16_bits(X[:rows_x].contiguous())
    ws = synth.bf16_bits(W[:rows_w].contiguous())
    oracle.load()
    t0 = time.perf_counter()
    cx, sx = oracle.quant_group_1x128(xs)
    cw, sw = oracle.quant_block_128x128(ws)
    oracle.gemm_ref(oracle.dequant_group(cx, sx), oracle.dequant_block(cw, sw))
    spec = [dict(tag=1, kind=oracle.KIND_FP8, recipe=oracle.RECIPE_BLOCKWISE, rows=rows_w, cols=K,
                 layout=oracle.LAYOUT_BLOCK_128x128, data=cw, scales=sw)]
    payload = oracle.sync_pack(spec)
    dst = [dict(spec[0], data=np.zeros_like(cw), scales=np.zeros_like(sw))]
    assert oracle.sync_install(payload, dst) == 0
    dt = time.perf_counter() - t0
    return dt, 2.0 * rows_x * rows_w * K, (f"oracle on X[:{rows_x}] and W[:{rows_w}] (K=4096): quantize both, "
                                           f"fp64 GEMM {rows_x}x{K}x{rows_w}, pack+install the W slice")


def oracle_kernel_timings(X, W, rows=1024, gemm_shape=(512, 1024)):
    """Each of the oracle's quantizers (and the fused producers, the
    fp8_param re-quantization and the sync pack + install), as it stands, on
    a bounded slice of the dense-MLP inputs (rows x 4096), timed once on one
    thread and once on all of this host's cores; the fp64 GEMM reference
    (gemm_shape[0] x 4096 x gemm_shape[1]) on all cores.  Bytes are each
    kernel's algorithmic bytes for that slice, as on the GPU."""
    import oracle
    from block_scaled_fp8_e4m3_gb300 import synth
    oracle.load()
    ncores = cores()
    xs = synth.bf16_bits(X[:rows].contiguous())
    ws = synth.bf16_bits(W[:rows].contiguous())
    wf = np.ascontiguousarray(W[:rows].float().numpy())
    gu = synth.bf16_bits(torch.cat([X[:rows], X[rows:2 * rows]], dim=1).contiguous())
    gam = np.full((K,), 0x3F80, np.uint16)  # bf16 1.0
    cx, sx = oracle.quant_group_1x128(xs)
    cw, sw = oracle.quant_block_128x128(ws)
    spec = [dict(tag=1, kind=oracle.KIND_FP8, recipe=oracle.RECIPE_BLOCKWISE, rows=rows, cols=K,
                 layout=oracle.LAYOUT_BLOCK_128x128, data=cw, scales=sw)]
    dst = [dict(spec[0], data=np.zeros_like(cw), scales=np.zeros_like(sw))]
    payload_bytes = oracle.sync_payload_size(spec)

    def sync_round_trip():
        pay = oracle.sync_pack(spec)
        assert oracle.sync_install(pay, dst) == 0

    n = rows * K
    cases = [
        ("quant_group_1x128", lambda: oracle.quant_group_1x128(xs), n * (3 + 4 / 128)),
        ("quant_group_128x1_T", lambda: oracle.quant_group_128x1_T(xs), n * (3 + 4 / 128)),
        ("quant_block_128x128_with_T", lambda: oracle.quant_block_128x128(ws, transposed=True), n * (4 + 8 / 16384)),
        ("quant_mx_1x32", lambda: oracle.quant_mx_1x32(ws), n * (3 + 1 / 32)),
        ("quant_mx_32x1_T", lambda: oracle.quant_mx_32x1_T(xs), n * (3 + 1 / 32)),
        ("requant_1x128_to_128x1_T", lambda: oracle.requant_1x128_to_128x1_T(cx, sx), n * (2 + 8 / 128)),
        ("param_requant_fp32_master", lambda: oracle.quant_block_128x128_f32(wf), n * (5 + 4 / 16384)),
        ("rmsnorm_quant", lambda: oracle.quant_group_1x128(oracle.rmsnorm(xs, gam, 1e-6)[0]), n * (3 + 4 / 128)),
        ("swiglu_quant", lambda: oracle.quant_group_1x128(oracle.swiglu(gu)), n * (5 + 4 / 128)),
        ("sync_pack_install", sync_round_trip, 4.0 * payload_bytes),
    ]
    out = {"cores": ncores, "slice": f"{rows} rows x {K} of X / W (dense-MLP workload)"}
    for name, fn, nbytes in cases:
        rec = {}
        for label, th in (("threads_1", 1), ("threads_all", ncores)):
            oracle.set_threads(th)
            t0 = time.perf_counter()
            fn()
            dt = time.perf_counter() - t0
            rec[label] = {"s": round(dt, 4), "GB/s": round(nbytes / dt / 1e9, 3)}
        out[name] = rec
    oracle.set_threads(ncores)
    gm, gn = gemm_shape
    a = oracle.dequant_group(cx[:gm], np.ascontiguousarray(sx[:, :gm]))
    b = oracle.dequant_block(cw[:gn], np.ascontiguousarray(sw[:gn // 128]))
    t0 = time.perf_counter()
    oracle.gemm_ref(a, b)
    dt = time.perf_counter() - t0
    out["gemm_ref_fp64"] = {"shape": f"{gm}x{K}x{gn}", "threads_all": {"s": round(dt, 4),
                            "TFLOP/s": round(2.0 * gm * gn * K / dt / 1e12, 5)}}
    return out


def cores():
    try:
        return len(os.sched_getaffinity(0))
    except Exception:
        return os.cpu_count() or 1


def run_reference(args):
    """CPU oracle arm: each step is a bounded sample of the workload."""
    from block_scaled_fp8_e4m3_gb300 import synth
    wl = synth.mlp()
    X, W = wl.tensors["X"], wl.tensors["W"]
    rx, rw = 128, 256
    for _ in range(args.warmup):
        cpu_baseline_sample(X, W, rx, rw)
    tot, flops, desc = 0.0, 0.0, ""
    for _ in range(args.steps):
        dt, fl, desc = cpu_baseline_sample(X, W, rx, rw)
        tot += dt
        flops += fl
    value = flops / tot / 1e12
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * tot / args.steps,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": WORKLOAD, "sample_per_step": desc, "l2": "n/a (CPU)"},
            "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": cores(), "kind": "oracle", "sample": desc},
            "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=100)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--no-breakdown", action="store_true", help="skip the per-kernel table")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--kernel-reps", type=int, default=40)
    ap.add_argument("--kernel", default=None, choices=sorted(KERNEL_CASES),
                    help="run only this kernel on its workload (for profilers); prints its timing")
    ap.add_argument("--no-oracle-kernels", action="store_true",
                    help="skip the per-kernel oracle timings of the cpu_baseline leg")
    ap.add_argument("--experiment", default=None, choices=["fp8_param_drift"],
                    help="run a measurement from the pages instead of the benchmark; prints one JSON line")
    ap.add_argument("--drift-size", type=int, default=4096)
    ap.add_argument("--drift-steps", type=int, default=2000)
    args = ap.parse_args()
    args.warmup = max(args.warmup, 3)

    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))

    if args.impl == "reference":
        if rank == 0:
            run_reference(args)
        return

    import block_scaled_fp8_e4m3_gb300 as fp8
    from block_scaled_fp8_e4m3_gb300 import _build, synth
    _build.build()
    fp8.library()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if args.kernel is not None:
        run_single_kernel(args, fp8, synth, dev)
        return
    if args.experiment == "fp8_param_drift":
        run_fp8_param_drift(args, dev)
        return
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=dev)
    pk = peaks()

    wl = synth.mlp()
    Xh, Wh = wl.tensors["X"], wl.tensors["W"]
    X, W = Xh.to(dev), Wh.to(dev)
    step, payload_bytes, keep = make_step(fp8, X, W, dev)
    flush = Flusher(dev)

    for _ in range(args.warmup):
        flush()
        step()
    torch.cuda.synchronize()

    phys = os.environ.get("CUDA_VISIBLE_DEVICES", str(local)).split(",")[local] if os.environ.get(
        "CUDA_VISIBLE_DEVICES") else str(local)
    sampler = ClockSampler(int(phys) if phys.isdigit() else local)
    time.sleep(0.2)
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    evs = []
    for _ in range(args.steps):
        flush()
        e = [torch.cuda.Event(enable_timing=True) for _ in range(6)]
        step(e)
        evs.append(e)
    torch.cuda.synchronize()
    if world > 1:
        torch.distributed.barrier()
    clocks = sampler.stop()

    per_kernel = np.zeros(5)
    total_ms = 0.0
    for e in evs:
        seg = [e[i].elapsed_time(e[i + 1]) for i in range(5)]
        per_kernel += seg
        total_ms += e[0].elapsed_time(e[5])
    per_kernel /= args.steps
    ms_step = max_over_ranks(total_ms / args.steps, world, dev)
    flops = 2.0 * M * N * K
    value = whole_job_tflops(flops, ms_step, world)

    # dominant kernel (the GEMM) against the FP8 dense peak
    fp8_peak = 2.0 * pk["bf16_tflops"]
    gemm_tf = flops / (per_kernel[2] * 1e-3) / 1e12
    roofline = {"bound": "tensor", "kernel": "k_gemm_blockwise (fwd, fused 1x128 quant of Y)",
                "achieved": round(gemm_tf, 1), "peak": round(fp8_peak, 1), "unit": "TFLOP/s",
                "frac": round(gemm_tf / fp8_peak, 4),
                "peak_basis": f"2 x {pk['source']} bf16 burst {pk['bf16_tflops']} TFLOP/s (FP8:BF16 = 2:1)",
                "traffic": gemm_traffic()}
    qx_gbs = M * K * (3 + 4 / 128) / (per_kernel[0] * 1e-3) / 1e9
    qw_gbs = N * K * (3 + 4 / 16384) / (per_kernel[1] * 1e-3) / 1e9
    step_kernels = {
        "quant_group_1x128_X": {"ms": round(per_kernel[0], 5), "GB/s": round(qx_gbs, 1),
                                "frac_hbm": round(qx_gbs / pk["hbm_gbs"], 4)},
        "quant_block_128x128_W": {"ms": round(per_kernel[1], 5), "GB/s": round(qw_gbs, 1),
                                  "frac_hbm": round(qw_gbs / pk["hbm_gbs"], 4)},
        "gemm_blockwise_fwd_fused_quant": {"ms": round(per_kernel[2], 5), "TFLOP/s": round(gemm_tf, 1),
                                           "frac_fp8_peak": round(gemm_tf / fp8_peak, 4)},
        "sync_pack_W": {"ms": round(per_kernel[3], 5),
                        "GB/s": round(2 * payload_bytes / (per_kernel[3] * 1e-3) / 1e9, 1)},
        "sync_install_W": {"ms": round(per_kernel[4], 5),
                           "GB/s": round(2 * payload_bytes / (per_kernel[4] * 1e-3) / 1e9, 1)},
    }

    # end to end through the public API with host buffers: every step copies
    # its inputs X and W in from pinned host memory and its bf16 result Y out.
    # The loop is the one a user would write: two device buffer sets, the
    # inputs of step i+1 and the output of step i-1 moving on their own
    # streams while step i's kernels run.
    Xp, Wp = Xh.pin_memory(), Wh.pin_memory()
    Yp = torch.empty((M, N), dtype=torch.bfloat16).pin_memory()
    X2, W2 = torch.empty_like(X), torch.empty_like(W)
    step2, _, keep2 = make_step(fp8, X2, W2, dev)
    sets = [(X, W, step), (X2, W2, step2)]
    s_in, s_comp, s_out = torch.cuda.Stream(), torch.cuda.Stream(), torch.cuda.Stream()
    e2e_steps = min(args.steps, 20)
    ev = lambda: torch.cuda.Event(enable_timing=False)

    def run_e2e(n):
        """n pipelined steps; returns the device time from the first input
        copy to the last output copy (ms)."""
        in_done = [ev() for _ in range(n)]
        comp_done = [ev() for _ in range(n)]
        out_done = [ev() for _ in range(n)]
        torch.cuda.synchronize()
        t0 = torch.cuda.Event(enable_timing=True)
        t1 = torch.cuda.Event(enable_timing=True)
        t0.record(s_in)
        for i in range(n):
            Xb, Wb, stepb = sets[i % 2]
            with torch.cuda.stream(s_in):
                if i >= 2:
                    s_in.wait_event(comp_done[i - 2])      # step i-2 has finished reading this set
                Xb.copy_(Xp, non_blocking=True)
                Wb.copy_(Wp, non_blocking=True)
                in_done[i].record(s_in)
            with torch.cuda.stream(s_comp):
                s_comp.wait_event(in_done[i])
                if i >= 2:
                    s_comp.wait_event(out_done[i - 2])     # this set's Y has been copied out
                Y = stepb()
                comp_done[i].record(s_comp)
            with torch.cuda.stream(s_out):
                s_out.wait_event(comp_done[i])
                Yp.copy_(Y, non_blocking=True)
                out_done[i].record(s_out)
        s_out.wait_event(out_done[n - 1])
        t1.record(s_out)
        torch.cuda.synchronize()
        return t0.elapsed_time(t1)

    run_e2e(max(args.warmup, 3))                           # untimed: both buffer sets in use once
    e2e_ms = max_over_ranks(run_e2e(e2e_steps) / e2e_steps, world, dev)
    e2e = {"value": whole_job_tflops(flops, e2e_ms, world), "unit": "TFLOP/s",
           "h2d_bytes_per_step": int(Xh.numel() * 2 + Wh.numel() * 2), "d2h_bytes_per_step": int(M * N * 2),
           "ms_per_step": e2e_ms, "steps": e2e_steps,
           "schedule": "double-buffered: copies in (step i+1) and out (step i-1) on their own streams"}

    # the host link alone, for context: the same copies without the kernels
    def copies_ms(fn, reps=10):
        fn()
        torch.cuda.synchronize()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record()
        for _ in range(reps):
            fn()
        b.record()
        torch.cuda.synchronize()
        return a.elapsed_time(b) / reps

    def h2d():
        X.copy_(Xp, non_blocking=True)
        W.copy_(Wp, non_blocking=True)

    def both():
        cur = torch.cuda.current_stream()
        s_in.wait_stream(cur)
        s_out.wait_stream(cur)
        with torch.cuda.stream(s_in):
            h2d()
        with torch.cuda.stream(s_out):
            Yp.copy_(keep[2], non_blocking=True)
        cur.wait_stream(s_in)
        cur.wait_stream(s_out)

    e2e["host_link"] = {"h2d_ms": round(copies_ms(h2d), 4),
                        "d2h_ms": round(copies_ms(lambda: Yp.copy_(keep[2], non_blocking=True)), 4),
                        "both_concurrent_ms": round(copies_ms(both), 4)}
    del keep2, X2, W2, sets

    kernels = None
    if not args.no_breakdown and rank == 0:
        del keep
        torch.cuda.empty_cache()
        kernels = breakdown(fp8, synth, dev, flush, pk, args.kernel_reps)

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        dt, fl, desc = cpu_baseline_sample(Xh, Wh, 4096, 6144)
        cpu = {"value": fl / dt / 1e12, "unit": "TFLOP/s", "cores": cores(), "kind": "oracle", "sample": desc,
               "seconds": round(dt, 2)}
        if not args.no_oracle_kernels:
            cpu["per_kernel"] = oracle_kernel_timings(Xh, Wh)

    if rank == 0:
        line = {"metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": world, "steps": args.steps,
                "warmup": args.warmup, "ms_per_step": ms_step, "higher_is_better": True, "scaling": "weak",
                "vs_baseline": None, "dtype": "e4m3 (fp32 accumulate, bf16 out)", "data": "synthetic",
                "config": {"workload": WORKLOAD, "M": M, "K": K, "N": N, "seed": 2,
                           "step": "quant X 1x128, quant W 128x128, GEMM+fused quant of Y, sync pack W, install W",
                           "l2": "flushed between steps (256 MB write, then 256 MB read)",
                           "parallelism": f"replicas x{world}", "input_sha256": wl.sha256()},
                "roofline": roofline, "step_kernels": step_kernels, "cpu_baseline": cpu, "e2e": e2e,
                "gpu_launches": KERNELS_PER_STEP * args.steps, "clocks": clocks, "peaks": pk,
                "kernels": kernels}
        print(json.dumps(line), flush=True)
    if world > 1:
        torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()
