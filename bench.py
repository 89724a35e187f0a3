#!/usr/bin/env python3
"""Throughput of the tensor-parallel MLP forward + backward on GB300.

One step = tp_mlp_fwd + tp_mlp_bwd of the GPT-style workload
(X [S=2048, B=4, H=4096] bf16, W1 [16384, 4096] column-split over T=8,
W2 [4096, 16384] row-split, GeLU-tanh, bias, residual) on seeded synthetic
inputs.  The metric is algorithmic TFLOP/s (12*M*H*F per step).

  python bench.py [--gpus N] [--steps K] [--warmup W] [--workload gpt]
  python bench.py --impl reference ...   # the fp64 CPU oracle on host cores
  python bench.py --block layer ...      # the TransformerLayer MLP sub-block:
                                         # LayerNorm -> MLP -> dropout + residual

Under torchrun (N > 1) every rank runs an independent replica of the step on
its own GPU (the library's shards all live on one GPU); the reported value is
the total over ranks divided by the slowest rank's time.
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

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import synth  # noqa: E402

METRIC = "TP-sharded MLP fwd+bwd TFLOP/s on 1 GB300; % of dense BF16 tensor peak"
UNIT = "TFLOP/s"
L2_BYTES = 129 * 1024 * 1024


# The measured peaks give cuBLAS bf16 twice: as a burst (best of 10 short
# GEMMs) and sustained (back to back for 4 s, where the power cap lowers the
# clock).  A timed region shorter than that runs mostly before the cap bites
# and is compared against the burst figure; a region of 4 s or more against
# the sustained one.
SUSTAINED_REGION_S = 4.0


def pick_peak(peaks, region_s, dtype):
    """(peak TFLOP/s, description) for a tensor-bound region of region_s
    seconds; FP8 takes twice the bf16 figure (the 4.5 : 2.25 PFLOP/s nominal
    dense ratio)."""
    sustained = region_s >= SUSTAINED_REGION_S
    peak = peaks["bf16_tflops_sustained"] if sustained else peaks["bf16_tflops"]
    kind = (f"bf16 {'sustained' if sustained else 'burst'} ({peaks['source']}): timed region "
            f"{region_s:.2f} s {'>=' if sustained else '<'} {SUSTAINED_REGION_S:.0f} s")
    if dtype == "fp8":
        peak, kind = 2.0 * peak, "fp8 = 2 x " + kind + " x nominal fp8:bf16 ratio"
    return peak, kind


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            p = json.load(f)
        return {"bf16_tflops": float(p["bf16_tflops"]), "bf16_tflops_sustained": float(p["bf16_tflops_sustained"]),
                "hbm_gbs": float(p["hbm_gbs"]), "sm_max_mhz": float(p.get("sm_max_mhz", 2070.0)),
                "source": "measured"}
    except Exception:
        return {"bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0, "hbm_gbs": 6800.0, "sm_max_mhz": 2070.0,
                "source": "fallback"}


def fp32_alu_peak(sms, peaks):
    """(TFLOP/s, description) of the fp32 FFMA rate the fp32 engine is bound
    by: SMs x 128 FP32 lanes x 2 FLOP per FMA x the maximum SM clock."""
    mhz = peaks["sm_max_mhz"]
    return (sms * 128 * 2 * mhz * 1e6 / 1e12,
            f"fp32 FFMA, nominal: {sms} SMs x 128 lanes x 2 FLOP x {mhz:.0f} MHz (maximum SM clock)")


# ---------------------------------------------------------------------------
# distributed helpers (replicas only; no data-path collective)
# ---------------------------------------------------------------------------
def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def dist_init(ws, backend):
    if ws <= 1:
        return None
    import torch.distributed as dist
    os.environ.setdefault("MASTER_ADDR", "127.0.0.1")
    dist.init_process_group(backend=backend)
    return dist


def barrier(dist, device=None):
    if dist is not None:
        if device is not None:
            dist.barrier(device_ids=[device])
        else:
            dist.barrier()


def max_over_ranks(dist, value, device="cpu"):
    if dist is None:
        return value
    import torch
    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_throughput(world_size, flops_per_step, steps, ms_slowest):
    """Whole-job TFLOP/s: every rank runs `steps` steps of its own replica; the
    job takes as long as the slowest rank."""
    return world_size * flops_per_step * steps / (ms_slowest * 1e-3) / 1e12


# ---------------------------------------------------------------------------
# clocks
# ---------------------------------------------------------------------------
class ClockSampler:
    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.gpu = gpu_index
        self.proc = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "100"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None
        time.sleep(0.3)

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except Exception:
            self.proc.kill()
            out, _ = self.proc.communicate()
        sm, smax, reasons, power = [], [], set(), []
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in out.strip().splitlines():
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 7:
                continue
            try:
                sm.append(float(parts[0]))
                smax.append(float(parts[1]))
                power.append(float(parts[2]))
            except ValueError:
                continue
            for n, v in zip(names, parts[3:7]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(smax), "samples": len(sm),
                "power_w_max": max(power) if power else None, "reasons": sorted(reasons)}


# ---------------------------------------------------------------------------
# the GPU step
# ---------------------------------------------------------------------------
def kernel_flops(w):
    """Algorithmic FLOP of one launch of each GEMM kernel for workload w."""
    M, H, F, g = w.M, w.H, w.F, w.g
    if w.kind == "attn_proj":  # QKV column layer (F = 3H) and output row layer (F_o -> H)
        Fo = w.F_o
        return {"col_fwd": 2.0 * M * H * F, "wgrad_col": 2.0 * M * H * F, "col_dgrad": 2.0 * M * F * H,
                "row_fwd": 2.0 * M * Fo * H, "row_dgrad": 2.0 * M * H * Fo, "wgrad_row": 2.0 * M * H * Fo}
    return {"col_fwd": 2.0 * M * H * F * g, "row_fwd": 2.0 * M * F * H, "row_dgrad_act": 2.0 * M * H * F,
            "wgrad_row": 2.0 * M * H * F, "wgrad_col": 2.0 * M * H * F * g, "col_dgrad": 2.0 * M * F * g * H,
            "fused_mlp_fwd": 2.0 * M * H * F * g + 2.0 * M * F * H}


def gemm_bytes(w):
    """Algorithmic HBM bytes of one launch of each GEMM kernel (bf16 operands
    and activations, or fp32 ones for the fp32 workloads, fp32 weight
    gradients; every operand read once, every
    output written once) -- with kernel_flops, the arithmetic intensity that
    decides which roof bounds the kernel."""
    M, H, F, g = w.M, w.H, w.F, w.g
    e = 4 if w.dtype == "f32" else 2
    if w.kind == "attn_proj":
        Fo = w.F_o
        return {"col_fwd": e * (M * H + F * H + M * F), "wgrad_col": e * (M * F + M * H) + 4 * F * H,
                "col_dgrad": e * (M * F + F * H + M * H), "row_fwd": e * (M * Fo + H * Fo + M * H),
                "row_dgrad": e * (M * H + H * Fo + M * Fo), "wgrad_row": e * (M * H + M * Fo) + 4 * H * Fo}
    res = M * H * e if w.residual else 0
    return {"col_fwd": e * (M * H + g * F * H + M * g * F + M * F),
            "row_fwd": e * (M * F + H * F + M * H) + res,
            "row_dgrad_act": e * (M * H + H * F + 2 * M * g * F),
            "wgrad_row": e * (M * H + M * F) + 4 * H * F,
            "wgrad_col": e * (M * g * F + M * H) + 4 * g * F * H,
            "col_dgrad": e * (M * g * F + g * F * H + M * H) + res,
            "fused_mlp_fwd": e * (M * H + g * F * H + H * F + M * g * F + M * F + M * H) + res}


def step_bytes(w):
    """Bytes of the device tensors one step reads or writes (operands,
    activations, outputs, fp32 weight gradients), each counted once."""
    M, H, F, g = w.M, w.H, w.F, w.g
    e = 4 if w.dtype == "f32" else 2
    if w.kind == "attn_proj":
        Fo = w.F_o
        return e * (4 * M * H + 2 * M * F + 2 * M * Fo + F * H + H * Fo) + 4 * (F * H + H * Fo)
    return e * (4 * M * H + M * g * F + M * F + (g + 1) * F * H) + 4 * (g + 1) * F * H


LAYER_DROPOUT_P = 0.1  # Megatron's default hidden dropout
LAYER_SEED = 0x5EED_0000_0001


def hbm_kernel_bytes(w):
    """Algorithmic HBM bytes of one launch of the sub-block's memory-bound
    kernels (each operand read or written once)."""
    M, H = w.M, w.H
    es = 4 if w.dtype == "f32" else 2
    return {"layernorm_fwd": 2 * M * H * es + 2 * H * es + 8 * M,
            "layernorm_bwd": 4 * M * H * es + H * es + 8 * M,
            "dropout_bwd": 2 * M * H * es}


def recorded_traffic(w, tile_mode, kernel):
    """DRAM bytes per launch of `kernel` from the committed ncu summary, or None
    when there is none for this workload and tiling or the kernel source has
    changed since it was captured."""
    import hashlib
    path = os.path.join(ROOT, "profiles", f"dram_traffic_{w.name}.json")
    try:
        with open(path) as f:
            rec = json.load(f)
        h = hashlib.sha256()
        for src in rec["kernel_sources"]:
            with open(os.path.join(ROOT, src), "rb") as f:
                h.update(f.read())
        digest = h.hexdigest()
    except (OSError, KeyError, ValueError):
        return None
    if digest != rec.get("sha256") or rec.get("tile_mode") not in (tile_mode, "pair" if tile_mode == "auto" else None):
        return None
    return rec.get("bytes_per_launch", {}).get(kernel)


def mlp_step(args, w, tp, torch, dev, stream):
    """The MLP (or sub-block) step on device-resident shards.  Returns
    step(k) -- one fwd+bwd on buffer set k -- and the two buffer sets, each
    (inputs uploaded per step, outputs read back per step)."""
    bf = torch.bfloat16
    T, M, H, F, g = w.T, w.M, w.H, w.F, w.g
    Fs = F // T
    layer = args.block == "layer"
    if layer:
        lay = tp.TPLayer(S=w.S, B=w.B, H=H, F=F, T=T, act=w.act, dtype=w.dtype, has_bias=w.has_bias,
                         seq_parallel=w.seq_parallel, dropout_p=LAYER_DROPOUT_P)
    else:
        lay = tp.TPMLP(S=w.S, B=w.B, H=H, F=F, T=T, act=w.act, dtype=w.dtype, has_bias=w.has_bias,
                       residual=w.residual, seq_parallel=w.seq_parallel, wgrad_accumulate=args.wgrad_accumulate)
    if w.dtype == "fp8" and not layer and args.fp8_history:
        lay.set_fp8_history(args.fp8_history)
    full = synth.mlp_tensors(w)
    td = torch.float32 if w.dtype == "f32" else bf

    def up(a):
        return torch.from_numpy(np.ascontiguousarray(a)).to(device=dev, dtype=td)

    # shards: W1 rows (gate/up stacked per shard for SwiGLU), W2 columns
    if w.act == "swiglu":
        W1 = [up(np.concatenate([full["W1"][i * Fs:(i + 1) * Fs], full["W1"][F + i * Fs:F + (i + 1) * Fs]]))
              for i in range(T)]
    else:
        W1 = [up(full["W1"][i * Fs:(i + 1) * Fs]) for i in range(T)]
    W2 = [up(full["W2"][:, i * Fs:(i + 1) * Fs]) for i in range(T)]
    if not w.has_bias:
        b1 = None
    elif w.act == "swiglu":
        b1 = [up(np.concatenate([full["b1"][i * Fs:(i + 1) * Fs], full["b1"][F + i * Fs:F + (i + 1) * Fs]]))
              for i in range(T)]
    else:
        b1 = [up(full["b1"][i * Fs:(i + 1) * Fs]) for i in range(T)]
    b2 = up(full["b2"]) if w.has_bias else None
    rows = lay.xrows
    X = [up(full["X"][j * rows:(j + 1) * rows]) for j in range(lay.nx)]
    dY = [up(full["dY"][j * rows:(j + 1) * rows]) for j in range(lay.nx)]
    Y = [torch.empty(rows, H, dtype=td, device=dev) for _ in range(lay.nx)]
    dX = [torch.empty(rows, H, dtype=td, device=dev) for _ in range(lay.nx)]
    pre = [torch.empty(M, g * Fs, dtype=td, device=dev) for _ in range(T)]
    A = [torch.empty(M, Fs, dtype=td, device=dev) for _ in range(T)]
    f32 = torch.float32
    dW1 = [torch.empty(g * Fs, H, dtype=f32, device=dev) for _ in range(T)]
    dW2 = [torch.empty(H, Fs, dtype=f32, device=dev) for _ in range(T)]
    db1 = [torch.empty(g * Fs, dtype=f32, device=dev) for _ in range(T)] if w.has_bias else None
    db2 = torch.empty(H, dtype=f32, device=dev) if w.has_bias else None
    wsp = tp.alloc_workspace(lay.workspace_bytes(), device=dev)
    # the end-to-end loop alternates two device buffer sets for the step's
    # inputs (X, dY) and activation results (Y, dX); the weight and bias
    # gradients stay on the device for the optimizer
    bufs = [(X, dY, Y, dX), ([torch.empty_like(x) for x in X], [torch.empty_like(d) for d in dY],
                             [torch.empty_like(y) for y in Y], [torch.empty_like(d) for d in dX])]
    if layer:
        lnp = synth.layer_tensors(1, H, w.dtype)
        gamma, beta = up(lnp["gamma"]), up(lnp["beta"])
        Xn = torch.empty(M, H, dtype=td, device=dev)
        mean = torch.empty(M, dtype=f32, device=dev)
        rstd = torch.empty(M, dtype=f32, device=dev)
        dgamma = torch.empty(H, dtype=f32, device=dev)
        dbeta = torch.empty(H, dtype=f32, device=dev)

        def step(k=0):
            X, dY, Y, dX = bufs[k]
            lay.fwd(X, gamma, beta, W1, b1, W2, b2, LAYER_SEED, Y, Xn, mean, rstd, pre, A, workspace=wsp,
                    stream=stream)
            lay.bwd(dY, X, gamma, Xn, mean, rstd, W1, W2, pre, A, LAYER_SEED, dX, dgamma, dbeta, dW1, db1, dW2,
                    db2, wsp, stream=stream)
    else:
        def step(k=0):
            X, dY, Y, dX = bufs[k]
            lay.fwd(X, W1, b1, W2, b2, Y, pre, A, stream=stream, workspace=wsp)
            lay.bwd(dY, X, W1, W2, pre, A, dX, dW1, db1, dW2, db2, wsp, stream=stream)
    return step, [(x + d, y + dx) for x, d, y, dx in bufs], lay


def attn_step(args, w, tp, torch, dev, stream):
    """The attention projections' step: the QKV ColumnParallelLinear
    (H -> F = 3H, no activation) and the output RowParallelLinear (F_o -> H),
    forward and backward through the single-layer entry points.  Returns
    step(k) and the two buffer sets (inputs X, Z, dYqkv, dYo; output Yo)."""
    bf, f32 = torch.bfloat16, torch.float32
    T, M, H, F, Fo = w.T, w.M, w.H, w.F, w.F_o
    Fs, Fos = F // T, Fo // T
    full = synth.attn_tensors(w)

    def up(a):
        return torch.from_numpy(np.ascontiguousarray(a)).to(device=dev, dtype=bf)

    colL = tp.Layout(S=w.S, B=w.B, H=H, F=F, T=T, act="none", dtype=w.dtype)
    rowL = tp.Layout(S=w.S, B=w.B, H=H, F=Fo, T=T, act="none", dtype=w.dtype)
    Wq = [up(full["Wqkv"][i * Fs:(i + 1) * Fs]) for i in range(T)]
    Wo = [up(full["Wo"][:, i * Fos:(i + 1) * Fos]) for i in range(T)]
    X = up(full["X"])
    Z = [up(full["Z"][:, i * Fos:(i + 1) * Fos]) for i in range(T)]
    dYq = [up(full["dYqkv"][:, i * Fs:(i + 1) * Fs]) for i in range(T)]
    dYo = up(full["dYo"])
    Yq = [torch.empty(M, Fs, dtype=bf, device=dev) for _ in range(T)]
    Yo = torch.empty(M, H, dtype=bf, device=dev)
    dX = torch.empty(M, H, dtype=bf, device=dev)
    dZ = [torch.empty(M, Fos, dtype=bf, device=dev) for _ in range(T)]
    dWq = [torch.empty(Fs, H, dtype=f32, device=dev) for _ in range(T)]
    dWo = [torch.empty(H, Fos, dtype=f32, device=dev) for _ in range(T)]
    wsc = tp.alloc_workspace(tp.linear_workspace_bytes(colL), device=dev)
    wsr = tp.alloc_workspace(tp.linear_workspace_bytes(rowL), device=dev)
    # inputs (X, Z, the two upstream gradients) and outputs per buffer set;
    # the e2e leg reads back the results at the block's boundary -- the output
    # projection and the input gradient dX, as for the MLP -- while the QKV
    # projection and dZ stay on the device for the attention core
    bufs = [(X, Z, dYq, dYo, (Yq, Yo, dX, dZ)),
            (torch.empty_like(X), [torch.empty_like(z) for z in Z], [torch.empty_like(d) for d in dYq],
             torch.empty_like(dYo), ([torch.empty_like(y) for y in Yq], torch.empty_like(Yo), torch.empty_like(dX),
                                     [torch.empty_like(d) for d in dZ]))]

    def step(k=0):
        X, Z, dYq, dYo, (Yq, Yo, dX, dZ) = bufs[k]
        # the forward's workspace goes, unchanged, to the backward (FP8: the
        # forward's quantised X and W; bf16: the row GEMM's tail-split scratch)
        tp.linear_col(colL, [X], Wq, None, Yq, stream=stream, workspace=wsc)
        tp.linear_row(rowL, Z, Wo, None, None, [Yo], stream=stream, workspace=wsr)
        tp.linear_col_bwd(colL, dYq, [X], Wq, [dX], dWq, None, workspace=wsc, stream=stream)
        tp.linear_row_bwd(rowL, [dYo], Z, Wo, dZ, dWo, None, workspace=wsr, stream=stream)
    return step, [([X] + Z + dYq + [dYo], [Yo, dX]) for X, Z, dYq, dYo, (Yq, Yo, dX, dZ) in bufs], None


def run_gpu(args, w, dist, rank, local, ws):
    import torch

    import tensor_transformer_mlp_shard_gb300 as tp
    from tensor_transformer_mlp_shard_gb300 import build
    build.build()
    torch.cuda.set_device(local)
    tp.set_tile_mode(args.tile_mode)
    tp.set_fused_fwd(args.fused)
    tp.set_tail_split(args.tail_split == "on")
    tp.set_k_order(args.k_order == "alternate")
    tp.set_launch_overlap(args.launch_overlap == "on")
    tp.set_band_rows(args.band_rows)
    dev = torch.device("cuda", local)
    layer = args.block == "layer"
    # all work on one non-default stream (a CUDA graph cannot capture the legacy stream)
    stream = torch.cuda.Stream(dev)
    torch.cuda.set_stream(stream)
    make = attn_step if w.kind == "attn_proj" else mlp_step
    step, e2e_sets, handle = make(args, w, tp, torch, dev, stream)

    def status():
        """Device status of the step's calls: the handle's word and the word
        of the calls without a handle."""
        s = tp.sync_status(stream)
        return s if s != 0 or handle is None else handle.sync_status(stream)

    # ---- device-resident timing --------------------------------------------
    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    if status() != 0:
        raise RuntimeError("device status not OK after warm-up")
    graph_launches = 0
    eager_step = step
    if args.graph:
        # one step per graph and input set (the e2e loop alternates two sets)
        graphs = []
        n_before = tp.launch_count()
        for k in range(2):
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=stream):
                eager_step(k)
            graphs.append(g)
        graph_launches = (tp.launch_count() - n_before) // 2

        def step(k=0):
            graphs[k].replay()
    # ---- per-kernel profile pass, before the timed region ------------------
    # Every launch bracketed by CUDA events on its stream: the per-kernel
    # table and the choice of the roofline kernel (the GEMM with the most
    # time).  An event pair costs the stream a few microseconds between two
    # kernels, so the timed region brackets only the roofline kernel's
    # launches.
    prof_steps = max(3, min(args.steps, 10))
    kf = kernel_flops(w)
    tp.prof_select(None)
    tp.prof_enable(True)
    tp.prof_collect()
    for _ in range(prof_steps):
        eager_step()
    kprof = tp.prof_collect(clocks=True)
    tp.prof_enable(False)
    gemm_ms = {k: v[1] for k, v in kprof.items() if k in kf and v[0] > 0}
    dom = max(gemm_ms, key=gemm_ms.get) if gemm_ms else None
    clocks = ClockSampler(local)
    clocks.start()
    tp.prof_select(dom)
    tp.prof_enable(True)
    tp.prof_collect()  # drop earlier records
    n0 = tp.launch_count()
    barrier(dist, local)
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(args.steps):
        step()
    e1.record(stream)
    torch.cuda.synchronize()
    barrier(dist, local)
    ms = e0.elapsed_time(e1)
    launches = tp.launch_count() - n0 if not args.graph else graph_launches * args.steps
    kclk = tp.prof_collect(clocks=True)
    tp.prof_enable(False)
    tp.prof_select(None)
    clk = clocks.stop()
    # the SM clock the GEMMs ran at (clock64 against %globaltimer in every CTA)
    cyc, ns = sum(v[2] for v in kclk.values()), sum(v[3] for v in kclk.values())
    clk["kernel_mhz"] = round(cyc / ns * 1e3, 1) if ns else None
    st = status()
    if st != 0:
        raise RuntimeError(f"device status {tp.status_str(st)} in timed region")
    ms_max = max_over_ranks(dist, ms, dev)
    flops_step = w.flops()
    value = job_throughput(ws, flops_step, args.steps, ms_max)

    # ---- end to end through the C ABI with host buffers ---------------------
    # Every step copies its inputs (X and dY; for the projections X, Z and the
    # two upstream gradients) from pinned host memory and its activation
    # results (Y and dX; for the projections the output projection and dX) back.
    # The copies run on a second stream into two alternating device buffer
    # sets, so that step i's compute overlaps step i+1's inputs and step i-1's
    # output (events order each copy against the compute that uses the set).
    h_in = [x.cpu().pin_memory() for x in e2e_sets[0][0]]
    h_out = [torch.empty(y.shape, dtype=y.dtype).pin_memory() for y in e2e_sets[0][1]]
    h2d = sum(t.numel() * t.element_size() for t in h_in)
    d2h = sum(t.numel() * t.element_size() for t in h_out)
    sets = e2e_sets
    # uploads and downloads on two streams of their own, so that the two copy
    # directions run at the same time as each other and as the compute (two
    # upload streams sharing the inputs measured no faster)
    in_stream, out_stream = torch.cuda.Stream(dev), torch.cuda.Stream(dev)

    def e2e_run(n):
        """n steps; returns after enqueueing everything (compute stream last)."""
        in_ready = [torch.cuda.Event(), torch.cuda.Event()]
        done = [torch.cuda.Event(), torch.cuda.Event()]
        out_done = [torch.cuda.Event(), torch.cuda.Event()]
        in_stream.wait_stream(stream)
        out_stream.wait_stream(stream)

        def upload(k):
            with torch.cuda.stream(in_stream):
                for d, h in zip(sets[k % 2][0], h_in):
                    d.copy_(h, non_blocking=True)
                in_ready[k % 2].record(in_stream)

        upload(0)
        for i in range(n):
            if i + 1 < n:
                if i >= 1:
                    in_stream.wait_event(done[(i + 1) % 2])  # inputs of set (i+1)%2 last read by step i-1
                upload(i + 1)
            stream.wait_event(in_ready[i % 2])
            if i >= 2:
                stream.wait_event(out_done[i % 2])  # step i-2's output (same set) has been read back
            step(i % 2)
            done[i % 2].record(stream)
            out_stream.wait_event(done[i % 2])
            with torch.cuda.stream(out_stream):
                for h, d in zip(h_out, sets[i % 2][1]):
                    h.copy_(d, non_blocking=True)
                out_done[i % 2].record(out_stream)
        for e in out_done[:min(n, 2)]:
            stream.wait_event(e)

    e2e_run(max(1, args.warmup))
    torch.cuda.synchronize()
    barrier(dist, local)
    e2, e3 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e2.record(stream)
    e2e_run(args.steps)
    e3.record(stream)
    torch.cuda.synchronize()
    ms_e2e = max_over_ranks(dist, e2.elapsed_time(e3), dev)
    e2e_value = job_throughput(ws, flops_step, args.steps, ms_e2e)

    # ---- roofline of the dominant kernel -----------------------------------
    peaks = load_peaks()
    region_s = ms_max * 1e-3
    peak_t, peak_kind_t = pick_peak(peaks, region_s, w.dtype)
    kb = hbm_kernel_bytes(w)
    # per-kernel table from the profile pass; SM clocks from the timed region
    kernels = {k: v[:2] for k, v in kprof.items() if v[0] > 0}
    per_kernel = {}
    for name, (n, tot) in kernels.items():
        avg = tot / max(1, n)
        ent = {"launches": n, "avg_ms": round(avg, 4), "share": None}
        if name in kf and avg > 0:
            ent["tflops"] = round(kf[name] / (avg * 1e-3) / 1e12, 1)
        if name in kclk and kclk[name][3]:
            ent["sm_mhz"] = round(kclk[name][2] / kclk[name][3] * 1e3, 1)
        if name in kb and avg > 0:
            gbs = kb[name] / (avg * 1e-3) / 1e9
            ent["gbs"] = round(gbs, 1)
            ent["hbm_frac"] = round(gbs / peaks["hbm_gbs"], 4)
        per_kernel[name] = ent
    tot_all = sum(t for _, t in kernels.values()) or 1.0
    for name, (n, tot) in kernels.items():
        per_kernel[name]["share"] = round(tot / tot_all, 4)
    roofline = None
    # the roofline kernel's launches in the timed region (events around them
    # only; none under --graph, whose replays carry no events)
    if dom and dom in kclk and kclk[dom][0] > 0:
        n, tot = kclk[dom][:2]
        avg_s = (tot / n) * 1e-3
        peak, peak_kind, bound = peak_t, peak_kind_t, "tensor"
        if w.dtype == "f32":  # the fp32 engine runs on the CUDA cores' FFMA
            peak, peak_kind = fp32_alu_peak(torch.cuda.get_device_properties(dev).multi_processor_count, peaks)
            bound = "alu"
        gb = gemm_bytes(w)[dom]
        # below the ridge point (peak FLOP/s / peak B/s) the kernel is bound by HBM
        if kf[dom] / gb < peak * 1e12 / (peaks["hbm_gbs"] * 1e9):
            achieved = gb / avg_s / 1e9
            roofline = {"kernel": dom, "bound": "hbm", "achieved": round(achieved, 1), "peak": peaks["hbm_gbs"],
                        "unit": "GB/s", "frac": round(achieved / peaks["hbm_gbs"], 4), "traffic": None,
                        "peak_kind": f"HBM copy ({peaks['source']})", "algorithmic_bytes_per_launch": gb,
                        "tflops": round(kf[dom] / avg_s / 1e12, 1)}
        else:
            achieved = kf[dom] / avg_s / 1e12
            roofline = {"kernel": dom, "bound": bound, "achieved": round(achieved, 1), "peak": round(peak, 1),
                        "unit": "TFLOP/s", "frac": round(achieved / peak, 4), "traffic": None,
                        "peak_kind": peak_kind, "algorithmic_flop_per_launch": kf[dom]}
    if roofline is not None and w.dtype == "bf16" and not layer and roofline["bound"] == "tensor" \
            and not args.seq_len and not args.ffn:
        roofline["traffic"] = recorded_traffic(w, args.tile_mode, dom)
    step_frac = value / ws / peak_t
    return {
        "value": round(value, 2), "ms_per_step": round(ms_max / args.steps, 4),
        "timed_region_s": round(region_s, 4),
        "pct_of_dense_bf16_peak": round(100 * step_frac, 2), "pct_peak_kind": peak_kind_t,
        "e2e": {"value": round(e2e_value, 2), "unit": UNIT, "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h},
        "gpu_launches": launches, "roofline": roofline, "kernels": per_kernel,
        "kernels_timing": f"CUDA events around every launch in a pass of {prof_steps} steps before the timed "
                          "region (the timed region brackets only the roofline kernel); sm_mhz from the timed "
                          "region's in-kernel counters",
        "clocks": clk,
        "peaks": peaks,
    }


# ---------------------------------------------------------------------------
# CPU oracle (cpu_baseline leg and --impl reference)
# ---------------------------------------------------------------------------
def oracle_sample(w, tokens, full=None, block="mlp"):
    """Time the fp64 oracle's fwd+bwd (of the MLP, or of the sub-block) on the
    first `tokens` tokens of the workload with the full weights; returns
    (seconds, algorithmic FLOP)."""
    import oracle
    from oracle import layer as olayer
    if w.kind == "attn_proj":
        return oracle_sample_attn(w, tokens, full)
    if full is None:
        full = synth.mlp_tensors(w, M=tokens)
    W1s = oracle.shard_column_weight(full["W1"], w.T, w.act)
    b1s = oracle.shard_column_bias(full["b1"], w.T, w.act) if w.has_bias else None
    W2s = oracle.shard_row_weight(full["W2"], w.T)
    X, dY = full["X"][:tokens], full["dY"][:tokens]
    t0 = time.perf_counter()
    if block == "layer":
        lnp = synth.layer_tensors(1, w.H, w.dtype)
        f = olayer.layer_fwd(X, lnp["gamma"], lnp["beta"], W1s, b1s, W2s, full["b2"], w.act, LAYER_DROPOUT_P,
                             LAYER_SEED)
        olayer.layer_bwd(dY, X, lnp["gamma"], W1s, W2s, f, w.act, LAYER_DROPOUT_P)
    else:
        pre, A, _ = oracle.mlp_fwd(X, W1s, b1s, W2s, full["b2"], w.act, w.residual)
        oracle.mlp_bwd(dY, X, W1s, W2s, pre, A, w.act, w.residual)
    dt = time.perf_counter() - t0
    flops = 3.0 * (2.0 * tokens * w.H * w.F * w.g + 2.0 * tokens * w.F * w.H)
    return dt, flops


def oracle_sample_attn(w, tokens, full=None):
    """The fp64 oracle's forward and backward of the QKV column layer and the
    output row layer on the first `tokens` tokens; (seconds, FLOP)."""
    import oracle
    if full is None:
        full = synth.attn_tensors(w, M=tokens)
    T = w.T
    Wq = oracle.shard_column_weight(full["Wqkv"], T)
    Wo = oracle.shard_row_weight(full["Wo"], T)
    X, dYo = full["X"][:tokens], full["dYo"][:tokens]
    Zs = oracle.shard_row_weight(full["Z"][:tokens], T)        # column blocks of Z, one per shard
    dYq = oracle.shard_row_weight(full["dYqkv"][:tokens], T)   # column blocks of the QKV gradient
    t0 = time.perf_counter()
    oracle.column_fwd(X, Wq, None, "none")
    oracle.row_fwd(Zs, Wo)
    oracle.column_bwd(dYq, X, Wq)
    oracle.row_bwd(dYo, Zs, Wo)
    dt = time.perf_counter() - t0
    return dt, 3.0 * (2.0 * tokens * w.H * w.F + 2.0 * tokens * w.F_o * w.H)


def workload_tensors(w, M=None):
    return synth.attn_tensors(w, M=M) if w.kind == "attn_proj" else synth.mlp_tensors(w, M=M)


def flop_per_token(w):
    return w.flops() / w.M


def cpu_threads():
    try:
        return len(os.sched_getaffinity(0))
    except Exception:
        return os.cpu_count() or 1


def run_reference(args, w, rank, block="mlp"):
    # per-step sample sized so that warm-up + timed steps take ~2 minutes
    probe_tokens = 64
    full = workload_tensors(w, M=2048)
    dt, fl = oracle_sample(w, probe_tokens, full, block)
    rate = fl / dt
    budget = 120.0 / max(1, args.steps + args.warmup)
    per_token = flop_per_token(w)
    tokens = int(max(64, min(2048, budget * rate / per_token)))
    for _ in range(args.warmup):
        oracle_sample(w, tokens, full, block)
    tot_t, tot_f = 0.0, 0.0
    for _ in range(args.steps):
        dt, fl = oracle_sample(w, tokens, full, block)
        tot_t += dt
        tot_f += fl
    value = tot_f / tot_t / 1e12
    sample = f"first {tokens} of {w.M} tokens per step, full weights, fp64 numpy"
    return {"value": round(value, 5), "ms_per_step": round(1e3 * tot_t / args.steps, 2),
            "cpu_baseline": {"value": round(value, 5), "unit": UNIT, "cores": cpu_threads(), "kind": "oracle",
                             "sample": sample},
            "e2e": {"value": round(value, 5), "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}


def single_core_rate(w, block="mlp"):
    """The oracle's rate on the whole (small) step with one BLAS thread, in a
    child process whose thread counts are fixed before numpy loads."""
    env = dict(os.environ, OPENBLAS_NUM_THREADS="1", OMP_NUM_THREADS="1", MKL_NUM_THREADS="1")
    code = ("import sys; sys.path.insert(0, %r); import bench, synth; w = synth.WORKLOADS[%r]; "
            "dt, fl = bench.oracle_sample(w, w.M, None, %r); print(fl / dt)" % (ROOT, w.name, block))
    try:
        r = subprocess.run([sys.executable, "-c", code], env=env, capture_output=True, text=True, timeout=300)
        return float(r.stdout.strip().splitlines()[-1])
    except Exception:
        return None


def cpu_baseline(w, block="mlp"):
    """The oracle on host cores over a token sample sized to about 15 s of
    work (a probe of up to 512 tokens sets the size; at most the whole step),
    with the full step's time extrapolated from the sample's rate; for the
    tiny workload also the whole step on one core."""
    probe = min(512, w.M)
    full = workload_tensors(w)
    dt, fl = oracle_sample(w, probe, full, block)
    rate = fl / dt
    per_token = fl / probe
    tokens = min(w.M, max(probe, int(15.0 * rate / per_token)))
    if tokens < w.M:
        tokens = tokens // probe * probe
    dt, fl = oracle_sample(w, tokens, full, block)
    reps = 1
    while dt < 5.0 and reps < 10000:  # a small whole step: repeat it for a stable rate
        d2, f2 = oracle_sample(w, tokens, full, block)
        dt, fl, reps = dt + d2, fl + f2, reps + 1
    what = "the whole step" if tokens == w.M else f"the first {tokens} of {w.M} tokens"
    if reps > 1:
        what += f", {reps} times"
    out = {"value": round(fl / dt / 1e12, 5), "unit": UNIT, "cores": cpu_threads(), "kind": "oracle",
           "sample": f"fp64 numpy oracle fwd+bwd on {what} with the full weights "
                     f"({fl / 1e9:.0f} GFLOP, {dt:.1f} s)",
           "step_s": round(w.flops() * dt / fl, 4),
           "step_s_kind": "measured" if tokens == w.M else "extrapolated from the sample's rate"}
    if w.name == "tiny":
        one = single_core_rate(w, block)
        if one:
            out["single_core"] = {"value": round(one / 1e12, 6), "unit": UNIT, "cores": 1,
                                  "sample": "the whole step, one BLAS thread"}
    return out


# ---------------------------------------------------------------------------
def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=100)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default="gpt", choices=sorted(synth.WORKLOADS))
    ap.add_argument("--seq-len", type=int, default=0,
                    help="override the workload's sequence length S (a smaller case of the same kernels, for "
                         "profiling); the printed config names the changed workload")
    ap.add_argument("--ffn", type=int, default=0,
                    help="override the workload's FFN width F (a smaller case of the same kernels with the same K "
                         "of the weight gradients, for profiling); the printed config names the changed workload")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--dtype", default="workload", choices=["workload", "fp8"],
                    help="fp8: the FP8 variant (E4M3 forward, E5M2 backward, bf16 buffers) of the workload")
    ap.add_argument("--block", default="mlp", choices=["mlp", "layer"],
                    help="layer: the TransformerLayer MLP sub-block, Y = X + dropout(MLP(LayerNorm(X))), "
                         f"p = {LAYER_DROPOUT_P}")
    ap.add_argument("--graph", action="store_true",
                    help="replay each step from a CUDA graph captured after the warm-up (no host launch cost)")
    ap.add_argument("--fp8-history", type=int, default=0,
                    help="FP8 delayed scaling over the last N amaxes of every operand (0: current scaling)")
    ap.add_argument("--fused", default="auto", choices=["auto", "on", "off"],
                    help="forward as one fused kernel for narrow MLPs (H <= 256): auto / on / off")
    ap.add_argument("--tile-mode", default="auto", choices=["auto", "single", "pair"],
                    help="bf16 GEMM tiling: CTA-pair 256-row tiles (auto) or single-CTA 128-row tiles")
    ap.add_argument("--wgrad-accumulate", action="store_true",
                    help="micro-batch step: the weight gradients are added into persistent fp32 buffers")
    ap.add_argument("--k-order", default="alternate", choices=["alternate", "forward"],
                    help="K order of the pair GEMMs' whole tiles: every other persistent round backwards "
                         "(alternate, fewer operand re-reads from HBM) or always forwards")
    ap.add_argument("--launch-overlap", default="on", choices=["on", "off"],
                    help="programmatic dependent launch of the pair GEMMs (set-up overlaps the previous kernel)")
    ap.add_argument("--band-rows", type=int, default=0,
                    help="rows of 256-row tiles per raster band of the pair GEMMs' tile order (0: library choice)")
    ap.add_argument("--tail-split", default="on", choices=["on", "off"],
                    help="cut the persistent GEMMs' part-filled last round of tiles along K over all CTA pairs")
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3
    w = synth.WORKLOADS[args.workload]
    import dataclasses
    if args.dtype == "fp8":
        w = dataclasses.replace(w, dtype="fp8")
    if args.seq_len > 0:
        w = dataclasses.replace(w, S=args.seq_len)
    if args.ffn > 0:
        w = dataclasses.replace(w, F=args.ffn)
    if w.kind == "attn_proj" and (w.dtype not in ("bf16", "fp8") or args.block != "mlp"):
        raise SystemExit("the attention projections are timed in bf16 or FP8 as plain layers")
    if w.kind == "attn_proj" and args.fp8_history:
        raise SystemExit("the single layers quantise with current scaling (no amax history)")
    ws, rank, local = dist_env()
    if w.kind == "attn_proj":
        desc = (f"{w.name}: X [S={w.S},B={w.B},H={w.H}] {w.dtype}, QKV column layer H -> {w.F} and output row "
                f"layer {w.F_o} -> H, T={w.T}, no activation, no bias")
    else:
        desc = (f"{w.name}: X [S={w.S},B={w.B},H={w.H}] {w.dtype}, F={w.F}, T={w.T}, {w.act}"
                f"{', bias' if w.has_bias else ''}{', residual' if w.residual else ''}"
                f"{', sequence-parallel' if w.seq_parallel else ''}")
    config = {"workload": desc,
              "S": w.S, "B": w.B, "H": w.H, "F": w.F, "T": w.T, "act": w.act, "global_batch": w.B * ws,
              "seq_len": w.S, "parallelism": f"tp{w.T} shards on one GPU; {ws} replica(s)",
              "l2": f"inputs larger than L2 (~{step_bytes(w) / 1e9:.1f} GB of operands, activations and "
                    f"gradients per step)",
              "tile_mode": args.tile_mode, "fused_fwd": args.fused, "tail_split": args.tail_split,
              "k_order": args.k_order, "band_rows": args.band_rows or "library choice",
              "launch_overlap": args.launch_overlap,
              "wgrad_accumulate": args.wgrad_accumulate,
              "launch": "CUDA graph replay per step" if args.graph else "eager C-ABI calls per step"}
    if w.dtype == "fp8":
        config["fp8_scaling"] = (f"delayed, amax history {args.fp8_history}" if args.fp8_history
                                 else "current (each tensor's own amax)")
    if args.block == "layer":
        config["workload"] += f"; TransformerLayer MLP sub-block: LayerNorm -> MLP -> dropout(p={LAYER_DROPOUT_P})" \
                              " + residual"
        config["block"] = "layer"
    base = {"metric": METRIC, "unit": UNIT, "n_gpus": ws, "steps": args.steps, "warmup": args.warmup,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": w.dtype,
            "data": "synthetic (seeded SplitMix64 + Box-Muller), random-init weights", "config": config}

    if args.impl == "reference":
        if rank != 0:
            return
        out = dict(base)
        out["impl"] = "reference"
        out["n_gpus"] = 1
        out["dtype"] = "f64"
        out.update(run_reference(args, w, rank, args.block))
        print(json.dumps(out))
        return

    import torch
    dist = dist_init(ws, "nccl" if torch.cuda.is_available() else "gloo")
    res = run_gpu(args, w, dist, rank, local, ws)
    if rank == 0:
        out = dict(base)
        out.update(res)
        if not args.no_cpu_baseline and ws == 1:  # the CPU baseline is an N = 1 measurement
            out["cpu_baseline"] = cpu_baseline(w, args.block)
        print(json.dumps(out))
    if dist is not None:
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
