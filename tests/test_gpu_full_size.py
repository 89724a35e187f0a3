"""Parity at the measured workloads' full sizes, in the launch configuration
bench.py times, against the fp64 oracle evaluated on samples it can afford:

* token rows (first, last, every sequence-parallel shard boundary and seeded
  random rows): Y, dX, pre_i, A_i -- exact per row, because tokens are
  independent in both passes;
* hidden units (first and last of every shard plus seeded random units):
  dW1 rows, dW2 columns, db1 -- exact per unit;
* db2 in full.

Tolerance: max|gpu - ref| <= 1e-2 * max|ref| over the sampled elements.
"""
import numpy as np
import pytest
import torch

import oracle
import synth
from harness import MlpRun, host, rel_err, status_ok

pytestmark = pytest.mark.gpu

TOL = 1e-2


@pytest.fixture(scope="module")
def tp():
    import tensor_transformer_mlp_shard_gb300 as tp
    from tensor_transformer_mlp_shard_gb300 import build
    build.build()
    return tp


def sample_rows(M, T, sp, n=64, seed=1):
    rng = np.random.default_rng(seed)
    rows = {0, M - 1}
    if sp:
        ms = M // T
        for j in range(1, T):
            rows |= {j * ms - 1, j * ms}
    while len(rows) < n:
        rows.add(int(rng.integers(0, M)))
    return np.array(sorted(rows))


def sample_units(Fs, T, n=16, seed=2):
    rng = np.random.default_rng(seed)
    out = []
    for _ in range(T):
        u = {0, Fs - 1}
        while len(u) < n:
            u.add(int(rng.integers(0, Fs)))
        out.append(np.array(sorted(u)))
    return out


def shard_inputs(w, full):
    t = dict(full)
    t["W1s"] = [np.ascontiguousarray(x) for x in oracle.shard_column_weight(full["W1"], w.T, w.act)]
    t["b1s"] = [np.ascontiguousarray(x) for x in oracle.shard_column_bias(full["b1"], w.T, w.act)] \
        if w.has_bias else None
    t["W2s"] = [np.ascontiguousarray(x) for x in oracle.shard_row_weight(full["W2"], w.T)]
    return t


@pytest.mark.parametrize("name", ["gpt", "swiglu", "sp"])
def test_mlp_workload_sampled(tp, name):
    w = synth.WORKLOADS[name]
    lay = tp.TPMLP(S=w.S, B=w.B, H=w.H, F=w.F, T=w.T, act=w.act, dtype=w.dtype, has_bias=w.has_bias,
                   residual=w.residual, seq_parallel=w.seq_parallel)
    t = shard_inputs(w, synth.mlp_tensors(w))
    run = MlpRun(lay, t)
    run.fwd()
    run.bwd()
    assert status_ok(tp, lay)
    M, T, Fs = w.M, w.T, w.F // w.T
    rows = sample_rows(M, T, w.seq_parallel)
    r = oracle.mlp_rows(rows, t["X"], t["W1s"], t["b1s"], t["W2s"], t["b2"], t["dY"], w.act, w.residual)
    errs = {"Y": rel_err(run.gathered(run.Y)[rows], r["Y"]), "dX": rel_err(run.gathered(run.dX)[rows], r["dX"])}
    for i in range(T):
        errs[f"pre{i}"] = rel_err(host(run.pre[i])[rows], r["pre"][i])
        errs[f"A{i}"] = rel_err(host(run.A[i])[rows], r["A"][i])
    units = sample_units(Fs, T)
    u = oracle.mlp_units(units, t["X"], t["W1s"], t["b1s"], t["W2s"], t["dY"], w.act)
    for i in range(T):
        sel = np.concatenate([units[i], Fs + units[i]]) if w.act == "swiglu" else units[i]
        errs[f"dW1_{i}"] = rel_err(host(run.dW1[i])[sel], u["dW1"][i])
        errs[f"dW2_{i}"] = rel_err(host(run.dW2[i])[:, units[i]], u["dW2"][i])
        if w.has_bias:
            errs[f"db1_{i}"] = rel_err(host(run.db1[i])[sel], u["db1"][i])
    if w.has_bias:
        errs["db2"] = rel_err(host(run.db2), np.asarray(t["dY"], np.float64).sum(axis=0))
    bad = {k: v for k, v in errs.items() if not v <= TOL}
    assert not bad, bad


def test_attention_projections_sampled(tp):
    """QKV ColumnParallelLinear (4096 -> 3x4096, 32 heads over T=8, no
    activation) and the output RowParallelLinear (4096 -> 4096, sum over
    shards), forward and backward, at X [4096, 2, 4096]."""
    w = synth.WORKLOADS["attn_proj"]
    T, M, H, F, Fo = w.T, w.M, w.H, w.F, w.F_o
    full = synth.attn_tensors(w)
    dev = lambda a: torch.from_numpy(np.ascontiguousarray(a)).to("cuda", torch.bfloat16)
    Wq = [np.ascontiguousarray(x) for x in oracle.shard_column_weight(full["Wqkv"], T)]
    Wo = [np.ascontiguousarray(x) for x in oracle.shard_row_weight(full["Wo"], T)]
    Zs = [np.ascontiguousarray(x) for x in oracle.shard_row_weight(full["Z"], T)]   # column blocks of Z
    dYq = [np.ascontiguousarray(x) for x in oracle.shard_row_weight(full["dYqkv"], T)]
    colL = tp.Layout(S=w.S, B=w.B, H=H, F=F, T=T, act="none", dtype="bf16")
    rowL = tp.Layout(S=w.S, B=w.B, H=H, F=Fo, T=T, act="none", dtype="bf16")
    X = dev(full["X"])
    Wqd, Wod, Zd, dYqd = [dev(x) for x in Wq], [dev(x) for x in Wo], [dev(x) for x in Zs], [dev(x) for x in dYq]
    dYo = dev(full["dYo"])
    bf = dict(dtype=torch.bfloat16, device="cuda")
    f32 = dict(dtype=torch.float32, device="cuda")
    Fs, Fos = F // T, Fo // T
    Yq = [torch.empty(M, Fs, **bf) for _ in range(T)]
    Yo = torch.empty(M, H, **bf)
    dX = torch.empty(M, H, **bf)
    dWq = [torch.empty(Fs, H, **f32) for _ in range(T)]
    dZ = [torch.empty(M, Fos, **bf) for _ in range(T)]
    dWo = [torch.empty(H, Fos, **f32) for _ in range(T)]
    tp.linear_col(colL, [X], Wqd, None, Yq)
    tp.linear_row(rowL, Zd, Wod, None, None, [Yo])
    tp.linear_col_bwd(colL, dYqd, [X], Wqd, [dX], dWq, None)
    tp.linear_row_bwd(rowL, [dYo], Zd, Wod, dZ, dWo, None)
    assert tp.sync_status() == 0

    rows = sample_rows(M, T, False)
    Xr = full["X"][rows]
    errs = {}
    pre, _ = oracle.column_fwd(Xr, Wq, None, "none")
    for i in range(T):
        errs[f"Yq{i}"] = rel_err(host(Yq[i])[rows], pre[i])
    errs["Yo"] = rel_err(host(Yo)[rows], oracle.row_fwd([z[rows] for z in Zs], Wo))
    dXr, _, _ = oracle.column_bwd([d[rows] for d in dYq], Xr, Wq)
    errs["dX"] = rel_err(host(dX)[rows], dXr)
    dZr, _, _ = oracle.row_bwd(full["dYo"][rows], [z[rows] for z in Zs], Wo)
    for i in range(T):
        errs[f"dZ{i}"] = rel_err(host(dZ[i])[rows], dZr[i])
    us = sample_units(Fs, T)
    uo = sample_units(Fos, T)
    for i in range(T):
        _, dWu, _ = oracle.column_bwd([dYq[i][:, us[i]]], full["X"], [Wq[i][us[i]]])
        errs[f"dWq{i}"] = rel_err(host(dWq[i])[us[i]], dWu[0])
        _, dWo_u, _ = oracle.row_bwd(full["dYo"], [Zs[i][:, uo[i]]], [Wo[i][:, uo[i]]])
        errs[f"dWo{i}"] = rel_err(host(dWo[i])[:, uo[i]], dWo_u[0])
    bad = {k: v for k, v in errs.items() if not v <= TOL}
    assert not bad, bad


def test_tiny_workload_through_linear_layers(tp):
    """The fp32 Tiny problem run layer by layer (column then row) equals the
    fused MLP entry point bit for bit: same kernels, same order."""
    w = synth.WORKLOADS["tiny"]
    full = synth.mlp_tensors(w)
    t = shard_inputs(w, full)
    lay = tp.TPMLP(S=w.S, B=w.B, H=w.H, F=w.F, T=w.T, act=w.act, dtype="f32", has_bias=True)
    run = MlpRun(lay, t)
    run.fwd()
    colL = tp.Layout(S=w.S, B=w.B, H=w.H, F=w.F, T=w.T, act=w.act, dtype="f32", has_bias=True)
    rowL = tp.Layout(S=w.S, B=w.B, H=w.H, F=w.F, T=w.T, act="none", dtype="f32", has_bias=True)
    A = [torch.empty_like(a) for a in run.A]
    pre = [torch.empty_like(p) for p in run.pre]
    Y = torch.empty_like(run.Y[0])
    tp.linear_col(colL, run.X, run.W1, run.b1, A, pre)
    tp.linear_row(rowL, A, run.W2, run.b2, None, [Y])
    assert status_ok(tp, lay)
    assert torch.equal(Y, run.Y[0])
    for a, b in zip(A + pre, run.A + run.pre):
        assert torch.equal(a, b)
