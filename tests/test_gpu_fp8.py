"""GPU parity of the FP8 variant ("Megatron-LM 源码精读" s8.2: E4M3 forward,
E5M2 backward, per-tensor scaling from the amax) against the FP8 oracle
(oracle/fp8.py), through the C ABI.

* The quantiser's codes are compared bit for bit (both sides take the
  rounding decision on the same fp32 product x * scale).
* The MLP is compared with the oracle's FP8 pipeline element by element on
  ragged multi-tile sizes, tolerance 3e-2 * max|ref|.  The two sides form the
  quantiser inputs A and dPre slightly differently (fp32 sums and the SFU tanh
  against fp64), so when a tensor's amax moves by one bf16 step (2^-8
  relative) a fraction of about 2^-8 / 2^-3 of its E4M3 codes (2^-8 / 2^-2 of
  E5M2 codes) lands one FP8 step (2^-3 / 2^-2 relative) apart; summed over K
  with random signs that is about sqrt(p) * step = 2-3% of a typical output,
  about 1% of max|ref|.
* At the GPT workload's full size the same comparison runs on sampled token
  rows and hidden units (oracle.fp8.mlp_sampled_fp8).
"""
import numpy as np
import pytest
import torch

import oracle
import synth
from harness import MlpRun, host, mlp_inputs, rel_err, status_ok
from oracle import fp8

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def tp():
    import tensor_transformer_mlp_shard_gb300 as tp
    from tensor_transformer_mlp_shard_gb300 import build
    build.build()
    return tp


@pytest.fixture(params=["single", "pair"])
def tile_mode(request, tp):
    tp.set_tile_mode(request.param)
    yield request.param
    tp.set_tile_mode("auto")


def _decode(codes: torch.Tensor, fmt: str) -> np.ndarray:
    dt = torch.float8_e4m3fn if fmt == "e4m3" else torch.float8_e5m2
    return codes.view(dt).to(torch.float64).cpu().numpy()


@pytest.mark.parametrize("fmt", ["e4m3", "e5m2"])
def test_quantize_codes_bit_exact(tp, fmt):
    g = torch.Generator().manual_seed(7)
    sizes = [4096 * 3, 8, 1000 * 8]
    parts = [(torch.randn(n, generator=g) * 3.0).to(torch.bfloat16) for n in sizes]
    parts[1][:] = 0.0
    parts[2][17] = -41.5   # the amax element sits in one shard
    dev_in = [p.cuda() for p in parts]
    dev_out = [torch.empty(n, dtype=torch.uint8, device="cuda") for n in sizes]
    amax = torch.zeros(1, dtype=torch.float32, device="cuda")
    tp.fp8_quantize(dev_in, dev_out, fmt, amax)
    assert tp.sync_status() == 0
    ref, s = fp8.quantize([p.float().numpy() for p in parts], fmt)
    assert amax.item() == fp8.amax_of([p.float().numpy() for p in parts])
    for o, r in zip(dev_out, ref):
        assert np.array_equal(_decode(o, fmt), r)
    # a tensor of zeros: scale 1, all codes zero
    z = [torch.zeros(64, dtype=torch.bfloat16, device="cuda")]
    zo = [torch.full((64,), 7, dtype=torch.uint8, device="cuda")]
    tp.fp8_quantize(z, zo, fmt, amax)
    assert amax.item() == 0.0 and int(zo[0].sum()) == 0


CASES = [
    # M, H, F, T, act, bias, residual, sp
    (300, 272, 832, 4, "gelu_tanh", True, True, False),
    (300, 272, 832, 4, "swiglu", False, False, False),
    (512, 256, 1024, 4, "gelu_tanh", False, False, True),
    (256, 256, 1024, 4, "swiglu", True, True, False),
    (2048, 1024, 8192, 8, "gelu_tanh", True, True, False),
    (4096, 256, 512, 2, "gelu_tanh", True, False, False),  # split-K weight gradients
]


@pytest.mark.parametrize("M,H,F,T,act,bias,residual,sp", CASES)
def test_fp8_mlp_matches_fp8_oracle(tp, tile_mode, M, H, F, T, act, bias, residual, sp):
    lay = tp.TPMLP(S=M // 2, B=2, H=H, F=F, T=T, act=act, dtype="fp8", has_bias=bias, residual=residual,
                   seq_parallel=sp)
    t = mlp_inputs(M, H, F, T, act, "fp8", has_bias=bias)
    run = MlpRun(lay, t)
    run.fwd()
    run.bwd()
    assert status_ok(tp, lay)
    f = fp8.mlp_fwd_fp8(t["X"], t["W1s"], t["b1s"], t["W2s"], t["b2"], act, residual)
    gr = fp8.mlp_bwd_fp8(t["dY"], f, act, residual)
    errs = {"Y": rel_err(run.gathered(run.Y), f["Y"]), "dX": rel_err(run.gathered(run.dX), gr["dX"])}
    for i in range(T):
        errs[f"pre{i}"] = rel_err(host(run.pre[i]), f["pre"][i])
        errs[f"A{i}"] = rel_err(host(run.A[i]), f["A"][i])
        errs[f"dW1_{i}"] = rel_err(host(run.dW1[i]), gr["dW1"][i])
        errs[f"dW2_{i}"] = rel_err(host(run.dW2[i]), gr["dW2"][i])
        if bias:
            errs[f"db1_{i}"] = rel_err(host(run.db1[i]), gr["db1"][i])
    if bias:
        errs["db2"] = rel_err(host(run.db2), gr["db2"])
    bad = {k: v for k, v in errs.items() if not v <= 3e-2}
    assert not bad, bad


def test_fp8_forward_needs_a_workspace(tp):
    lay = tp.TPMLP(S=64, B=2, H=256, F=1024, T=4, act="gelu_tanh", dtype="fp8")
    t = mlp_inputs(128, 256, 1024, 4, "gelu_tanh", "fp8", has_bias=False)
    run = MlpRun(lay, t)
    with pytest.raises(tp.TpError) as e:
        lay.fwd(run.X, run.W1, None, run.W2, None, run.Y, run.pre, run.A)  # no workspace
    assert e.value.status == 1
    L = tp.Layout(S=64, B=2, H=256, F=1024, T=4, act="none", dtype="fp8")
    with pytest.raises(tp.TpError) as e:
        tp.linear_col(L, run.X, run.W1, None, run.A)  # no workspace
    assert e.value.status == 1
    assert status_ok(tp, lay)


def test_fp8_gpt_full_size_sampled(tp):
    """GPT workload (S=2048, B=4, H=4096, F=16384, T=8) in FP8, in the launch
    configuration bench.py times, against the FP8 oracle on sampled token rows
    and hidden units (the oracle forms A and dPre in full for their amax)."""
    w = synth.WORKLOADS["gpt"]
    lay = tp.TPMLP(S=w.S, B=w.B, H=w.H, F=w.F, T=w.T, act=w.act, dtype="fp8", has_bias=w.has_bias,
                   residual=w.residual)
    full = synth.mlp_tensors(w)
    t = dict(full)
    t["W1s"] = [np.ascontiguousarray(x) for x in oracle.shard_column_weight(full["W1"], w.T)]
    t["b1s"] = [np.ascontiguousarray(x) for x in oracle.shard_column_bias(full["b1"], w.T)]
    t["W2s"] = [np.ascontiguousarray(x) for x in oracle.shard_row_weight(full["W2"], w.T)]
    run = MlpRun(lay, t)
    run.fwd()
    run.bwd()
    assert status_ok(tp, lay)
    rows = np.array(sorted({0, 1, 777, 4095, 4096, 8190, 8191} | set(np.random.default_rng(5).integers(0, w.M, 25))))
    Fs = w.F // w.T
    units = [np.array([0, 100, Fs - 1]) for _ in range(w.T)]
    r = fp8.mlp_sampled_fp8(rows, units, t["X"], t["W1s"], t["b1s"], t["W2s"], t["b2"], t["dY"], w.act,
                            w.residual)
    errs = {"Y": rel_err(run.gathered(run.Y)[rows], r["Y"]), "dX": rel_err(run.gathered(run.dX)[rows], r["dX"]),
            "db2": rel_err(host(run.db2), r["db2"])}
    for i in range(w.T):
        errs[f"dW1_{i}"] = rel_err(host(run.dW1[i])[units[i]], r["dW1"][i])
        errs[f"dW2_{i}"] = rel_err(host(run.dW2[i])[:, units[i]], r["dW2"][i])
        errs[f"db1_{i}"] = rel_err(host(run.db1[i])[units[i]], r["db1"][i])
    bad = {k: v for k, v in errs.items() if not v <= 3e-2}
    assert not bad, bad


@pytest.mark.parametrize("n", [1, 3])
def test_fp8_delayed_scaling_matches_oracle_over_steps(tp, n):
    """Delayed scaling (amax history of length n) over four steps whose inputs
    change scale (X x1, x1.6, x0.8, x1.2; dY x1, x0.5, x2, x1): every step's
    outputs against the FP8 oracle driven by the same history (step 2 of the
    n = 1 run saturates the X codes that outgrew the first step's scale)."""
    M, H, F, T, act = 384, 256, 1024, 4, "gelu_tanh"
    lay = tp.TPMLP(S=M // 2, B=2, H=H, F=F, T=T, act=act, dtype="fp8", has_bias=True, residual=True)
    lay.set_fp8_history(n)
    base = mlp_inputs(M, H, F, T, act, "fp8", has_bias=True)
    hist = fp8.AmaxHistory(n)
    run = MlpRun(lay, base)
    for step, (sx, sdy) in enumerate([(1.0, 1.0), (1.6, 0.5), (0.8, 2.0), (1.2, 1.0)]):
        t = dict(base)
        t["X"] = fp8.round_bf16(base["X"] * sx).astype(np.float32)
        t["dY"] = fp8.round_bf16(base["dY"] * sdy).astype(np.float32)
        run.X[0].copy_(torch.from_numpy(t["X"]).to(torch.bfloat16))
        run.dY[0].copy_(torch.from_numpy(t["dY"]).to(torch.bfloat16))
        run.fwd()
        run.bwd()
        assert status_ok(tp, lay)
        f = fp8.mlp_fwd_fp8(t["X"], t["W1s"], t["b1s"], t["W2s"], t["b2"], act, True, hist)
        gr = fp8.mlp_bwd_fp8(t["dY"], f, act, True, hist)
        errs = {"Y": rel_err(run.gathered(run.Y), f["Y"]), "dX": rel_err(run.gathered(run.dX), gr["dX"]),
                "db2": rel_err(host(run.db2), gr["db2"])}
        for i in range(T):
            errs[f"A{i}"] = rel_err(host(run.A[i]), f["A"][i])
            errs[f"dW1_{i}"] = rel_err(host(run.dW1[i]), gr["dW1"][i])
            errs[f"dW2_{i}"] = rel_err(host(run.dW2[i]), gr["dW2"][i])
            errs[f"db1_{i}"] = rel_err(host(run.db1[i]), gr["db1"][i])
        bad = {k: v for k, v in errs.items() if not v <= 3e-2}
        assert not bad, (step, bad)


def test_fp8_history_setter_validates(tp):
    lay = tp.TPMLP(S=64, B=2, H=256, F=1024, T=4, act="gelu_tanh", dtype="fp8")
    for bad in (-1, 65):
        with pytest.raises(tp.TpError) as e:
            lay.set_fp8_history(bad)
        assert e.value.status == 1
    lay.set_fp8_history(0)
    lay.set_fp8_history(64)


@pytest.mark.parametrize("n", [0, 1])
@pytest.mark.parametrize("act,F", [("gelu_tanh", 1024), ("gelu_tanh", 320), ("swiglu", 1024)])
def test_fp8_amax_of_every_operand(tp, n, act, F):
    """The amaxes a step records (tp_mlp_fp8_amax; "Megatron-LM 源码精读" s8.2,
    the amax reduced over all shards of a tensor) equal max |x| of X, W1, W2,
    dY and of the bf16 A the forward stored, exactly.  Under delayed scaling
    (n = 1) the second step takes A's amax from the column GEMM's epilogue (a
    max over the packed bf16 pairs it stores) and dPre's from the act' dgrad's;
    under current scaling both come from separate passes.  F = 320 (F/T = 80)
    leaves a part-filled 32-column block in every tile row.  dPre is formed
    with different rounding on the two sides (see the module docstring), so
    its amax is compared with the FP8 oracle's to 2^-5."""
    M, H, T = 384, 256, 4
    lay = tp.TPMLP(S=M // 2, B=2, H=H, F=F, T=T, act=act, dtype="fp8", has_bias=True, residual=True)
    lay.set_fp8_history(n)
    t = mlp_inputs(M, H, F, T, act, "fp8", has_bias=True)
    run = MlpRun(lay, t)
    hist = fp8.AmaxHistory(n) if n else None
    for _ in range(2):
        run.fwd()
        run.bwd()
        f = fp8.mlp_fwd_fp8(t["X"], t["W1s"], t["b1s"], t["W2s"], t["b2"], act, True, hist)
        gr = fp8.mlp_bwd_fp8(t["dY"], f, act, True, hist)
    assert status_ok(tp, lay)
    got = host(lay.fp8_amax(run.ws)).astype(np.float64)

    def amax(bufs):
        return max(float(b.float().abs().max()) for b in bufs)

    want = [amax(run.X), amax(run.W1), amax(run.W2), amax(run.A), amax(run.dY)]
    assert list(got[:5]) == want, dict(zip(lay.FP8_AMAX_NAMES, zip(got, want)))
    ref_dp = float(fp8.amax_of(gr["dPre"]))
    assert abs(got[5] - ref_dp) <= 2 ** -5 * ref_dp, (got[5], ref_dp)


# ---------------------------------------------------------------------------
# single layers in FP8 (tp_linear_*_ws and the backward with the same
# workspace).  The quantiser inputs are the bf16 inputs themselves, so both
# sides quantise identical values with identical scales; the outputs differ
# by the fp32 summation and the bf16 store only: the bf16 tolerance applies.
# ---------------------------------------------------------------------------
LAYER_CASES = [
    # M, H, F, T, bias, sp
    (300, 272, 832, 4, True, False),
    (512, 256, 1024, 4, False, True),
    (4096, 256, 512, 2, True, False),  # split-K weight gradients
    (2048, 1024, 8192, 8, False, False),
]


def _layer_tensors(M, H, F, T, seed):
    base = synth.SEED_BASE + 7000 + 10 * seed
    Fs = F // T
    r = lambda k, shape, std=1.0: synth.round_bf16(synth.normal(base + k, shape, std))
    return {"X": r(0, (M, H)), "W": [r(1 + i, (Fs, H), 0.02) for i in range(T)],
            "b": [r(20 + i, (Fs,), 0.02) for i in range(T)], "dO": [r(40 + i, (M, Fs)) for i in range(T)],
            "Xr": [r(60 + i, (M, Fs)) for i in range(T)], "W2": [r(80 + i, (H, Fs), 0.02) for i in range(T)],
            "b2": r(100, (H,), 0.02), "R": r(101, (M, H)), "dY": r(102, (M, H))}


def _dev(a):
    return torch.from_numpy(np.ascontiguousarray(a)).to("cuda", torch.bfloat16)


@pytest.mark.parametrize("M,H,F,T,bias,sp", LAYER_CASES)
def test_fp8_linear_layers_match_fp8_oracle(tp, tile_mode, M, H, F, T, bias, sp):
    t = _layer_tensors(M, H, F, T, 1)
    Fs = F // T
    bf, f32 = dict(dtype=torch.bfloat16, device="cuda"), dict(dtype=torch.float32, device="cuda")
    split = (lambda a: [np.ascontiguousarray(x) for x in oracle.sp_split(a, T)]) if sp else (lambda a: [a])
    # column layer (no activation) forward and backward, one workspace
    col = tp.Layout(S=M // 2, B=2, H=H, F=F, T=T, act="none", dtype="fp8", has_bias=bias, seq_parallel=sp)
    ws = tp.alloc_workspace(tp.linear_workspace_bytes(col))
    X = [_dev(x) for x in split(t["X"])]
    W = [_dev(w) for w in t["W"]]
    b = [_dev(x) for x in t["b"]] if bias else None
    out = [torch.empty(M, Fs, **bf) for _ in range(T)]
    tp.linear_col(col, X, W, b, out, workspace=ws)
    dX = [torch.empty(col.xrows, H, **bf) for _ in range(col.nx)]
    dW = [torch.empty(Fs, H, **f32) for _ in range(T)]
    db = [torch.empty(Fs, **f32) for _ in range(T)] if bias else None
    tp.linear_col_bwd(col, [_dev(d) for d in t["dO"]], X, W, dX, dW, db, workspace=ws)
    # row layer (bias, residual) forward and backward
    row = tp.Layout(S=M // 2, B=2, H=H, F=F, T=T, act="none", dtype="fp8", has_bias=bias, residual=bias,
                    seq_parallel=sp)
    ws2 = tp.alloc_workspace(tp.linear_workspace_bytes(row))
    Xr, W2 = [_dev(x) for x in t["Xr"]], [_dev(w) for w in t["W2"]]
    Y = [torch.empty(row.xrows, H, **bf) for _ in range(row.nx)]
    tp.linear_row(row, Xr, W2, _dev(t["b2"]) if bias else None, [_dev(x) for x in split(t["R"])] if bias else None,
                  Y, workspace=ws2)
    dXr = [torch.empty(M, Fs, **bf) for _ in range(T)]
    dWr = [torch.empty(H, Fs, **f32) for _ in range(T)]
    dbr = torch.empty(H, **f32) if bias else None
    tp.linear_row_bwd(row, [_dev(x) for x in split(t["dY"])], Xr, W2, dXr, dWr, dbr, workspace=ws2)
    assert tp.sync_status() == 0

    gather = lambda bufs: np.concatenate([host(x) for x in bufs], axis=0)
    pre, o = fp8.column_fwd_fp8(t["X"], t["W"], t["b"] if bias else None, "none")
    cdX, cdW, cdb = fp8.column_bwd_fp8(t["dO"], t["X"], t["W"])
    Yr = fp8.row_fwd_fp8(t["Xr"], t["W2"], t["b2"] if bias else None, t["R"] if bias else None)
    rdX, rdW, rdb = fp8.row_bwd_fp8(t["dY"], t["Xr"], t["W2"])
    errs = {"col_dX": rel_err(gather(dX), cdX), "row_Y": rel_err(gather(Y), Yr)}
    for i in range(T):
        errs[f"col_out{i}"] = rel_err(host(out[i]), o[i])
        errs[f"col_dW{i}"] = rel_err(host(dW[i]), cdW[i])
        errs[f"row_dX{i}"] = rel_err(host(dXr[i]), rdX[i])
        errs[f"row_dW{i}"] = rel_err(host(dWr[i]), rdW[i])
        if bias:
            errs[f"col_db{i}"] = rel_err(host(db[i]), cdb[i])
    if bias:
        errs["row_db"] = rel_err(host(dbr), rdb)
    bad = {k: v for k, v in errs.items() if not v <= 1e-2}
    assert not bad, bad


def test_fp8_column_layer_with_activation(tp):
    """The FP8 column forward with its GeLU epilogue: pre and the activation
    against the oracle."""
    M, H, F, T = 300, 272, 832, 4
    t = _layer_tensors(M, H, F, T, 2)
    Fs = F // T
    col = tp.Layout(S=M // 2, B=2, H=H, F=F, T=T, act="gelu_tanh", dtype="fp8", has_bias=True)
    ws = tp.alloc_workspace(tp.linear_workspace_bytes(col))
    out = [torch.empty(M, Fs, dtype=torch.bfloat16, device="cuda") for _ in range(T)]
    pre = [torch.empty(M, Fs, dtype=torch.bfloat16, device="cuda") for _ in range(T)]
    tp.linear_col(col, [_dev(t["X"])], [_dev(w) for w in t["W"]], [_dev(b) for b in t["b"]], out, pre,
                  workspace=ws)
    assert tp.sync_status() == 0
    rp, ro = fp8.column_fwd_fp8(t["X"], t["W"], t["b"], "gelu_tanh")
    for i in range(T):
        assert rel_err(host(pre[i]), rp[i]) <= 1e-2
        assert rel_err(host(out[i]), ro[i]) <= 1e-2


def test_fp8_attention_projections_sampled(tp):
    """The attention projections' workload (QKV column layer 4096 -> 3 x 4096
    and output row layer 4096 -> 4096 over T = 8, X [4096, 2, 4096]) in FP8,
    in the launch configuration bench.py times, against the FP8 oracle on
    sampled token rows and units."""
    from test_gpu_full_size import sample_rows, sample_units
    w = synth.WORKLOADS["attn_proj"]
    T, M, H, F, Fo = w.T, w.M, w.H, w.F, w.F_o
    Fs, Fos = F // T, Fo // T
    full = synth.attn_tensors(w)
    Wq = [np.ascontiguousarray(x) for x in oracle.shard_column_weight(full["Wqkv"], T)]
    Wo = [np.ascontiguousarray(x) for x in oracle.shard_row_weight(full["Wo"], T)]
    Zs = [np.ascontiguousarray(x) for x in oracle.shard_row_weight(full["Z"], T)]
    dYq = [np.ascontiguousarray(x) for x in oracle.shard_row_weight(full["dYqkv"], T)]
    colL = tp.Layout(S=w.S, B=w.B, H=H, F=F, T=T, act="none", dtype="fp8")
    rowL = tp.Layout(S=w.S, B=w.B, H=H, F=Fo, T=T, act="none", dtype="fp8")
    wsc = tp.alloc_workspace(tp.linear_workspace_bytes(colL))
    wsr = tp.alloc_workspace(tp.linear_workspace_bytes(rowL))
    bf, f32 = dict(dtype=torch.bfloat16, device="cuda"), dict(dtype=torch.float32, device="cuda")
    X, Wqd, Wod, Zd = _dev(full["X"]), [_dev(x) for x in Wq], [_dev(x) for x in Wo], [_dev(x) for x in Zs]
    Yq = [torch.empty(M, Fs, **bf) for _ in range(T)]
    Yo = torch.empty(M, H, **bf)
    dX = torch.empty(M, H, **bf)
    dWq = [torch.empty(Fs, H, **f32) for _ in range(T)]
    dZ = [torch.empty(M, Fos, **bf) for _ in range(T)]
    dWo = [torch.empty(H, Fos, **f32) for _ in range(T)]
    tp.linear_col(colL, [X], Wqd, None, Yq, workspace=wsc)
    tp.linear_row(rowL, Zd, Wod, None, None, [Yo], workspace=wsr)
    tp.linear_col_bwd(colL, [_dev(x) for x in dYq], [X], Wqd, [dX], dWq, None, workspace=wsc)
    tp.linear_row_bwd(rowL, [_dev(full["dYo"])], Zd, Wod, dZ, dWo, None, workspace=wsr)
    assert tp.sync_status() == 0
    rows = sample_rows(M, T, False)
    us, uo = sample_units(Fs, T), sample_units(Fos, T)
    c = fp8.column_sampled_fp8(rows, us, full["X"], Wq, dYq)
    r = fp8.row_sampled_fp8(rows, uo, Zs, Wo, full["dYo"])
    errs = {"dX": rel_err(host(dX)[rows], c["dX"]), "Yo": rel_err(host(Yo)[rows], r["Y"])}
    for i in range(T):
        errs[f"Yq{i}"] = rel_err(host(Yq[i])[rows], c["pre"][i])
        errs[f"dWq{i}"] = rel_err(host(dWq[i])[us[i]], c["dW"][i])
        errs[f"dZ{i}"] = rel_err(host(dZ[i])[rows], r["dX"][i])
        errs[f"dWo{i}"] = rel_err(host(dWo[i])[:, uo[i]], r["dW"][i])
    bad = {k: v for k, v in errs.items() if not v <= 1e-2}
    assert not bad, bad


def test_fp8_column_layer_swiglu_and_accumulated_weight_gradients(tp):
    """The FP8 column forward with the SwiGLU epilogue (gate and up rows of a
    shard in one tile) against the oracle, and the FP8 single-layer
    backward with wgrad_accumulate: two calls from zero give exactly twice
    one call's weight gradients (one fp32 add per element and call)."""
    M, H, F, T = 300, 272, 832, 4
    Fs = F // T
    t = _layer_tensors(M, H, 2 * F, T, 3)  # W shards of 2 * F/T rows: gate rows, then up rows
    Wg = t["W"]
    col = tp.Layout(S=M // 2, B=2, H=H, F=F, T=T, act="swiglu", dtype="fp8")
    ws = tp.alloc_workspace(tp.linear_workspace_bytes(col))
    bf = dict(dtype=torch.bfloat16, device="cuda")
    out = [torch.empty(M, Fs, **bf) for _ in range(T)]
    pre = [torch.empty(M, 2 * Fs, **bf) for _ in range(T)]
    tp.linear_col(col, [_dev(t["X"])], [_dev(w) for w in Wg], None, out, pre, workspace=ws)
    assert tp.sync_status() == 0
    rp, ro = fp8.column_fwd_fp8(t["X"], Wg, None, "swiglu")
    for i in range(T):
        assert rel_err(host(pre[i]), rp[i]) <= 1e-2
        assert rel_err(host(out[i]), ro[i]) <= 1e-2
    # accumulated weight gradients of the row layer
    acc = tp.Layout(S=M // 2, B=2, H=H, F=F, T=T, act="none", dtype="fp8", wgrad_accumulate=True)
    one = tp.Layout(S=M // 2, B=2, H=H, F=F, T=T, act="none", dtype="fp8")
    f32 = dict(dtype=torch.float32, device="cuda")
    r = _layer_tensors(M, H, F, T, 4)
    Xr, W2, dY = [_dev(x) for x in r["Xr"]], [_dev(w) for w in r["W2"]], [_dev(r["dY"])]
    res = []
    for lay, calls in ((one, 1), (acc, 2)):
        w2 = tp.alloc_workspace(tp.linear_workspace_bytes(lay))
        Y = [torch.empty(M, H, **bf)]
        tp.linear_row(lay, Xr, W2, None, None, Y, workspace=w2)
        dX = [torch.empty(M, Fs, **bf) for _ in range(T)]
        dW = [torch.zeros(H, Fs, **f32) for _ in range(T)]
        for _ in range(calls):
            tp.linear_row_bwd(lay, dY, Xr, W2, dX, dW, None, workspace=w2)
        assert tp.sync_status() == 0
        res.append(dW)
    for a, b in zip(*res):
        assert torch.equal(2 * a, b)
