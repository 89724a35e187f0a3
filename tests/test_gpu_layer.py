"""GPU parity of the TransformerLayer MLP sub-block (the gitcode.csdn.net
Megatron Core walk-through, s03: LayerNorm -> MLP -> bias/dropout/residual
add) against oracle/layer.py, through the C ABI (tp_layer_fwd / tp_layer_bwd).

* The dropout keep flags are integer decisions taken on both sides from the
  same Philox4x32-10 words: they are compared bit for bit (recovered from Y
  with the MLP's weights zeroed, so that Y - X = keep * b2 / (1 - p)).
* Everything else is compared element by element with the fp64 oracle on
  ragged multi-tile sizes, the LayerNorm row widths of every kernel variant
  (a warp per row up to 1024 bf16 / 512 fp32 columns, then a block per row
  with 1, 2 or 4 vectors per thread up to 8192 bf16 / 4096 fp32 columns),
  sequence parallelism and both GEMM tilings: tolerance 1e-2 * max|ref| for bf16 (2^-8 relative storage
  rounding of Xn, pre, A, dPre, dXn plus fp32 sums), 1e-5 for fp32 and, for
  the FP8 MLP inside, 3e-2 against the FP8 oracle (the FP8 MLP's own bound).
"""
import numpy as np
import pytest
import torch

import oracle
import synth
from harness import TOL, dev, host, mlp_inputs, rel_err, split_tokens, status_ok
from oracle import layer as olayer

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


def layer_inputs(M, H, F, T, act, dtype, has_bias, seed_off=0):
    t = mlp_inputs(M, H, F, T, act, dtype, has_bias=has_bias, seed_off=seed_off)
    t.update(synth.layer_tensors(M, H, dtype, seed_off))
    return t


class LayerRun:
    """Device buffers and one forward/backward of tp_layer_* for a handle."""

    def __init__(self, lay, t, device="cuda"):
        import tensor_transformer_mlp_shard_gb300 as tp
        self.lay, self.t = lay, t
        dt = lay.dtype
        T, M, H, Fs, g, sp = lay.T, lay.M, lay.H, lay.Fs, lay.g, lay.seq_parallel
        td = torch.float32 if dt == "f32" else torch.bfloat16
        f32 = torch.float32
        nan = float("nan")
        self.X = [dev(x, dt) for x in split_tokens(t["X"], T, sp)]
        self.dY = [dev(x, dt) for x in split_tokens(t["dY"], T, sp)]
        self.gamma, self.beta = dev(t["gamma"], dt), dev(t["beta"], dt)
        self.W1 = [dev(w, dt) for w in t["W1s"]]
        self.W2 = [dev(w, dt) for w in t["W2s"]]
        self.b1 = [dev(b, dt) for b in t["b1s"]] if lay.has_bias else None
        self.b2 = dev(t["b2"], dt) if lay.has_bias else None
        rows = lay.xrows
        self.Y = [torch.full((rows, H), nan, dtype=td, device=device) for _ in range(lay.nx)]
        self.dX = [torch.full((rows, H), nan, dtype=td, device=device) for _ in range(lay.nx)]
        self.Xn = torch.full((M, H), nan, dtype=td, device=device)
        self.mean = torch.full((M,), nan, dtype=f32, device=device)
        self.rstd = torch.full((M,), nan, dtype=f32, device=device)
        self.pre = [torch.full((M, g * Fs), nan, dtype=td, device=device) for _ in range(T)]
        self.A = [torch.full((M, Fs), nan, dtype=td, device=device) for _ in range(T)]
        self.dW1 = [torch.full((g * Fs, H), nan, dtype=f32, device=device) for _ in range(T)]
        self.dW2 = [torch.full((H, Fs), nan, dtype=f32, device=device) for _ in range(T)]
        self.db1 = [torch.full((g * Fs,), nan, dtype=f32, device=device) for _ in range(T)] \
            if lay.has_bias else None
        self.db2 = torch.full((H,), nan, dtype=f32, device=device) if lay.has_bias else None
        self.dgamma = torch.full((H,), nan, dtype=f32, device=device)
        self.dbeta = torch.full((H,), nan, dtype=f32, device=device)
        self.ws = tp.alloc_workspace(lay.workspace_bytes())

    def fwd(self, seed):
        self.lay.fwd(self.X, self.gamma, self.beta, self.W1, self.b1, self.W2, self.b2, seed, self.Y, self.Xn,
                     self.mean, self.rstd, self.pre, self.A, workspace=self.ws)

    def bwd(self, seed):
        self.lay.bwd(self.dY, self.X, self.gamma, self.Xn, self.mean, self.rstd, self.W1, self.W2, self.pre,
                     self.A, seed, self.dX, self.dgamma, self.dbeta, self.dW1, self.db1, self.dW2, self.db2,
                     self.ws)

    @staticmethod
    def gathered(bufs):
        return np.concatenate([host(b) for b in bufs], axis=0)


def _p32(p):
    """The dropout probability as the C ABI holds it (fp32)."""
    return float(np.float32(p))


SEED = 0x1234_5678_9ABC_DEF0

CASES = [
    # M, H, F, T, act, dtype, bias, sp, p
    (300, 272, 832, 4, "gelu_tanh", "bf16", True, False, 0.1),
    (512, 256, 1024, 4, "swiglu", "bf16", False, True, 0.1),
    (256, 256, 1024, 2, "gelu_tanh", "bf16", True, False, 0.0),
    (130, 4096, 512, 2, "gelu_tanh", "bf16", True, False, 0.25),
    (130, 8192, 256, 2, "swiglu", "bf16", False, False, 0.1),
    (136, 2048, 256, 2, "gelu_tanh", "bf16", True, False, 0.1),
    (72, 1024, 256, 2, "gelu_tanh", "f32", False, False, 0.2),
    (300, 272, 832, 4, "gelu_tanh", "f32", True, False, 0.1),
    (64, 4096, 256, 2, "gelu_tanh", "f32", True, False, 0.5),
    (96, 264, 512, 4, "swiglu", "f32", True, True, 0.1),
]


@pytest.mark.parametrize("M,H,F,T,act,dtype,bias,sp,p", CASES)
def test_layer_matches_oracle(tp, tile_mode, M, H, F, T, act, dtype, bias, sp, p):
    if dtype == "f32" and tile_mode == "pair":
        pytest.skip("the fp32 engine has one tiling")
    lay = tp.TPLayer(S=M // 2, B=2, H=H, F=F, T=T, act=act, dtype=dtype, has_bias=bias, seq_parallel=sp,
                     dropout_p=p)
    t = layer_inputs(M, H, F, T, act, dtype, bias)
    run = LayerRun(lay, t)
    run.fwd(SEED)
    run.bwd(SEED)
    assert status_ok(tp, lay)
    p = _p32(p)
    f = olayer.layer_fwd(t["X"], t["gamma"], t["beta"], t["W1s"], t["b1s"], t["W2s"], t["b2"], act, p, SEED)
    gr = olayer.layer_bwd(t["dY"], t["X"], t["gamma"], t["W1s"], t["W2s"], f, act, p)
    errs = {"Y": rel_err(run.gathered(run.Y), f["Y"]), "Xn": rel_err(host(run.Xn), f["Xn"]),
            "mean": rel_err(host(run.mean), f["mean"]), "rstd": rel_err(host(run.rstd), f["rstd"]),
            "dX": rel_err(run.gathered(run.dX), gr["dX"]), "dgamma": rel_err(host(run.dgamma), gr["dgamma"]),
            "dbeta": rel_err(host(run.dbeta), gr["dbeta"])}
    for i in range(T):
        errs[f"pre{i}"] = rel_err(host(run.pre[i]), f["pre"][i])
        errs[f"A{i}"] = rel_err(host(run.A[i]), f["A"][i])
        errs[f"dW1_{i}"] = rel_err(host(run.dW1[i]), gr["dW1"][i])
        errs[f"dW2_{i}"] = rel_err(host(run.dW2[i]), gr["dW2"][i])
        if bias:
            errs[f"db1_{i}"] = rel_err(host(run.db1[i]), gr["db1"][i])
    if bias:
        errs["db2"] = rel_err(host(run.db2), gr["db2"])
    tol = TOL[dtype]
    bad = {k: v for k, v in errs.items() if not v <= tol}
    assert not bad, bad


@pytest.mark.parametrize("dtype,sp,p", [("bf16", False, 0.1), ("bf16", True, 0.5), ("f32", False, 0.3),
                                         ("f32", True, 0.9)])
def test_dropout_keep_flags_bit_exact(tp, dtype, sp, p):
    """W1 = W2 = 0 and b2 = 1 (b1 = 0) make Z = 1, so Y - X = keep / (1 - p):
    the recovered flags must equal the oracle's for every element."""
    M, H, F, T = 512, 264 if dtype == "f32" else 256, 256, 4
    lay = tp.TPLayer(S=M // 2, B=2, H=H, F=F, T=T, act="gelu_tanh", dtype=dtype, has_bias=True, seq_parallel=sp,
                     dropout_p=p)
    t = layer_inputs(M, H, F, T, "gelu_tanh", dtype, True, seed_off=3)
    t["W1s"] = [np.zeros_like(w) for w in t["W1s"]]
    t["W2s"] = [np.zeros_like(w) for w in t["W2s"]]
    t["b1s"] = [np.zeros_like(b) for b in t["b1s"]]
    t["b2"] = np.ones_like(t["b2"])
    run = LayerRun(lay, t)
    seed = 987654321987
    run.fwd(seed)
    assert status_ok(tp, lay)
    jump = run.gathered(run.Y) - run.gathered(run.X)
    keep = jump > 0.5 / (1.0 - _p32(p))
    ref = olayer.dropout_keep(seed, np.arange(M), H, _p32(p))
    assert np.array_equal(keep, ref)
    # a different seed draws different flags
    run.fwd(seed + 1)
    keep2 = (run.gathered(run.Y) - run.gathered(run.X)) > 0.5 / (1.0 - _p32(p))
    assert not np.array_equal(keep2, keep)


def test_layer_is_deterministic(tp):
    M, H, F, T = 384, 256, 1024, 4
    lay = tp.TPLayer(S=M // 2, B=2, H=H, F=F, T=T, act="gelu_tanh", dtype="bf16", has_bias=True, dropout_p=0.1)
    t = layer_inputs(M, H, F, T, "gelu_tanh", "bf16", True, seed_off=5)
    run = LayerRun(lay, t)
    outs = []
    for _ in range(2):
        run.fwd(SEED)
        run.bwd(SEED)
        outs.append([run.gathered(run.Y), run.gathered(run.dX), host(run.dgamma), host(run.dbeta),
                     host(run.dW1[0]), host(run.db2)])
    assert status_ok(tp, lay)
    for a, b in zip(*outs):
        assert np.array_equal(a, b)


@pytest.mark.parametrize("fused", ["off", "on"])
def test_dropout_backward_mask_equals_redrawn_flags(tp, fused):
    """The backward reads the keep-mask its forward stored in the workspace
    when it gets that workspace and seed back, and redraws the flags from the
    seed otherwise or when the mask fails the kernel's check: all give the
    same bits (also when the fused forward kernel wrote the mask)."""
    M, H, F, T = 300, 256, 1024, 2
    lay = tp.TPLayer(S=M // 2, B=2, H=H, F=F, T=T, act="gelu_tanh", dtype="bf16", has_bias=True, dropout_p=0.25)
    t = layer_inputs(M, H, F, T, "gelu_tanh", "bf16", True, seed_off=7)
    tp.set_fused_fwd(fused)
    run = LayerRun(lay, t)
    run.fwd(SEED)
    fwd_ws = run.ws
    other_ws = tp.alloc_workspace(lay.workspace_bytes())
    outs = []
    for ws, scribble in ((fwd_ws, False), (other_ws, False), (fwd_ws, True)):
        # stored mask; redrawn flags; a mask the workspace no longer holds (the
        # kernel's check of each block's first row catches it and redraws)
        if scribble:
            ws.random_(0, 256)
        run.ws = ws
        run.bwd(SEED)
        outs.append([run.gathered(run.dX), host(run.dgamma), host(run.dbeta), host(run.db2),
                     host(run.dW1[0]), host(run.dW2[1])])
    assert status_ok(tp, lay)
    for later in outs[1:]:
        for a, b in zip(outs[0], later):
            assert np.array_equal(a, b)
    tp.set_fused_fwd("auto")
    f = olayer.layer_fwd(t["X"], t["gamma"], t["beta"], t["W1s"], t["b1s"], t["W2s"], t["b2"], "gelu_tanh",
                         _p32(0.25), SEED)
    gr = olayer.layer_bwd(t["dY"], t["X"], t["gamma"], t["W1s"], t["W2s"], f, "gelu_tanh", _p32(0.25))
    assert rel_err(outs[0][0], gr["dX"]) <= 1e-2
    assert rel_err(outs[0][3], gr["db2"]) <= 1e-2


def test_layer_fp8_matches_fp8_oracle(tp, tile_mode):
    M, H, F, T, act, p = 512, 256, 1024, 4, "gelu_tanh", 0.1
    lay = tp.TPLayer(S=M // 2, B=2, H=H, F=F, T=T, act=act, dtype="fp8", has_bias=True, dropout_p=p)
    t = layer_inputs(M, H, F, T, act, "fp8", True, seed_off=7)
    run = LayerRun(lay, t)
    run.fwd(SEED)
    run.bwd(SEED)
    assert status_ok(tp, lay)
    p = _p32(p)
    f = olayer.layer_fwd_fp8(t["X"], t["gamma"], t["beta"], t["W1s"], t["b1s"], t["W2s"], t["b2"], act, p, SEED)
    gr = olayer.layer_bwd_fp8(t["dY"], t["X"], t["gamma"], act, p, f)
    errs = {"Y": rel_err(run.gathered(run.Y), f["Y"]), "Xn": rel_err(host(run.Xn), f["Xn"]),
            "dX": rel_err(run.gathered(run.dX), gr["dX"]), "dgamma": rel_err(host(run.dgamma), gr["dgamma"]),
            "dbeta": rel_err(host(run.dbeta), gr["dbeta"]), "db2": rel_err(host(run.db2), gr["db2"])}
    for i in range(T):
        errs[f"A{i}"] = rel_err(host(run.A[i]), f["A"][i])
        errs[f"dW1_{i}"] = rel_err(host(run.dW1[i]), gr["dW1"][i])
        errs[f"dW2_{i}"] = rel_err(host(run.dW2[i]), gr["dW2"][i])
        errs[f"db1_{i}"] = rel_err(host(run.db1[i]), gr["db1"][i])
    bad = {k: v for k, v in errs.items() if not v <= 3e-2}
    assert not bad, bad


def test_layer_fp8_amax(tp):
    """tp_layer_fp8_amax: the amaxes of the MLP inside the block equal max |x|
    of the LayerNorm output Xn, W1, W2, the stored bf16 A and (dropout off, so
    the gradient at the MLP's output is the block's dY) dY, exactly; dPre's is
    positive and finite (its exact value is pinned for the MLP entry points)."""
    M, H, F, T, act = 512, 256, 1024, 4, "gelu_tanh"
    lay = tp.TPLayer(S=M // 2, B=2, H=H, F=F, T=T, act=act, dtype="fp8", has_bias=True, dropout_p=0.0)
    lay.set_fp8_history(1)
    t = layer_inputs(M, H, F, T, act, "fp8", True, seed_off=11)
    run = LayerRun(lay, t)
    for _ in range(2):
        run.fwd(SEED)
        run.bwd(SEED)
    assert status_ok(tp, lay)
    got = host(lay.fp8_amax(run.ws)).astype(np.float64)

    def amax(bufs):
        return max(float(b.float().abs().max()) for b in bufs)

    want = [amax([run.Xn]), amax(run.W1), amax(run.W2), amax(run.A), amax(run.dY)]
    assert list(got[:5]) == want, dict(zip(lay.FP8_AMAX_NAMES, zip(got, want)))
    assert 0.0 < got[5] < float("inf")


def test_layer_empty_tokens_zero_the_gradients(tp):
    lay = tp.TPLayer(S=0, B=2, H=256, F=1024, T=4, act="gelu_tanh", dtype="bf16", has_bias=True, dropout_p=0.1)
    t = layer_inputs(0, 256, 1024, 4, "gelu_tanh", "bf16", True)
    run = LayerRun(lay, t)
    run.fwd(SEED)
    run.bwd(SEED)
    assert status_ok(tp, lay)
    for b in [run.dgamma, run.dbeta, run.db2, *run.dW1, *run.dW2, *run.db1]:
        assert torch.count_nonzero(b).item() == 0


def test_layer_gpt_full_size_sampled(tp):
    """The GPT workload (S=2048, B=4, H=4096, F=16384, T=8, GeLU, bias) in the
    sub-block, in the launch configuration `bench.py --block layer` times
    (dropout 0.1, the same seed), against the layer oracle evaluated where it
    is exact on samples: token rows (Y, dX, pre, A through a per-row
    LayerNorm, the row's dropout flags and the MLP rows), hidden units (dW1,
    dW2, db1 over all tokens, from the full LayerNorm output and dZ) and db2
    in full.  dgamma and dbeta need every row's dXn and are checked at the
    mid sizes above."""
    from test_gpu_full_size import sample_rows, sample_units, shard_inputs
    w = synth.WORKLOADS["gpt"]
    p, seed = 0.1, 0x5EED_0000_0001
    lay = tp.TPLayer(S=w.S, B=w.B, H=w.H, F=w.F, T=w.T, act=w.act, dtype=w.dtype, has_bias=w.has_bias,
                     dropout_p=p)
    t = shard_inputs(w, synth.mlp_tensors(w))
    lnp = synth.layer_tensors(1, w.H, w.dtype)
    t["gamma"], t["beta"] = lnp["gamma"], lnp["beta"]
    run = LayerRun(lay, t)
    run.fwd(seed)
    run.bwd(seed)
    assert status_ok(tp, lay)
    p = _p32(p)
    M, H, T, Fs = w.M, w.H, w.T, w.F // w.T
    X = np.asarray(t["X"], np.float64)
    dY = np.asarray(t["dY"], np.float64)
    # token rows
    rows = sample_rows(M, T, False)
    Xn_r, mean_r, rstd_r = olayer.layernorm_fwd(X[rows], t["gamma"], t["beta"])
    keep_r = olayer.dropout_keep(seed, rows, H, p)
    dZ_r = np.where(keep_r, dY[rows] / (1.0 - p), 0.0)
    r = oracle.mlp_rows(np.arange(len(rows)), Xn_r, t["W1s"], t["b1s"], t["W2s"], t["b2"], dZ_r, w.act, False)
    Y_r = X[rows] + np.where(keep_r, r["Y"] / (1.0 - p), 0.0)
    dX_r = dY[rows] + olayer.layernorm_bwd(r["dX"], X[rows], t["gamma"], mean_r, rstd_r)[0]
    errs = {"Y": rel_err(run.gathered(run.Y)[rows], Y_r), "dX": rel_err(run.gathered(run.dX)[rows], dX_r),
            "Xn": rel_err(host(run.Xn)[rows], Xn_r)}
    for i in range(T):
        errs[f"pre{i}"] = rel_err(host(run.pre[i])[rows], r["pre"][i])
        errs[f"A{i}"] = rel_err(host(run.A[i])[rows], r["A"][i])
    # hidden units over all tokens
    Xn = olayer.layernorm_fwd(X, t["gamma"], t["beta"])[0]
    dZ = np.empty_like(dY)
    for r0 in range(0, M, 1024):
        rr = np.arange(r0, min(M, r0 + 1024))
        dZ[rr] = np.where(olayer.dropout_keep(seed, rr, H, p), dY[rr] / (1.0 - p), 0.0)
    units = sample_units(Fs, T)
    u = oracle.mlp_units(units, Xn, t["W1s"], t["b1s"], t["W2s"], dZ, w.act)
    for i in range(T):
        errs[f"dW1_{i}"] = rel_err(host(run.dW1[i])[units[i]], u["dW1"][i])
        errs[f"dW2_{i}"] = rel_err(host(run.dW2[i])[:, units[i]], u["dW2"][i])
        errs[f"db1_{i}"] = rel_err(host(run.db1[i])[units[i]], u["db1"][i])
    errs["db2"] = rel_err(host(run.db2), dZ.sum(axis=0))
    bad = {k: v for k, v in errs.items() if not v <= 1e-2}
    assert not bad, bad


def test_layer_fp8_delayed_scaling_over_steps(tp):
    """The FP8 sub-block with an amax history of 2 over three steps whose
    input grows (x1, x1.5, x0.75) against the FP8 layer oracle driven by the
    same history."""
    from oracle import fp8
    M, H, F, T, act, p = 384, 256, 1024, 4, "gelu_tanh", 0.1
    lay = tp.TPLayer(S=M // 2, B=2, H=H, F=F, T=T, act=act, dtype="fp8", has_bias=True, dropout_p=p)
    lay.set_fp8_history(2)
    base = layer_inputs(M, H, F, T, act, "fp8", True, seed_off=9)
    hist = fp8.AmaxHistory(2)
    run = LayerRun(lay, base)
    for step, sx in enumerate((1.0, 1.5, 0.75)):
        t = dict(base)
        t["X"] = fp8.round_bf16(base["X"] * sx).astype(np.float32)
        run.X[0].copy_(torch.from_numpy(t["X"]).to(torch.bfloat16))
        run.fwd(SEED + step)
        run.bwd(SEED + step)
        assert status_ok(tp, lay)
        f = olayer.layer_fwd_fp8(t["X"], t["gamma"], t["beta"], t["W1s"], t["b1s"], t["W2s"], t["b2"], act,
                                 _p32(p), SEED + step, history=hist)
        gr = olayer.layer_bwd_fp8(t["dY"], t["X"], t["gamma"], act, _p32(p), f, history=hist)
        errs = {"Y": rel_err(run.gathered(run.Y), f["Y"]), "dX": rel_err(run.gathered(run.dX), gr["dX"]),
                "dgamma": rel_err(host(run.dgamma), gr["dgamma"]), "db2": rel_err(host(run.db2), gr["db2"])}
        for i in range(T):
            errs[f"dW1_{i}"] = rel_err(host(run.dW1[i]), gr["dW1"][i])
            errs[f"dW2_{i}"] = rel_err(host(run.dW2[i]), gr["dW2"][i])
        bad = {k: v for k, v in errs.items() if not v <= 3e-2}
        assert not bad, (step, bad)
