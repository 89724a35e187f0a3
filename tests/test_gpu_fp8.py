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


def test_fp8_needs_workspace_and_mlp_entry_points(tp):
    lay = tp.TPMLP(S=64, B=2, H=256, F=1024, T=4, act="gelu_tanh", dtype="fp8")
    t = mlp_inputs(128, 256, 1024, 4, "gelu_tanh", "fp8", has_bias=False)
    run = MlpRun(lay, t)
    with pytest.raises(tp.TpError) as e:
        lay.fwd(run.X, run.W1, None, run.W2, None, run.Y, run.pre, run.A)  # no workspace
    assert e.value.status == 1
    L = tp.Layout(S=64, B=2, H=256, F=1024, T=4, act="none", dtype="fp8")
    with pytest.raises(tp.TpError) as e:
        tp.linear_col(L, run.X, run.W1, None, run.A)
    assert e.value.status == 3
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
