"""GPU parity of the tensor-parallel MLP against the fp64 oracle, through the
C ABI.  Sizes span several 128 x 256 tiles with ragged tails in M, N and K;
tolerances are max|gpu - ref| <= tol * max|ref| with tol = 1e-5 (fp32) and
1e-2 (bf16)."""
import numpy as np
import pytest
import torch

import oracle
from harness import TOL, MlpRun, host, mlp_inputs, oracle_full, rel_err, status_ok

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def tp():
    import tensor_transformer_mlp_shard_gb300 as tp
    from tensor_transformer_mlp_shard_gb300 import build
    build.build()
    return tp


def _check_all(run, ref, lay, tol):
    T = lay.T
    errs = {}
    errs["Y"] = rel_err(run.gathered(run.Y), ref["Y"])
    for i in range(T):
        errs[f"A{i}"] = rel_err(host(run.A[i]), ref["A"][i])
        errs[f"pre{i}"] = rel_err(host(run.pre[i]), ref["pre"][i])
        errs[f"dW1_{i}"] = rel_err(host(run.dW1[i]), ref["dW1"][i])
        errs[f"dW2_{i}"] = rel_err(host(run.dW2[i]), ref["dW2"][i])
        if lay.has_bias:
            errs[f"db1_{i}"] = rel_err(host(run.db1[i]), ref["db1"][i])
    errs["dX"] = rel_err(run.gathered(run.dX), ref["dX"])
    if lay.has_bias:
        errs["db2"] = rel_err(host(run.db2), ref["db2"])
    bad = {k: v for k, v in errs.items() if not (v <= tol)}
    assert not bad, bad
    return errs


CASES = [
    # M, H, F, T, act, dtype, bias, residual, sp
    (300, 264, 800, 4, "gelu_tanh", "bf16", True, True, False),
    (300, 264, 800, 4, "swiglu", "bf16", True, False, False),
    (300, 264, 800, 2, "none", "bf16", False, True, False),
    (200, 136, 64, 1, "gelu_tanh", "bf16", True, False, False),
    (1024, 264, 1600, 8, "gelu_tanh", "bf16", False, False, True),
    (512, 200, 1024, 4, "swiglu", "bf16", False, True, True),
    (384, 136, 384, 3, "gelu_tanh", "bf16", True, True, True),
    (256, 264, 1024, 4, "swiglu", "bf16", True, False, False),
    (2048, 1024, 8192, 8, "gelu_tanh", "bf16", True, True, False),
    (256, 256, 1024, 2, "gelu_tanh", "f32", True, False, False),
    (300, 264, 800, 4, "swiglu", "f32", True, True, False),
    (120, 72, 240, 3, "gelu_tanh", "f32", True, True, True),
    # enough 64 x 64 tiles that the fp32 engine splits no K range (the other
    # fp32 cases split theirs over clusters of 2 to 8 blocks)
    (1024, 512, 2048, 2, "gelu_tanh", "f32", True, True, False),
    # few weight-gradient tiles and many tokens: split-K weight gradients
    (4100, 256, 512, 2, "gelu_tanh", "bf16", True, True, False),
    (4096, 192, 640, 2, "swiglu", "bf16", False, False, True),
    # the largest shard count (TP_MAX_SHARDS = 16): 16 buffers per operand, 16 K segments
    (2048, 264, 2048, 16, "gelu_tanh", "bf16", True, True, True),
    (300, 136, 512, 16, "swiglu", "bf16", True, False, False),
    (96, 72, 256, 16, "gelu_tanh", "f32", True, True, False),
]


@pytest.fixture(params=["single", "pair"])
def tile_mode(request, tp):
    """Run a test with 128-row single-CTA tiles and with 256-row CTA-pair tiles."""
    tp.set_tile_mode(request.param)
    yield request.param
    tp.set_tile_mode("auto")


@pytest.mark.parametrize("M,H,F,T,act,dtype,bias,residual,sp", CASES)
def test_mlp_matches_oracle(tp, tile_mode, M, H, F, T, act, dtype, bias, residual, sp):
    if dtype == "f32" and tile_mode == "pair":
        pytest.skip("fp32 problems run on the SIMT engine; tiling applies to bf16 only")
    S, B = M // 2, 2
    lay = tp.TPMLP(S=S, B=B, H=H, F=F, T=T, act=act, dtype=dtype, has_bias=bias, residual=residual,
                   seq_parallel=sp)
    t = mlp_inputs(M, H, F, T, act, dtype, has_bias=bias)
    run = MlpRun(lay, t)
    run.fwd()
    run.bwd()
    assert status_ok(tp, lay)
    ref = oracle_full(lay, t)
    _check_all(run, ref, lay, TOL[dtype])


def test_tiny_workload_full(tp):
    """The Tiny problem: X [128,2,256] fp32, W1 [1024,256], W2 [256,1024],
    T=2, GeLU-tanh, biases present and zero; checked in full at 1e-5."""
    import synth
    w = synth.WORKLOADS["tiny"]
    lay = tp.TPMLP(S=w.S, B=w.B, H=w.H, F=w.F, T=w.T, act=w.act, dtype=w.dtype, has_bias=True)
    full = synth.mlp_tensors(w)
    t = dict(full)
    t["W1s"] = oracle.shard_column_weight(full["W1"], w.T, w.act)
    t["b1s"] = oracle.shard_column_bias(full["b1"], w.T, w.act)
    t["W2s"] = oracle.shard_row_weight(full["W2"], w.T)
    t = {k: (np.ascontiguousarray(v) if isinstance(v, np.ndarray) else
             [np.ascontiguousarray(x) for x in v] if isinstance(v, list) else v) for k, v in t.items()}
    run = MlpRun(lay, t)
    run.fwd()
    run.bwd()
    assert status_ok(tp, lay)
    _check_all(run, oracle_full(lay, t), lay, 1e-5)


def test_column_shards_are_independent_bitwise(tp, tile_mode):
    """Changing W1_j / b1_j leaves pre_i and A_i (i != j) bitwise unchanged."""
    lay = tp.TPMLP(S=150, B=2, H=264, F=800, T=4, act="gelu_tanh", dtype="bf16", has_bias=True)
    t = mlp_inputs(300, 264, 800, 4, "gelu_tanh", "bf16")
    run = MlpRun(lay, t)
    run.fwd()
    pre0 = [p.clone() for p in run.pre]
    A0 = [a.clone() for a in run.A]
    run.W1[2].mul_(-1.5)
    run.b1[2].add_(1.0)
    run.fwd()
    assert status_ok(tp, lay)
    for i in range(4):
        same = torch.equal(run.pre[i], pre0[i]) and torch.equal(run.A[i], A0[i])
        assert same == (i != 2)


def test_row_backward_needs_no_reduction_bitwise(tp, tile_mode):
    """Changing W2_j leaves dW2_i bitwise unchanged for every i and dW1_i for
    i != j: the row layer's backward has no cross-shard sum."""
    lay = tp.TPMLP(S=150, B=2, H=264, F=800, T=4, act="swiglu", dtype="bf16")
    t = mlp_inputs(300, 264, 800, 4, "swiglu", "bf16", has_bias=False)
    run = MlpRun(lay, t)
    run.fwd()
    run.bwd()
    dW2 = [d.clone() for d in run.dW2]
    dW1 = [d.clone() for d in run.dW1]
    run.W2[1].mul_(0.5)
    run.bwd()
    assert status_ok(tp, lay)
    for i in range(4):
        assert torch.equal(run.dW2[i], dW2[i])
        assert torch.equal(run.dW1[i], dW1[i]) == (i != 1)


def test_sharded_equals_unsharded_on_gpu(tp):
    """The library at T = 1, 2, 4, 8 on the same full weights gives the same Y
    and dX within tolerance."""
    M, H, F = 256, 256, 1024
    outs = {}
    for T in (1, 2, 4, 8):
        lay = tp.TPMLP(S=128, B=2, H=H, F=F, T=T, act="gelu_tanh", dtype="bf16", has_bias=True, residual=True)
        t = mlp_inputs(M, H, F, T, "gelu_tanh", "bf16")
        run = MlpRun(lay, t)
        run.fwd()
        run.bwd()
        assert status_ok(tp, lay)
        outs[T] = (run.gathered(run.Y), run.gathered(run.dX),
                   oracle.unshard_column([host(d) for d in run.dW1]))
    for T in (2, 4, 8):
        for a, b in zip(outs[T], outs[1]):
            assert rel_err(a, b) < 1e-2


def test_deterministic_and_accumulate(tp, tile_mode):
    lay = tp.TPMLP(S=150, B=2, H=264, F=800, T=4, act="gelu_tanh", dtype="bf16", has_bias=True, residual=True)
    t = mlp_inputs(300, 264, 800, 4, "gelu_tanh", "bf16")
    run = MlpRun(lay, t)
    run.fwd()
    run.bwd()
    Y0, dX0 = [y.clone() for y in run.Y], [d.clone() for d in run.dX]
    dW10 = [d.clone() for d in run.dW1]
    db10 = [d.clone() for d in run.db1]
    run.fwd()
    run.bwd()
    for a, b in zip(Y0 + dX0 + dW10 + db10, run.Y + run.dX + run.dW1 + run.db1):
        assert torch.equal(a, b)
    acc = tp.TPMLP(S=150, B=2, H=264, F=800, T=4, act="gelu_tanh", dtype="bf16", has_bias=True, residual=True,
                   wgrad_accumulate=True)
    acc.bwd(run.dY, run.X, run.W1, run.W2, run.pre, run.A, run.dX, run.dW1, run.db1, run.dW2, run.db2, run.ws)
    assert status_ok(tp, lay, acc)
    for a, b in zip(dW10, run.dW1):
        assert torch.equal(2 * a, b)


def test_split_k_weight_gradients_deterministic_and_accumulate(tp, tile_mode):
    """dW through split-K (8 token splits of a 4100-token K; the reduction adds
    the splits in order): run-to-run identical, and += with accumulation."""
    lay = tp.TPMLP(S=2050, B=2, H=256, F=512, T=2, act="gelu_tanh", dtype="bf16", has_bias=True)
    t = mlp_inputs(4100, 256, 512, 2, "gelu_tanh", "bf16")
    run = MlpRun(lay, t)
    run.fwd()
    run.bwd()
    dW10, dW20 = [d.clone() for d in run.dW1], [d.clone() for d in run.dW2]
    run.bwd()
    for a, b in zip(dW10 + dW20, run.dW1 + run.dW2):
        assert torch.equal(a, b)
    acc = tp.TPMLP(S=2050, B=2, H=256, F=512, T=2, act="gelu_tanh", dtype="bf16", has_bias=True,
                   wgrad_accumulate=True)
    acc.bwd(run.dY, run.X, run.W1, run.W2, run.pre, run.A, run.dX, run.dW1, run.db1, run.dW2, run.db2, run.ws)
    assert status_ok(tp, lay, acc)
    for a, b in zip(dW10 + dW20, run.dW1 + run.dW2):
        assert torch.equal(2 * a, b)


def test_empty_tokens(tp):
    lay = tp.TPMLP(S=0, B=2, H=64, F=256, T=2, act="gelu_tanh", dtype="bf16", has_bias=True)
    t = mlp_inputs(0, 64, 256, 2, "gelu_tanh", "bf16")
    run = MlpRun(lay, t)
    run.fwd()
    run.bwd()
    assert status_ok(tp, lay)
    for d in run.dW1 + run.dW2 + run.db1 + [run.db2]:
        assert torch.count_nonzero(d).item() == 0


def test_bounded_wait_reports_timeout(tp):
    """A kernel waiting on a flag that nothing sets gives up after its limit
    and records TP_ERR_TIMEOUT; the context stays usable."""
    assert tp.sync_status() == 0
    tp.debug_wait_timeout(2_000_000)  # 2 ms
    assert tp.sync_status() == 5
    assert tp.sync_status() == 0
    # the library still computes correctly afterwards
    lay = tp.TPMLP(S=64, B=2, H=64, F=256, T=2, act="gelu_tanh", dtype="bf16", has_bias=True)
    t = mlp_inputs(128, 64, 256, 2, "gelu_tanh", "bf16")
    run = MlpRun(lay, t)
    run.fwd()
    assert status_ok(tp, lay)
    assert rel_err(run.gathered(run.Y), oracle_full(lay, t)["Y"]) < 1e-2


def test_timeout_reaches_only_its_handle(tp):
    """Two MLP handles used on two streams: a bounded wait that runs out under
    handle A is reported by A's status word only.  Handle B's calls in the
    meantime neither see nor clear it, and the word of the calls without a
    handle stays clean."""
    assert tp.sync_status() == 0
    a = tp.TPMLP(S=64, B=2, H=64, F=256, T=2, act="gelu_tanh", dtype="bf16", has_bias=True)
    b = tp.TPMLP(S=64, B=2, H=64, F=256, T=2, act="gelu_tanh", dtype="bf16", has_bias=True)
    assert a.sync_status() == 0 and b.sync_status() == 0
    sa, sb = torch.cuda.Stream(), torch.cuda.Stream()
    t = mlp_inputs(128, 64, 256, 2, "gelu_tanh", "bf16")
    run = MlpRun(b, t)
    torch.cuda.synchronize()  # inputs uploaded before the two streams start
    a.debug_wait_timeout(2_000_000, stream=sa)  # 2 ms, on A's stream
    with torch.cuda.stream(sb):
        run.fwd()
        run.bwd()
    assert b.sync_status(sb) == 0
    assert tp.sync_status(sb) == 0
    assert a.sync_status(sa) == 5
    assert a.sync_status(sa) == 0  # read clears it
    assert rel_err(run.gathered(run.Y), oracle_full(b, t)["Y"]) < 1e-2


def test_kernel_timers_and_selection(tp):
    """The per-kernel timers (tp_prof_enable / tp_prof_collect): every
    launch of a forward+backward step is timed by events and the pair GEMMs
    report their SM clock; with tp_prof_select only the chosen kernel's
    launches carry events, while the other GEMMs are still listed through
    their clock counters (launches 0).  The results do not change."""
    M, H, F, T = 1024, 512, 2048, 4
    lay = tp.TPMLP(S=M // 2, B=2, H=H, F=F, T=T, act="gelu_tanh", dtype="bf16", has_bias=True, residual=True)
    t = mlp_inputs(M, H, F, T, "gelu_tanh", "bf16", has_bias=True)
    run = MlpRun(lay, t)
    gemms = {"col_fwd", "row_fwd", "row_dgrad_act", "wgrad_row", "wgrad_col", "col_dgrad"}
    outs = []
    try:
        for sel in (None, "row_fwd"):
            tp.prof_select(sel)
            tp.prof_enable(True)
            tp.prof_collect()
            run.fwd()
            run.bwd()
            got = tp.prof_collect(clocks=True)
            tp.prof_enable(False)
            assert status_ok(tp, lay)
            outs.append([host(x) for x in run.Y + run.dX + run.dW1 + run.dW2])
            assert gemms <= set(got), got
            for name in gemms:
                n, ms, cyc, ns = got[name]
                assert cyc > 0 and ns > 0 and 500 < cyc / ns * 1e3 < 2500, (name, got[name])  # MHz
                if sel is None or name == sel:
                    assert n == 1 and ms > 0, (name, got[name])
                else:
                    assert n == 0 and ms == 0, (name, got[name])
            if sel is not None:
                assert all(v[0] == 0 for k, v in got.items() if k != sel), got
    finally:
        tp.prof_select(None)
        tp.prof_enable(False)
    for a, b in zip(*outs):
        assert np.array_equal(a, b)


def test_binding_rejects_wrong_shapes(tp):
    lay = tp.TPMLP(S=64, B=2, H=64, F=256, T=2, act="gelu_tanh", dtype="bf16", has_bias=True)
    t = mlp_inputs(128, 64, 256, 2, "gelu_tanh", "bf16")
    run = MlpRun(lay, t)
    with pytest.raises(ValueError):
        lay.fwd(run.X, run.W1[:1], run.b1, run.W2, run.b2, run.Y, run.pre, run.A)
    with pytest.raises(ValueError):
        lay.fwd([run.X[0][:100]], run.W1, run.b1, run.W2, run.b2, run.Y, run.pre, run.A)


@pytest.mark.parametrize("bias", [False, True])
def test_single_layer_backward_with_split_k(tp, bias):
    """tp_linear_col_bwd / tp_linear_row_bwd where the weight gradient splits
    its 4100 tokens (2 output tiles per layer): the caller workspace carries
    the bias partials and the split partials side by side."""
    M, H, F, T = 4100, 256, 512, 2
    Fs = F // T
    g = torch.Generator().manual_seed(21)
    bf, f32 = torch.bfloat16, torch.float32
    rnd = lambda *s, sc=1.0: (torch.randn(*s, generator=g) * sc).to(bf)
    X, dOut, W = rnd(M, H), [rnd(M, Fs) for _ in range(T)], [rnd(Fs, H, sc=0.05) for _ in range(T)]
    colL = tp.Layout(S=M // 2, B=2, H=H, F=F, T=T, act="none", dtype="bf16", has_bias=bias)
    ws = tp.alloc_workspace(tp.linear_workspace_bytes(colL))
    dX = torch.empty(M, H, dtype=bf, device="cuda")
    dW = [torch.empty(Fs, H, dtype=f32, device="cuda") for _ in range(T)]
    db = [torch.empty(Fs, dtype=f32, device="cuda") for _ in range(T)] if bias else None
    tp.linear_col_bwd(colL, [d.cuda() for d in dOut], [X.cuda()], [w.cuda() for w in W], [dX], dW, db, ws)
    rowL = tp.Layout(S=M // 2, B=2, H=H, F=F, T=T, act="none", dtype="bf16", has_bias=bias)
    dY, Xr, W2 = rnd(M, H), [rnd(M, Fs) for _ in range(T)], [rnd(H, Fs, sc=0.05) for _ in range(T)]
    ws2 = tp.alloc_workspace(tp.linear_workspace_bytes(rowL))
    dXr = [torch.empty(M, Fs, dtype=bf, device="cuda") for _ in range(T)]
    dW2 = [torch.empty(H, Fs, dtype=f32, device="cuda") for _ in range(T)]
    db2 = torch.empty(H, dtype=f32, device="cuda") if bias else None
    tp.linear_row_bwd(rowL, [dY.cuda()], [x.cuda() for x in Xr], [w.cuda() for w in W2], dXr, dW2, db2, ws2)
    assert tp.sync_status() == 0
    n = lambda t: t.float().numpy()
    rdX, rdW, rdb = oracle.column_bwd([n(d) for d in dOut], n(X), [n(w) for w in W])
    errs = {"dX": rel_err(host(dX), rdX)}
    for i in range(T):
        errs[f"dW{i}"] = rel_err(host(dW[i]), rdW[i])
        if bias:
            errs[f"db{i}"] = rel_err(host(db[i]), rdb[i])
    qdX, qdW, qdb = oracle.row_bwd(n(dY), [n(x) for x in Xr], [n(w) for w in W2])
    for i in range(T):
        errs[f"row_dX{i}"] = rel_err(host(dXr[i]), qdX[i])
        errs[f"row_dW{i}"] = rel_err(host(dW2[i]), qdW[i])
    if bias:
        errs["row_db"] = rel_err(host(db2), qdb)
    bad = {k: v for k, v in errs.items() if not v <= 1e-2}
    assert not bad, bad
