"""GPU parity of the pair GEMMs' tail split (tp_set_tail_split): when the
tiles leave the persistent grid's last round part-filled, each tile of that
round is cut along K into s units spread over all CTA pairs; every unit parks
its fp32 partial sum in the workspace and the last unit of each slice adds
them in unit order and runs the epilogue.

The persistent grid is limited to a few CTA pairs (tp_set_max_gemm_pairs) so
that problems the oracle finishes in seconds run several rounds and split
their last one: the MLP's row forward, column dgrad and both weight
gradients, under sequence parallelism and SwiGLU, the single layers'
backward, the sub-block with dropout and FP8.  Each case is checked

* against the fp64 oracle at the MLP's bf16 tolerance (1e-2 max|ref|);
* against the same call with the split off: the sums differ only in how K is
  grouped, so fp32 outputs agree to 1e-5 max|ref| and bf16 outputs to one
  bf16 rounding step (2^-7 max|ref|);
* for run-to-run bit identity (the slice sums are in unit order, whichever
  unit finishes last);
* for the split having run (tp_tail_split_count).
"""
import numpy as np
import pytest
import torch

import oracle
from harness import MlpRun, host, mlp_inputs, oracle_full, rel_err, status_ok

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def tp():
    import tensor_transformer_mlp_shard_gb300 as tp
    from tensor_transformer_mlp_shard_gb300 import build
    build.build()
    yield tp
    tp.set_max_gemm_pairs(0)
    tp.set_tail_split(True)
    tp.set_launch_overlap(True)


def _outputs(run):
    outs = {"Y": run.gathered(run.Y), "dX": run.gathered(run.dX)}
    for i in range(run.lay.T):
        outs[f"dW1_{i}"] = host(run.dW1[i])
        outs[f"dW2_{i}"] = host(run.dW2[i])
        if run.db1 is not None:
            outs[f"db1_{i}"] = host(run.db1[i])
    if run.db2 is not None:
        outs["db2"] = host(run.db2)
    return outs


def _step(tp, lay, t, split, pairs):
    tp.set_tail_split(split)
    tp.set_max_gemm_pairs(pairs)
    run = MlpRun(lay, t)  # workspace sized at these settings
    n0 = tp.tail_split_count()
    run.fwd()
    run.bwd()
    assert status_ok(tp, lay)
    return run, tp.tail_split_count() - n0


def _close(a, b, name):
    tol = 2.0 ** -7 if name in ("Y", "dX") else 1e-5
    return rel_err(a, b.astype(np.float64)) <= tol


CASES = [
    # M, H, F, T, act, bias, residual, sp, pairs, splits expected (row fwd, col dgrad, dW2, dW1)
    (1024, 768, 4096, 8, "gelu_tanh", True, True, False, 11, 4),
    (1024, 768, 2048, 8, "swiglu", False, False, True, 11, 2),
    (1200, 520, 2048, 4, "gelu_tanh", True, False, False, 7, 2),
]


@pytest.mark.parametrize("M,H,F,T,act,bias,residual,sp,pairs,nsplit", CASES)
def test_mlp_tail_split_matches_oracle_and_unsplit(tp, M, H, F, T, act, bias, residual, sp, pairs, nsplit):
    lay = tp.TPMLP(S=M // 2, B=2, H=H, F=F, T=T, act=act, dtype="bf16", has_bias=bias, residual=residual,
                   seq_parallel=sp)
    t = mlp_inputs(M, H, F, T, act, "bf16", has_bias=bias)
    split, n_split = _step(tp, lay, t, True, pairs)
    plain, n_plain = _step(tp, lay, t, False, pairs)
    again, _ = _step(tp, lay, t, True, pairs)
    assert n_split >= nsplit and n_plain == 0, (n_split, n_plain)
    a, b, c = _outputs(split), _outputs(plain), _outputs(again)
    far = [k for k in a if not _close(a[k], b[k], k)]
    assert not far, far
    for k in a:
        assert np.array_equal(a[k], c[k]), k
    ref = oracle_full(lay, t)
    errs = {"Y": rel_err(a["Y"], ref["Y"]), "dX": rel_err(a["dX"], ref["dX"])}
    for i in range(T):
        errs[f"dW1_{i}"] = rel_err(a[f"dW1_{i}"], ref["dW1"][i])
        errs[f"dW2_{i}"] = rel_err(a[f"dW2_{i}"], ref["dW2"][i])
    bad = {k: v for k, v in errs.items() if not v <= 1e-2}
    assert not bad, bad


def test_linear_backward_tail_split(tp):
    """tp_linear_col_bwd and tp_linear_row_bwd (no activation) with their
    dgrad and weight-gradient GEMMs split, against the oracle and unsplit."""
    M, H, F, T = 1024, 768, 4096, 8
    Fs = F // T
    t = mlp_inputs(M, H, F, T, "none", "bf16", has_bias=True)
    col = tp.Layout(S=M // 2, B=2, H=H, F=F, T=T, act="none", dtype="bf16", has_bias=True)
    row = tp.Layout(S=M // 2, B=2, H=H, F=F, T=T, act="none", dtype="bf16", has_bias=True)
    d = lambda a: torch.from_numpy(np.ascontiguousarray(a, np.float32)).to("cuda", torch.bfloat16)
    X, dY = d(t["X"]), d(t["dY"])
    W1 = [d(w) for w in t["W1s"]]
    W2 = [d(w) for w in t["W2s"]]
    A = [d(a) for a in oracle.shard_row_weight(t["dY"] @ t["W2"], T)]  # any [M, Fs] activations
    dO = [d(a) for a in oracle.shard_row_weight(t["X"] @ t["W1"].T, T)]  # any [M, Fs] upstream grads
    results = []
    for split in (True, False, True):
        tp.set_tail_split(split)
        tp.set_max_gemm_pairs(11)
        ws = tp.alloc_workspace(tp.linear_workspace_bytes(col))
        f32 = dict(dtype=torch.float32, device="cuda")
        dXc = torch.empty(M, H, dtype=torch.bfloat16, device="cuda")
        dWc = [torch.empty(Fs, H, **f32) for _ in range(T)]
        dbc = [torch.empty(Fs, **f32) for _ in range(T)]
        dXr = [torch.empty(M, Fs, dtype=torch.bfloat16, device="cuda") for _ in range(T)]
        dWr = [torch.empty(H, Fs, **f32) for _ in range(T)]
        dbr = torch.empty(H, **f32)
        n0 = tp.tail_split_count()
        tp.linear_col_bwd(col, dO, [X], W1, [dXc], dWc, dbc, workspace=ws)
        tp.linear_row_bwd(row, [dY], A, W2, dXr, dWr, dbr, workspace=ws)
        assert tp.sync_status() == 0
        results.append(([host(dXc)] + [host(x) for x in dWc + dXr + dWr], tp.tail_split_count() - n0))
    (s, ns), (p, np_), (s2, _) = results
    assert ns >= 3 and np_ == 0, (ns, np_)
    bf16_out = [True] + [False] * T + [True] * T + [False] * T  # dX_col, dW_col, dX_row, dW_row
    for i, (a, b, c) in enumerate(zip(s, p, s2)):
        assert np.array_equal(a, c), i
        assert rel_err(a, b.astype(np.float64)) <= (2.0 ** -7 if bf16_out[i] else 1e-5), i
    # against the oracle
    dOn = [np.asarray(host(x), np.float64) for x in dO]
    An = [np.asarray(host(x), np.float64) for x in A]
    dXr_ref, dWc_ref, _ = oracle.column_bwd(dOn, t["X"], t["W1s"])
    dZ_ref, dWr_ref, _ = oracle.row_bwd(t["dY"], An, t["W2s"])
    assert rel_err(s[0], dXr_ref) <= 1e-2
    for i in range(T):
        assert rel_err(s[1 + i], dWc_ref[i]) <= 1e-2
        assert rel_err(s[1 + T + i], dZ_ref[i]) <= 1e-2
        assert rel_err(s[1 + 2 * T + i], dWr_ref[i]) <= 1e-2


def test_layer_tail_split_with_dropout(tp):
    """The sub-block (LayerNorm, MLP, dropout + residual) with the split,
    against the layer oracle and against itself unsplit."""
    from oracle import layer as olayer
    from test_gpu_layer import SEED, LayerRun, _p32, layer_inputs
    M, H, F, T, p = 1024, 768, 4096, 8, 0.1
    t = layer_inputs(M, H, F, T, "gelu_tanh", "bf16", True)
    runs = []
    for split in (True, False):
        tp.set_tail_split(split)
        tp.set_max_gemm_pairs(11)
        lay = tp.TPLayer(S=M // 2, B=2, H=H, F=F, T=T, act="gelu_tanh", dtype="bf16", has_bias=True, dropout_p=p)
        run = LayerRun(lay, t)
        n0 = tp.tail_split_count()
        run.fwd(SEED)
        run.bwd(SEED)
        assert status_ok(tp, lay)
        runs.append((run, tp.tail_split_count() - n0))
    (a, na), (b, nb) = runs
    assert na >= 4 and nb == 0, (na, nb)
    assert rel_err(a.gathered(a.Y), b.gathered(b.Y).astype(np.float64)) <= 2.0 ** -7
    assert rel_err(a.gathered(a.dX), b.gathered(b.dX).astype(np.float64)) <= 2.0 ** -7
    f = olayer.layer_fwd(t["X"], t["gamma"], t["beta"], t["W1s"], t["b1s"], t["W2s"], t["b2"], "gelu_tanh",
                         _p32(p), SEED)
    gr = olayer.layer_bwd(t["dY"], t["X"], t["gamma"], t["W1s"], t["W2s"], f, "gelu_tanh", _p32(p))
    errs = {"Y": rel_err(a.gathered(a.Y), f["Y"]), "dX": rel_err(a.gathered(a.dX), gr["dX"]),
            "dgamma": rel_err(host(a.dgamma), gr["dgamma"])}
    for i in range(T):
        errs[f"dW1_{i}"] = rel_err(host(a.dW1[i]), gr["dW1"][i])
        errs[f"dW2_{i}"] = rel_err(host(a.dW2[i]), gr["dW2"][i])
    bad = {k: v for k, v in errs.items() if not v <= 1e-2}
    assert not bad, bad


def test_fp8_tail_split_matches_unsplit(tp):
    """FP8 (current scaling): the split GEMMs dequantise the summed units like
    a whole tile; outputs agree with the unsplit run to fp32 reassociation."""
    M, H, F, T = 1024, 768, 4096, 8
    t = mlp_inputs(M, H, F, T, "gelu_tanh", "bf16", has_bias=True)
    outs = []
    for split in (True, False):
        lay = tp.TPMLP(S=M // 2, B=2, H=H, F=F, T=T, act="gelu_tanh", dtype="fp8", has_bias=True, residual=True)
        run, n = _step(tp, lay, t, split, 11)
        outs.append((_outputs(run), n))
    (a, na), (b, nb) = outs
    assert na >= 4 and nb == 0, (na, nb)
    far = [k for k in a if not _close(a[k], b[k], k)]
    assert not far, far


def test_tail_split_needs_its_scratch(tp):
    """A workspace without the tail scratch (the size before it) is accepted
    and the GEMMs run unsplit; the plain tp_mlp_fwd never splits."""
    M, H, F, T = 1024, 768, 4096, 8
    t = mlp_inputs(M, H, F, T, "gelu_tanh", "bf16", has_bias=True)
    tp.set_tail_split(False)
    tp.set_max_gemm_pairs(11)
    lay = tp.TPMLP(S=M // 2, B=2, H=H, F=F, T=T, act="gelu_tanh", dtype="bf16", has_bias=True, residual=True)
    core = lay.workspace_bytes()
    tp.set_tail_split(True)
    assert lay.workspace_bytes() > core
    run = MlpRun(lay, t)
    run.ws = tp.alloc_workspace(core)
    n0 = tp.tail_split_count()
    run.fwd()
    run.bwd()
    run.fwd(with_workspace=False)
    assert status_ok(tp, lay)
    assert tp.tail_split_count() == n0
    ref = oracle_full(lay, t)
    assert rel_err(run.gathered(run.Y), ref["Y"]) <= 1e-2
    assert rel_err(run.gathered(run.dX), ref["dX"]) <= 1e-2
    tp.set_max_gemm_pairs(0)


def test_tail_split_weight_gradient_accumulation(tp):
    """wgrad_accumulate through the split weight gradients: the fixup adds the
    units' sum into dW once (bulk reduce-add), so two accumulating backward
    calls from zero give exactly twice one call."""
    M, H, F, T = 1024, 768, 4096, 8
    t = mlp_inputs(M, H, F, T, "gelu_tanh", "bf16", has_bias=True)
    tp.set_tail_split(True)
    tp.set_max_gemm_pairs(11)
    lay = tp.TPMLP(S=M // 2, B=2, H=H, F=F, T=T, act="gelu_tanh", dtype="bf16", has_bias=True, residual=True,
                   wgrad_accumulate=True)
    run = MlpRun(lay, t)
    run.fwd()
    for d in run.dW1 + run.dW2:
        d.zero_()
    n0 = tp.tail_split_count()
    run.bwd()
    once = [d.clone() for d in run.dW1 + run.dW2]
    run.bwd()
    assert status_ok(tp, lay)
    assert tp.tail_split_count() - n0 >= 4
    for a, b in zip(once, run.dW1 + run.dW2):
        assert torch.equal(2 * a, b)
    ref = oracle_full(lay, t)
    for i in range(T):
        assert rel_err(host(once[i]), ref["dW1"][i]) <= 1e-2
        assert rel_err(host(once[T + i]), ref["dW2"][i]) <= 1e-2
    tp.set_max_gemm_pairs(0)


@pytest.mark.parametrize("sp", [False, True])
def test_alternate_k_order_matches_oracle_and_forward_order(tp, sp):
    """The pair GEMMs walk K backwards in every other persistent round
    (tp_set_k_order): with the grid cut to 7 pairs the row forward, column
    dgrad and both weight gradients run several rounds, so odd rounds take
    the reversed order.  Against the oracle, against the forward-only order
    (fp32 reassociation: 1e-5 for fp32 outputs, one bf16 step for bf16
    ones), and run to run bit for bit; under sequence parallelism the
    weight gradients' token-shard cursor walks backwards across shards."""
    M, H, F, T = 1024, 512, 2048, 4
    lay = tp.TPMLP(S=M // 2, B=2, H=H, F=F, T=T, act="gelu_tanh", dtype="bf16", has_bias=True, residual=not sp,
                   seq_parallel=sp)
    t = mlp_inputs(M, H, F, T, "gelu_tanh", "bf16", has_bias=True)
    outs = []
    try:
        for alternate in (True, False, True):
            tp.set_k_order(alternate)
            run, _ = _step(tp, lay, t, False, 7)
            outs.append(_outputs(run))
    finally:
        tp.set_k_order(True)
    a, b, c = outs
    far = [k for k in a if not _close(a[k], b[k], k)]
    assert not far, far
    for k in a:
        assert np.array_equal(a[k], c[k]), k
    assert any(not np.array_equal(a[k], b[k]) for k in a)  # the reversed rounds did run
    ref = oracle_full(lay, t)
    errs = {"Y": rel_err(a["Y"], ref["Y"]), "dX": rel_err(a["dX"], ref["dX"])}
    for i in range(T):
        errs[f"dW1_{i}"] = rel_err(a[f"dW1_{i}"], ref["dW1"][i])
        errs[f"dW2_{i}"] = rel_err(a[f"dW2_{i}"], ref["dW2"][i])
    bad = {k: v for k, v in errs.items() if not v <= 1e-2}
    assert not bad, bad


@pytest.mark.parametrize("band", [1, 3, 64])
def test_band_rows_match_oracle(tp, band):
    """Any band height of the pair GEMMs' tile order (tp_set_band_rows),
    including one taller than the problem and one that does not divide the
    row tiles, covers every output tile once: parity with the oracle over
    several persistent rounds (grid cut to 7 pairs)."""
    M, H, F, T = 1800, 512, 2048, 4
    lay = tp.TPMLP(S=M // 2, B=2, H=H, F=F, T=T, act="gelu_tanh", dtype="bf16", has_bias=True, residual=True)
    t = mlp_inputs(M, H, F, T, "gelu_tanh", "bf16", has_bias=True)
    try:
        tp.set_band_rows(band)
        run, _ = _step(tp, lay, t, True, 7)
    finally:
        tp.set_band_rows(0)
    a = _outputs(run)
    ref = oracle_full(lay, t)
    errs = {"Y": rel_err(a["Y"], ref["Y"]), "dX": rel_err(a["dX"], ref["dX"])}
    for i in range(T):
        errs[f"dW1_{i}"] = rel_err(a[f"dW1_{i}"], ref["dW1"][i])
        errs[f"dW2_{i}"] = rel_err(a[f"dW2_{i}"], ref["dW2"][i])
        errs[f"db1_{i}"] = rel_err(a[f"db1_{i}"], ref["db1"][i])
    bad = {k: v for k, v in errs.items() if not v <= 1e-2}
    assert not bad, bad


@pytest.mark.parametrize("sp,H", [(False, 512), (True, 512), (False, 256)])
def test_launch_overlap_keeps_stream_order(tp, sp, H):
    """Programmatic dependent launch of the pair GEMMs (tp_set_launch_overlap):
    two forward+backward steps on different inputs, issued back to back with
    no host synchronisation and sharing the pre, A and workspace buffers, so
    that a GEMM reading an operand before the kernel producing it finished
    (the row forward's A, the dgrads' dPre) or overwriting a buffer a GEMM
    before it still reads (the second column forward's pre and A under the
    first backward) would change the results.  Both steps give the bits of
    plain stream order and match the oracle; the grid cut to 7 pairs gives
    several persistent rounds and a tail split.  At H = 256 the forward is the
    fused kernel, also launched with programmatic dependent launch."""
    M, F, T = 1024, 2048, 4
    lay = tp.TPMLP(S=M // 2, B=2, H=H, F=F, T=T, act="gelu_tanh", dtype="bf16", has_bias=True, residual=not sp,
                   seq_parallel=sp)
    ins = [mlp_inputs(M, H, F, T, "gelu_tanh", "bf16", has_bias=True, seed_off=k) for k in (0, 1)]
    res = {}
    try:
        for on in (False, True, True):
            tp.set_launch_overlap(on)
            tp.set_max_gemm_pairs(7)
            runs = [MlpRun(lay, t) for t in ins]
            runs[1].pre, runs[1].A, runs[1].ws = runs[0].pre, runs[0].A, runs[0].ws
            torch.cuda.synchronize()
            for r in runs:
                r.fwd()
                r.bwd()
            assert status_ok(tp, lay)
            res.setdefault(on, []).append([_outputs(r) for r in runs])
    finally:
        tp.set_launch_overlap(True)
        tp.set_max_gemm_pairs(0)
    plain = res[False][0]
    for got in res[True]:
        for k in (0, 1):
            for name in plain[k]:
                assert np.array_equal(plain[k][name], got[k][name]), (k, name)
    for k in (0, 1):
        ref = oracle_full(lay, ins[k])
        a = plain[k]
        errs = {"Y": rel_err(a["Y"], ref["Y"]), "dX": rel_err(a["dX"], ref["dX"])}
        for i in range(T):
            errs[f"dW1_{i}"] = rel_err(a[f"dW1_{i}"], ref["dW1"][i])
            errs[f"dW2_{i}"] = rel_err(a[f"dW2_{i}"], ref["dW2"][i])
        bad = {n: v for n, v in errs.items() if not v <= 1e-2}
        assert not bad, (k, bad)
