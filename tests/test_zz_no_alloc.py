"""The allocation-free row-layer backward (tp_linear_row_bwd_noalloc).

Some callers cannot allocate device memory when they call: a plugin that is
handed only the op's tensors, a process whose device memory belongs to another
allocator, a latency-critical loop that cannot take cudaMalloc's implicit
synchronisation.  For them the library's scratch comes from a fixed 4 MiB
array compiled into it.  The entry point has two regimes, and each test below
first checks which one its shape falls in:

- the whole single-layer workspace fits in the array: the call runs the plan
  of tp_linear_row_bwd with a caller workspace, so the two agree bit for bit;
- it does not: the weight gradient runs without token or tail splitting and
  the array holds only the bias partials (4 * ceil(M/256) * H bytes), which
  must fit even when the layer's split width F is far larger than H.

Every result is compared with the fp64 oracle and with tp_linear_row_bwd.  The
calls come in sequences -- a larger problem, then a smaller one, with and
without a bias -- so that a call reading scratch an earlier call left behind
would show.  The file sorts last so that a run stopping at the first failure
has already run every other test.
"""
import numpy as np
import pytest
import torch

import oracle
import synth
from harness import TOL, host, rel_err

pytestmark = pytest.mark.gpu

SCRATCH = 4 << 20  # bytes of the library's built-in array


@pytest.fixture(scope="module")
def tp():
    import tensor_transformer_mlp_shard_gb300 as tp
    from tensor_transformer_mlp_shard_gb300 import build
    build.build()
    return tp


def _inputs(lay, seed):
    """Seeded bf16 inputs on the host (fp32 arrays holding bf16 values) and
    their device copies: dY [M, H] (token shards under sequence parallelism),
    X_i [M, Fs] and W_i [H, Fs]."""
    base = synth.SEED_BASE + 5000 + 10 * seed
    dY = synth.round_bf16(synth.normal(base, (lay.M, lay.H)))
    X = [synth.round_bf16(synth.normal(base + 1, (lay.M, lay.Fs), offset=i * lay.M * lay.Fs))
         for i in range(lay.T)]
    W = [synth.round_bf16(synth.normal(base + 2, (lay.H, lay.Fs), 0.02, offset=i * lay.H * lay.Fs))
         for i in range(lay.T)]
    up = lambda a: torch.from_numpy(np.ascontiguousarray(a)).to("cuda", torch.bfloat16)
    rows = lay.xrows
    d = {"dY": [up(dY[j * rows:(j + 1) * rows]) for j in range(lay.nx)], "X": [up(x) for x in X],
         "W": [up(w) for w in W]}
    return {"dY": dY, "X": X, "W": W}, d


def _outputs(lay):
    bf, f32 = dict(dtype=torch.bfloat16, device="cuda"), dict(dtype=torch.float32, device="cuda")
    nan = float("nan")
    return ([torch.full((lay.M, lay.Fs), nan, **bf) for _ in range(lay.T)],
            [torch.full((lay.H, lay.Fs), nan, **f32) for _ in range(lay.T)],
            torch.full((lay.H,), nan, **f32) if lay.has_bias else None)


def _run_both(tp, lay, d):
    """The allocation-free call and tp_linear_row_bwd with a caller
    workspace, on the same device inputs."""
    ref = _outputs(lay)
    ws = tp.alloc_workspace(tp.linear_workspace_bytes(lay))
    tp.linear_row_bwd(lay, d["dY"], d["X"], d["W"], *ref, ws)
    out = _outputs(lay)
    tp.linear_row_bwd_noalloc(lay, d["dY"], d["X"], d["W"], *out)
    assert tp.sync_status() == 0
    return out, ref


def _flat(res):
    dX, dW, db = res
    return [host(t) for t in dX + dW] + ([host(db)] if db is not None else [])


def _check_oracle(lay, h, res, cols=None):
    """Compare with the fp64 oracle's row backward (dX_i = dY W_i,
    dW_i = dY^T X_i, db = sum_m dY); with `cols`, on those split-width
    columns of every shard (each column of dX_i and dW_i depends on the same
    column of X_i and W_i only), db in full."""
    dX, dW, db = res
    Xs, Ws = h["X"], h["W"]
    if cols is not None:
        Xs, Ws = [x[:, cols] for x in Xs], [w[:, cols] for w in Ws]
    rdX, rdW, rdb = oracle.row_bwd(h["dY"], Xs, Ws)
    tol = TOL["bf16"]
    errs = {}
    for i in range(lay.T):
        gx, gw = host(dX[i]), host(dW[i])
        if cols is not None:
            gx, gw = gx[:, cols], gw[:, cols]
        errs[f"dX{i}"] = rel_err(gx, rdX[i])
        errs[f"dW{i}"] = rel_err(gw, rdW[i])
    if db is not None:
        errs["db"] = rel_err(host(db), rdb)
    bad = {k: v for k, v in errs.items() if not v <= tol}
    assert not bad, bad


def test_whole_workspace_fits_same_plan_bitwise(tp):
    """Both regimes' first: shapes whose whole workspace fits in the array
    (bias on and off, then a smaller problem after a larger one) give
    tp_linear_row_bwd's results bit for bit and match the oracle."""
    shapes = [dict(S=1024, B=2, H=256, F=512, T=2, has_bias=True),
              dict(S=1024, B=2, H=256, F=512, T=2, has_bias=False),
              dict(S=256, B=2, H=264, F=400, T=2, has_bias=True)]
    for k, sh in enumerate(shapes):
        lay = tp.Layout(act="none", dtype="bf16", **sh)
        assert tp.linear_workspace_bytes(lay) <= SCRATCH, sh
        h, d = _inputs(lay, k)
        out, ref = _run_both(tp, lay, d)
        for a, b in zip(_flat(out), _flat(ref)):
            assert np.array_equal(a, b), sh
        _check_oracle(lay, h, out)


@pytest.mark.parametrize("seq_parallel", [False, True])
def test_workspace_too_large_bias_partials_only(tp, seq_parallel):
    """Shapes whose workspace exceeds the array: the weight gradient runs
    unsplit and only the bias partials use the array.  Two calls in a row,
    with a bias and without."""
    for k, bias in enumerate((True, False)):
        lay = tp.Layout(S=512, B=2, H=520, F=1024, T=4, act="none", dtype="bf16", has_bias=bias,
                        seq_parallel=seq_parallel)
        assert tp.linear_workspace_bytes(lay) > SCRATCH
        h, d = _inputs(lay, 10 + k)
        out, ref = _run_both(tp, lay, d)
        for a, b in zip(_flat(out), _flat(ref)):
            assert rel_err(a, b) <= TOL["bf16"]
        _check_oracle(lay, h, out)


def test_wide_split_width_uses_only_the_row_bias_partials(tp):
    """F far above H: the bias partials of the row layer (4 * ceil(M/256) * H
    = 65 KB here) fit although the column layer's (4 * ceil(M/256) * F, over
    4 MiB) would not -- the row backward never needs those.  Checked against
    the oracle on sampled split-width columns, then a small problem runs
    after it on the same array."""
    lay = tp.Layout(S=8320, B=2, H=128, F=16384, T=4, act="none", dtype="bf16", has_bias=True)
    chunks = (lay.M + 255) // 256
    assert 4 * chunks * lay.H <= SCRATCH < 4 * chunks * lay.F
    assert tp.linear_workspace_bytes(lay) > SCRATCH
    h, d = _inputs(lay, 20)
    out, ref = _run_both(tp, lay, d)
    for a, b in zip(_flat(out), _flat(ref)):
        assert rel_err(a, b) <= TOL["bf16"]
    rng = np.random.default_rng(3)
    cols = np.unique(np.concatenate([[0, lay.Fs - 1], rng.choice(lay.Fs, 30, replace=False)]))
    _check_oracle(lay, h, out, cols)
    small = tp.Layout(S=256, B=2, H=264, F=400, T=2, act="none", dtype="bf16", has_bias=True)
    h2, d2 = _inputs(small, 21)
    out2, ref2 = _run_both(tp, small, d2)
    for a, b in zip(_flat(out2), _flat(ref2)):
        assert np.array_equal(a, b)
    _check_oracle(small, h2, out2)


def test_noalloc_rejects_oversized_scratch(tp):
    # bias partials: 4 * ceil(M/256) * H bytes; M = 65536, H = 8192 -> 8 MiB > 4 MiB
    lay = tp.Layout(S=65536, B=1, H=8192, F=64, T=8, act="none", dtype="bf16", has_bias=True)
    from tensor_transformer_mlp_shard_gb300.binding import TpError
    bf = dict(dtype=torch.bfloat16, device="cuda")
    with pytest.raises(TpError) as e:
        tp.linear_row_bwd_noalloc(lay, [torch.empty(lay.M, lay.H, **bf)],
                                  [torch.empty(lay.M, lay.Fs, **bf) for _ in range(lay.T)],
                                  [torch.empty(lay.H, lay.Fs, **bf) for _ in range(lay.T)],
                                  [torch.empty(lay.M, lay.Fs, **bf) for _ in range(lay.T)],
                                  [torch.empty(lay.H, lay.Fs, dtype=torch.float32, device="cuda")
                                   for _ in range(lay.T)],
                                  torch.empty(lay.H, dtype=torch.float32, device="cuda"))
    assert e.value.status == 3
    assert tp.sync_status() == 0
