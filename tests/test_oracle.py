"""Pins of the CPU oracle against facts fixed outside it (no GPU).

Each test pins the oracle to something other than itself:
  * torch fp64 autograd of an unsharded MLP written with library routines
    (F.linear, F.gelu(approximate='tanh'), F.silu): an independent forward and
    an independent (automatic) backward;
  * central finite differences of <dY, Y> (backward formulas, no torch);
  * sharded == unsharded for every T (the pages' claim that the Column/Row
    pairing computes the plain MLP, "Megatron-LM 源码精读" s3.3);
  * no forward reduction in the column layer and no backward reduction in the
    row layer (same page, s3.1 / s3.2);
  * sequence parallelism changes storage, not the result (same page s3.5;
    walk-through s06);
  * closed forms of the activations and the GeLU-tanh error bound against the
    exact erf GeLU.
"""
import math

import numpy as np
import pytest
import torch
import torch.nn.functional as F

import oracle
import synth


def _inputs(M, H, Fw, T, act, bias=True, seed=7, wstd=0.3):
    g = 2 if act == "swiglu" else 1
    rng = np.random.default_rng(seed)
    X = rng.standard_normal((M, H))
    W1 = rng.standard_normal((g * Fw, H)) * wstd
    W2 = rng.standard_normal((H, Fw)) * wstd
    b1 = rng.standard_normal(g * Fw) * 0.1 if bias else None
    b2 = rng.standard_normal(H) * 0.1 if bias else None
    dY = rng.standard_normal((M, H))
    W1s = oracle.shard_column_weight(W1, T, act)
    b1s = oracle.shard_column_bias(b1, T, act)
    W2s = oracle.shard_row_weight(W2, T)
    return dict(X=X, W1=W1, W2=W2, b1=b1, b2=b2, dY=dY, W1s=W1s, b1s=b1s, W2s=W2s)


def _torch_mlp(X, W1, b1, W2, b2, dY, act, residual):
    t = lambda a: None if a is None else torch.tensor(a, dtype=torch.float64, requires_grad=True)
    Xt, W1t, b1t, W2t, b2t = t(X), t(W1), t(b1), t(W2), t(b2)
    pre = F.linear(Xt, W1t, b1t)
    if act == "gelu_tanh":
        A = F.gelu(pre, approximate="tanh")
    elif act == "swiglu":
        Gt, Ut = pre.chunk(2, dim=1)
        A = F.silu(Gt) * Ut
    else:
        A = pre
    Y = F.linear(A, W2t, b2t)
    if residual:
        Y = Y + Xt
    (Y * torch.tensor(dY)).sum().backward()
    g = lambda a: None if a is None else a.grad.numpy()
    return dict(Y=Y.detach().numpy(), dX=g(Xt), dW1=g(W1t), db1=g(b1t), dW2=g(W2t), db2=g(b2t))


def _rel(a, b):
    a = np.asarray(a, np.float64)
    b = np.asarray(b, np.float64)
    return float(np.max(np.abs(a - b)) / max(np.max(np.abs(b)), 1e-300))


@pytest.mark.parametrize("act", ["gelu_tanh", "swiglu", "none"])
@pytest.mark.parametrize("T", [1, 2, 4])
@pytest.mark.parametrize("residual", [False, True])
def test_matches_torch_autograd(act, T, residual):
    d = _inputs(M=12, H=16, Fw=32, T=T, act=act)
    ref = _torch_mlp(d["X"], d["W1"], d["b1"], d["W2"], d["b2"], d["dY"], act, residual)
    pre, A, Y = oracle.mlp_fwd(d["X"], d["W1s"], d["b1s"], d["W2s"], d["b2"], act, residual)
    g = oracle.mlp_bwd(d["dY"], d["X"], d["W1s"], d["W2s"], pre, A, act, residual)
    assert _rel(Y, ref["Y"]) < 1e-13
    assert _rel(g["dX"], ref["dX"]) < 1e-13
    assert _rel(oracle.unshard_column(g["dW1"], act), ref["dW1"]) < 1e-13
    assert _rel(oracle.unshard_column(g["db1"], act), ref["db1"]) < 1e-13
    assert _rel(np.concatenate(g["dW2"], axis=1), ref["dW2"]) < 1e-13
    assert _rel(g["db2"], ref["db2"]) < 1e-13


@pytest.mark.parametrize("act", ["gelu_tanh", "swiglu"])
@pytest.mark.parametrize("T", [1, 2, 4])
@pytest.mark.parametrize("residual", [False, True])
def test_finite_differences(act, T, residual):
    # S=4, B=2 -> M=8 tokens, H=8, F=32
    d = _inputs(M=8, H=8, Fw=32, T=T, act=act, seed=11)
    pre, A, Y = oracle.mlp_fwd(d["X"], d["W1s"], d["b1s"], d["W2s"], d["b2"], act, residual)
    g = oracle.mlp_bwd(d["dY"], d["X"], d["W1s"], d["W2s"], pre, A, act, residual)
    rng = np.random.default_rng(3)
    h = 1e-6

    def loss():
        return oracle.mlp_loss(d["X"], d["W1s"], d["b1s"], d["W2s"], d["b2"], d["dY"], act, residual)

    def check(arr, grad, n=6):
        for _ in range(n):
            idx = tuple(int(rng.integers(0, s)) for s in arr.shape)
            old = arr[idx]
            arr[idx] = old + h
            lp = loss()
            arr[idx] = old - h
            lm = loss()
            arr[idx] = old
            fd = (lp - lm) / (2 * h)
            assert abs(fd - grad[idx]) <= 1e-6 * max(1.0, abs(grad[idx])), (idx, fd, grad[idx])

    check(d["X"], g["dX"])
    for i in range(T):
        check(d["W1s"][i], g["dW1"][i], 3)
        check(d["b1s"][i], g["db1"][i], 2)
        check(d["W2s"][i], g["dW2"][i], 3)
    check(d["b2"], g["db2"])


@pytest.mark.parametrize("act", ["gelu_tanh", "swiglu", "none"])
def test_sharded_equals_unsharded(act):
    Fw = 64
    base = _inputs(M=10, H=24, Fw=Fw, T=1, act=act, seed=5)
    pre1, A1, Y1 = oracle.mlp_fwd(base["X"], base["W1s"], base["b1s"], base["W2s"], base["b2"], act, True)
    g1 = oracle.mlp_bwd(base["dY"], base["X"], base["W1s"], base["W2s"], pre1, A1, act, True)
    for T in (2, 4, 8):
        W1s = oracle.shard_column_weight(base["W1"], T, act)
        b1s = oracle.shard_column_bias(base["b1"], T, act)
        W2s = oracle.shard_row_weight(base["W2"], T)
        pre, A, Y = oracle.mlp_fwd(base["X"], W1s, b1s, W2s, base["b2"], act, True)
        g = oracle.mlp_bwd(base["dY"], base["X"], W1s, W2s, pre, A, act, True)
        assert _rel(Y, Y1) < 1e-12
        assert _rel(g["dX"], g1["dX"]) < 1e-12
        assert _rel(oracle.unshard_column(g["dW1"], act), g1["dW1"][0]) < 1e-12
        assert _rel(oracle.unshard_column(g["db1"], act), g1["db1"][0]) < 1e-12
        assert _rel(np.concatenate(g["dW2"], axis=1), g1["dW2"][0]) < 1e-12
        assert _rel(g["db2"], g1["db2"]) < 1e-12
        # the activation of shard i is the column block i of the unsharded one
        fs = Fw // T
        for i in range(T):
            assert _rel(A[i], A1[0][:, i * fs:(i + 1) * fs]) < 1e-12


def test_column_needs_no_forward_reduction():
    d = _inputs(M=6, H=16, Fw=32, T=4, act="gelu_tanh")
    pre, A, _ = oracle.mlp_fwd(d["X"], d["W1s"], d["b1s"], d["W2s"], d["b2"], "gelu_tanh", False)
    for j in range(4):
        W1s = [w.copy() for w in d["W1s"]]
        b1s = [b.copy() for b in d["b1s"]]
        W1s[j] += 1.0
        b1s[j] -= 0.5
        pre2, A2, _ = oracle.mlp_fwd(d["X"], W1s, b1s, d["W2s"], d["b2"], "gelu_tanh", False)
        for i in range(4):
            if i != j:
                assert np.array_equal(pre[i], pre2[i]) and np.array_equal(A[i], A2[i])
            else:
                assert not np.array_equal(pre[i], pre2[i])


@pytest.mark.parametrize("act", ["gelu_tanh", "swiglu"])
def test_row_needs_no_backward_reduction(act):
    d = _inputs(M=6, H=16, Fw=32, T=4, act=act)
    pre, A, _ = oracle.mlp_fwd(d["X"], d["W1s"], d["b1s"], d["W2s"], d["b2"], act, False)
    g = oracle.mlp_bwd(d["dY"], d["X"], d["W1s"], d["W2s"], pre, A, act, False)
    for j in range(4):
        W2s = [w.copy() for w in d["W2s"]]
        W2s[j] *= -2.0
        g2 = oracle.mlp_bwd(d["dY"], d["X"], d["W1s"], W2s, pre, A, act, False)
        for i in range(4):
            same = i != j
            assert np.array_equal(g["dA"][i], g2["dA"][i]) == same
            assert np.array_equal(g["dPre"][i], g2["dPre"][i]) == same
            # dW2_i depends on A_i and dY only
            assert np.array_equal(g["dW2"][i], g2["dW2"][i])
        assert not np.array_equal(g["dX"], g2["dX"])


def test_sequence_parallel_changes_storage_only():
    T = 4
    d = _inputs(M=16, H=8, Fw=16, T=T, act="gelu_tanh")
    shards = oracle.sp_split(d["X"], T)
    assert all(s.shape == (4, 8) for s in shards)
    X = oracle.sp_gather(shards)
    assert np.array_equal(X, d["X"])
    pre, A, Y = oracle.mlp_fwd(X, d["W1s"], d["b1s"], d["W2s"], d["b2"], "gelu_tanh", True)
    pre0, A0, Y0 = oracle.mlp_fwd(d["X"], d["W1s"], d["b1s"], d["W2s"], d["b2"], "gelu_tanh", True)
    Ys = oracle.sp_split(Y, T)
    for j in range(T):
        assert np.array_equal(Ys[j], Y0[j * 4:(j + 1) * 4])


def test_divide_contract():
    assert oracle.divide(16384, 8) == 2048
    with pytest.raises(ValueError):
        oracle.divide(1000, 3)
    with pytest.raises(ValueError):
        oracle.shard_column_weight(np.zeros((10, 4)), 4)
    with pytest.raises(ValueError):
        oracle.shard_row_weight(np.zeros((4, 10)), 4)


def test_activation_closed_forms():
    x = np.array([0.0])
    assert oracle.gelu_tanh(x)[0] == 0.0
    assert oracle.gelu_tanh_grad(x)[0] == 0.5
    assert oracle.silu(x)[0] == 0.0
    # saturation: tanh -> +-1 so gelu -> x and 0; derivative -> 1 and 0
    big = np.array([12.0, -12.0])
    assert abs(oracle.gelu_tanh(big)[0] - 12.0) < 1e-12 and abs(oracle.gelu_tanh(big)[1]) < 1e-12
    assert abs(oracle.gelu_tanh_grad(big)[0] - 1.0) < 1e-12 and abs(oracle.gelu_tanh_grad(big)[1]) < 1e-12
    # sigmoid(0) = 1/2 so d/dx SiLU at 0 is 1/2: checked through the SwiGLU backward
    pre = np.array([[0.0, 3.0]])  # G = 0, U = 3
    dPre = oracle.act_bwd(pre, np.array([[1.0]]), "swiglu")
    assert dPre[0, 0] == 1.5 and dPre[0, 1] == 0.0
    # GeLU-tanh approximates x * Phi(x); the two differ by well under 1e-3
    xs = np.linspace(-6, 6, 2401)
    exact = np.array([0.5 * v * (1 + math.erf(v / math.sqrt(2))) for v in xs])
    err = np.max(np.abs(oracle.gelu_tanh(xs) - exact))
    assert 1e-5 < err < 1e-3


def test_activations_match_torch():
    xs = np.linspace(-8, 8, 1001)
    t = torch.tensor(xs, dtype=torch.float64, requires_grad=True)
    y = F.gelu(t, approximate="tanh")
    y.sum().backward()
    assert np.max(np.abs(oracle.gelu_tanh(xs) - y.detach().numpy())) < 1e-15
    assert np.max(np.abs(oracle.gelu_tanh_grad(xs) - t.grad.numpy())) < 1e-14
    assert np.max(np.abs(oracle.silu(xs) - F.silu(torch.tensor(xs)).numpy())) < 1e-15


@pytest.mark.parametrize("act", ["gelu_tanh", "swiglu"])
def test_sampled_evaluation_agrees_with_full(act):
    T = 2
    d = _inputs(M=20, H=16, Fw=32, T=T, act=act)
    pre, A, Y = oracle.mlp_fwd(d["X"], d["W1s"], d["b1s"], d["W2s"], d["b2"], act, True)
    g = oracle.mlp_bwd(d["dY"], d["X"], d["W1s"], d["W2s"], pre, A, act, True)
    rows = np.array([0, 7, 19])
    r = oracle.mlp_rows(rows, d["X"], d["W1s"], d["b1s"], d["W2s"], d["b2"], d["dY"], act, True)
    assert _rel(r["Y"], Y[rows]) < 1e-14
    assert _rel(r["dX"], g["dX"][rows]) < 1e-14
    units = [np.array([0, 5, 15]), np.array([3, 15])]
    u = oracle.mlp_units(units, d["X"], d["W1s"], d["b1s"], d["W2s"], d["dY"], act)
    fs = 16
    for i in range(T):
        sel = np.concatenate([units[i], fs + units[i]]) if act == "swiglu" else units[i]
        assert _rel(u["dW1"][i], g["dW1"][i][sel]) < 1e-13
        assert _rel(u["db1"][i], g["db1"][i][sel]) < 1e-13
        assert _rel(u["dW2"][i], g["dW2"][i][:, units[i]]) < 1e-13


def test_hand_computed_example():
    """A 1-token, H=2, F=2, T=2 MLP with no activation, worked by hand:
    X = [1, 2]; W1 = [[1, 0], [1, 1]] (shard 0 = row 0, shard 1 = row 1);
    W2 = [[2, 3], [0, 1]] (shard 0 = column 0, shard 1 = column 1).
    pre_0 = 1, pre_1 = 3; partial Y_0 = pre_0 * [2, 0] = [2, 0],
    Y_1 = pre_1 * [3, 1] = [9, 3]; Y = [11, 3].  With dY = [1, 1]:
    dA_0 = 2, dA_1 = 4; dX = 2*[1, 0] + 4*[1, 1] = [6, 4]."""
    X = np.array([[1.0, 2.0]])
    W1 = np.array([[1.0, 0.0], [1.0, 1.0]])
    W2 = np.array([[2.0, 3.0], [0.0, 1.0]])
    W1s = oracle.shard_column_weight(W1, 2)
    W2s = oracle.shard_row_weight(W2, 2)
    pre, A, Y = oracle.mlp_fwd(X, W1s, None, W2s, None, "none", False)
    assert pre[0][0, 0] == 1.0 and pre[1][0, 0] == 3.0
    assert np.array_equal(Y, [[11.0, 3.0]])
    g = oracle.mlp_bwd(np.array([[1.0, 1.0]]), X, W1s, W2s, pre, A, "none", False)
    assert np.array_equal(g["dX"], [[6.0, 4.0]])
    assert np.array_equal(g["dW2"][0], [[1.0], [1.0]])
    assert np.array_equal(g["dW1"][1], [[4.0, 8.0]])


def test_synth_generator_statistics():
    a = synth.normal(synth.SEED_BASE + 99, (1 << 20,))
    assert abs(a.mean()) < 5e-3 and abs(a.std() - 1.0) < 5e-3
    assert np.array_equal(synth.normal(5, (8,), offset=100), synth.normal(5, (108,))[100:])
    b = synth.round_bf16(a)
    # bf16 keeps 8 significant bits: relative rounding error <= half an ulp = 2^-8
    nz = a != 0
    assert np.max(np.abs(b[nz] - a[nz]) / np.abs(a[nz])) <= 2.0 ** -8
