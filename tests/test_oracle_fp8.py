"""Pins of the FP8 oracle (oracle/fp8.py) against torch's float8/bfloat16
casts (library routines), the formats' definitions and the plain fp64 oracle."""
import numpy as np
import pytest
import torch

import oracle
from oracle import fp8


def _torch_round(x, fmt):
    dt = torch.float8_e4m3fn if fmt == "e4m3" else torch.float8_e5m2
    return torch.tensor(x, dtype=torch.float32).to(dt).to(torch.float64).numpy()


@pytest.mark.parametrize("fmt", ["e4m3", "e5m2"])
def test_round_fp8_matches_torch_in_range(fmt):
    rng = np.random.default_rng(0)
    top = fp8.fmax(fmt)
    # log-uniform magnitudes over the whole range incl. subnormals, both signs
    mags = np.exp2(rng.uniform(np.log2(top) - 30, np.log2(top) + 0.0, 200000)).astype(np.float32)
    x = (mags * rng.choice([-1, 1], mags.size)).astype(np.float32)
    x = x[np.abs(x) <= top]
    assert np.array_equal(fp8.round_fp8(x, fmt), _torch_round(x, fmt))
    # every representable value and every midpoint between neighbours (ties)
    codes = torch.arange(256, dtype=torch.int32).to(torch.uint8)
    dt = torch.float8_e4m3fn if fmt == "e4m3" else torch.float8_e5m2
    vals = np.unique(codes.view(dt).to(torch.float64).numpy())
    vals = vals[np.isfinite(vals)]
    assert np.array_equal(fp8.round_fp8(vals, fmt), vals)
    pos = vals[vals >= 0]
    mids = ((pos[1:] + pos[:-1]) / 2).astype(np.float32)
    assert np.array_equal(fp8.round_fp8(mids, fmt), _torch_round(mids, fmt))


def test_format_definitions():
    assert fp8.round_fp8(np.array([1e6, -1e6]), "e4m3").tolist() == [448.0, -448.0]   # saturates
    assert fp8.round_fp8(np.array([460.0, 470.0]), "e4m3").tolist() == [448.0, 448.0]
    assert fp8.round_fp8(np.array([1e9]), "e5m2").tolist() == [57344.0]
    assert fp8.round_fp8(np.array([2.0 ** -9, 2.0 ** -10, 3 * 2.0 ** -11]), "e4m3").tolist() == \
        [2.0 ** -9, 0.0, 2.0 ** -9]
    assert fp8.round_fp8(np.array([2.0 ** -16, 2.0 ** -17]), "e5m2").tolist() == [2.0 ** -16, 0.0]
    assert fp8.round_fp8(np.array([1.0 + 2 ** -4, 1.0 + 3 * 2 ** -4]), "e4m3").tolist() == [1.0, 1.25]


def test_round_bf16_matches_torch():
    x = np.random.default_rng(1).standard_normal(100000).astype(np.float32) * 10
    assert np.array_equal(fp8.round_bf16(x), torch.tensor(x).to(torch.bfloat16).double().numpy())


def test_scale_maps_amax_to_fmax():
    x = np.random.default_rng(2).standard_normal((7, 9)).astype(np.float32)
    (q,), s = fp8.quantize([x], "e4m3")
    assert np.max(np.abs(q)) == 448.0
    assert s == np.float32(np.float32(448.0) / np.float32(np.max(np.abs(x))))
    (q0,), s0 = fp8.quantize([np.zeros((2, 2), np.float32)], "e5m2")
    assert s0 == 1.0 and not q0.any()
    # one scale across shards: the shard holding the amax reaches fmax, the other does not
    parts, s = fp8.quantize([x, x / 4], "e4m3")
    assert np.max(np.abs(parts[0])) == 448.0 and np.max(np.abs(parts[1])) <= 112.0


@pytest.mark.parametrize("act", ["gelu_tanh", "swiglu"])
def test_fp8_pipeline_close_to_exact_mlp(act):
    """The FP8 variant approximates the exact MLP within the formats' relative
    precision (E4M3 2^-4, E5M2 2^-3 per element); a transposed operand, an
    inverted scale or a missing term would be off by orders of magnitude."""
    rng = np.random.default_rng(3)
    M, H, F, T = 64, 96, 128, 4
    g = 2 if act == "swiglu" else 1
    X = fp8.round_bf16(rng.standard_normal((M, H)))
    W1 = fp8.round_bf16(rng.standard_normal((g * F, H)) * 0.1)
    W2 = fp8.round_bf16(rng.standard_normal((H, F)) * 0.1)
    b1 = fp8.round_bf16(rng.standard_normal(g * F) * 0.1)
    b2 = fp8.round_bf16(rng.standard_normal(H) * 0.1)
    dY = fp8.round_bf16(rng.standard_normal((M, H)))
    W1s = oracle.shard_column_weight(W1, T, act)
    b1s = oracle.shard_column_bias(b1, T, act)
    W2s = oracle.shard_row_weight(W2, T)
    f = fp8.mlp_fwd_fp8(X, W1s, b1s, W2s, b2, act, True)
    g8 = fp8.mlp_bwd_fp8(dY, f, act, True)
    pre, A, Y = oracle.mlp_fwd(X, W1s, b1s, W2s, b2, act, True)
    g64 = oracle.mlp_bwd(dY, X, W1s, W2s, pre, A, act, True)

    def rel(a, b):
        return np.max(np.abs(np.asarray(a) - np.asarray(b))) / np.max(np.abs(b))

    assert rel(f["Y"], Y) < 0.05
    assert rel(g8["dX"], g64["dX"]) < 0.1
    for i in range(T):
        assert rel(g8["dW1"][i], g64["dW1"][i]) < 0.15
        assert rel(g8["dW2"][i], g64["dW2"][i]) < 0.15
        assert rel(g8["db1"][i], g64["db1"][i]) < 0.1
    assert rel(g8["db2"], g64["db2"]) == 0.0


@pytest.mark.parametrize("act", ["gelu_tanh", "swiglu"])
def test_sampled_fp8_agrees_with_full(act):
    rng = np.random.default_rng(9)
    M, H, F, T = 40, 32, 64, 2
    g = 2 if act == "swiglu" else 1
    X = fp8.round_bf16(rng.standard_normal((M, H)))
    W1s = oracle.shard_column_weight(fp8.round_bf16(rng.standard_normal((g * F, H)) * 0.1), T, act)
    b1s = oracle.shard_column_bias(fp8.round_bf16(rng.standard_normal(g * F) * 0.1), T, act)
    W2s = oracle.shard_row_weight(fp8.round_bf16(rng.standard_normal((H, F)) * 0.1), T)
    b2 = fp8.round_bf16(rng.standard_normal(H) * 0.1)
    dY = fp8.round_bf16(rng.standard_normal((M, H)))
    f = fp8.mlp_fwd_fp8(X, W1s, b1s, W2s, b2, act, True)
    gr = fp8.mlp_bwd_fp8(dY, f, act, True)
    rows = np.array([0, 5, 39])
    units = [np.array([0, 31]), np.array([7])]
    s = fp8.mlp_sampled_fp8(rows, units, X, W1s, b1s, W2s, b2, dY, act, True)
    assert np.allclose(s["Y"], f["Y"][rows], rtol=0, atol=1e-12)
    assert np.allclose(s["dX"], gr["dX"][rows], rtol=0, atol=1e-12)
    assert np.array_equal(s["db2"], gr["db2"])
    fs = F // T
    for i in range(T):
        sel = np.concatenate([units[i], fs + units[i]]) if act == "swiglu" else units[i]
        assert np.allclose(s["dW1"][i], gr["dW1"][i][sel], rtol=0, atol=1e-12)
        assert np.allclose(s["dW2"][i], gr["dW2"][i][:, units[i]], rtol=0, atol=1e-12)
        assert np.allclose(s["db1"][i], gr["db1"][i][sel], rtol=0, atol=1e-12)


# ---- delayed scaling (F6: the pages' amax history) -------------------------

def test_amax_history_window_and_empty_history():
    h = fp8.AmaxHistory(3)
    assert h.amax_for("X", 7.0) == np.float32(7.0)  # empty history: the tensor's own amax
    for a in (1.0, 4.0, 2.0):
        h.record("X", a)
    assert h.amax_for("X", 100.0) == np.float32(4.0)  # max over the window, not the current amax
    h.record("X", 0.5)  # 1.0 leaves the window of 3
    assert h.hist["X"] == [np.float32(4.0), np.float32(2.0), np.float32(0.5)]
    h.record("X", 0.25)
    h.record("X", 0.125)  # 4.0 and 2.0 leave
    assert h.amax_for("X", 9.0) == np.float32(0.5)
    assert h.amax_for("W1", 3.0) == np.float32(3.0)  # tensors keep separate histories
    with pytest.raises(ValueError):
        fp8.AmaxHistory(0)


def test_history_of_one_scales_by_the_previous_step_and_saturates():
    rng = np.random.default_rng(3)
    x1 = rng.normal(size=(64, 32)).astype(np.float32)
    x2 = 2.0 * x1  # the tensor doubles between steps
    h = fp8.AmaxHistory(1)
    (q1,), s1 = fp8.quantize([x1], "e4m3", "X", h)
    (q2,), s2 = fp8.quantize([x2], "e4m3", "X", h)
    assert s1 == fp8.scale_of(fp8.amax_of([x1]), "e4m3")  # first step: current scaling
    assert s2 == s1  # second step: the first step's amax
    v = (x2 * s2).astype(np.float32)
    assert np.array_equal(q2, fp8.round_fp8(v, "e4m3"))
    # everything beyond fmax saturates to +-448; a current scale would have none
    assert np.count_nonzero(np.abs(q2) == 448.0) >= np.count_nonzero(np.abs(v) > 448.0) > 0
    assert h.hist["X"] == [fp8.amax_of([x2])]


def test_delayed_scaling_on_repeated_inputs_equals_current_scaling():
    """With the same tensors every step, the history's maximum is each
    tensor's own amax, so from the first step on delayed scaling reproduces
    current scaling exactly (and the first step always does)."""
    rng = np.random.default_rng(5)
    M, H, F, T = 48, 32, 64, 2
    X = fp8.round_bf16(rng.normal(size=(M, H)))
    W1s = [fp8.round_bf16(0.1 * rng.normal(size=(F // T, H))) for _ in range(T)]
    W2s = [fp8.round_bf16(0.1 * rng.normal(size=(H, F // T))) for _ in range(T)]
    b1s = [fp8.round_bf16(0.02 * rng.normal(size=F // T)) for _ in range(T)]
    b2 = fp8.round_bf16(0.02 * rng.normal(size=H))
    dY = fp8.round_bf16(rng.normal(size=(M, H)))
    ref = fp8.mlp_fwd_fp8(X, W1s, b1s, W2s, b2, "gelu_tanh", True)
    gref = fp8.mlp_bwd_fp8(dY, ref, "gelu_tanh", True)
    h = fp8.AmaxHistory(2)
    for _ in range(3):
        f = fp8.mlp_fwd_fp8(X, W1s, b1s, W2s, b2, "gelu_tanh", True, h)
        g = fp8.mlp_bwd_fp8(dY, f, "gelu_tanh", True, h)
        assert np.array_equal(f["Y"], ref["Y"]) and np.array_equal(g["dX"], gref["dX"])
        for a, b in zip(g["dW1"] + g["dW2"], gref["dW1"] + gref["dW2"]):
            assert np.array_equal(a, b)
    assert sorted(h.hist) == ["A", "W1", "W2", "X", "dPre", "dY"]
    assert all(len(v) == 2 for v in h.hist.values())


def _layer_inputs(seed, M=48, H=96, F=128, T=4):
    rng = np.random.default_rng(seed)
    r = lambda *s, sc=1.0: fp8.round_bf16(rng.standard_normal(s) * sc)
    return rng, r, M, H, F, T


def test_fp8_layers_close_to_exact_layers():
    """Each FP8 single layer approximates the exact fp64 layer within the
    formats' relative precision; a transposed operand, an inverted scale or a
    dropped term would be off by orders of magnitude."""
    _, r, M, H, F, T = _layer_inputs(5)
    Fs = F // T
    X, W, b = r(M, H), [r(Fs, H, sc=0.1) for _ in range(T)], [r(Fs, sc=0.1) for _ in range(T)]
    dO = [r(M, Fs) for _ in range(T)]
    Xr, W2, b2, R, dY = [r(M, Fs) for _ in range(T)], [r(H, Fs, sc=0.1) for _ in range(T)], r(H, sc=0.1), \
        r(M, H), r(M, H)

    def rel(a, b):
        return np.max(np.abs(np.asarray(a) - np.asarray(b))) / np.max(np.abs(b))

    for act in ("none", "gelu_tanh"):
        pre8, out8 = fp8.column_fwd_fp8(X, W, b, act)
        pre, out = oracle.column_fwd(X, W, b, act)
        for i in range(T):
            assert rel(pre8[i], pre[i]) < 0.05 and rel(out8[i], out[i]) < 0.05
    assert rel(fp8.row_fwd_fp8(Xr, W2, b2, R), oracle.row_fwd(Xr, W2, b2, R)) < 0.05
    dX8, dW8, db8 = fp8.column_bwd_fp8(dO, X, W)
    dX, dW, db = oracle.column_bwd(dO, X, W)
    assert rel(dX8, dX) < 0.1
    for i in range(T):
        assert rel(dW8[i], dW[i]) < 0.15 and rel(db8[i], db[i]) == 0.0
    rX8, rW8, rdb8 = fp8.row_bwd_fp8(dY, Xr, W2)
    rX, rW, rdb = oracle.row_bwd(dY, Xr, W2)
    for i in range(T):
        assert rel(rX8[i], rX[i]) < 0.1 and rel(rW8[i], rW[i]) < 0.15
    assert rel(rdb8, rdb) == 0.0


def test_fp8_layers_compose_to_the_fp8_mlp():
    """Column layer, activation and row layer in FP8, chained the way the MLP
    chains them (the row layer's input is the stored bf16 activation), give
    the FP8 MLP's outputs exactly; the row backward's dX_i is the MLP's dA_i
    before act', and its dW the MLP's dW2."""
    _, r, M, H, F, T = _layer_inputs(6)
    Fs = F // T
    X, dY = r(M, H), r(M, H)
    W1s = [r(Fs, H, sc=0.1) for _ in range(T)]
    b1s = [r(Fs, sc=0.1) for _ in range(T)]
    W2s = [r(H, Fs, sc=0.1) for _ in range(T)]
    b2 = r(H, sc=0.1)
    f = fp8.mlp_fwd_fp8(X, W1s, b1s, W2s, b2, "gelu_tanh", True)
    g = fp8.mlp_bwd_fp8(dY, f, "gelu_tanh", True)
    pre, A = fp8.column_fwd_fp8(X, W1s, b1s, "gelu_tanh")
    for i in range(T):
        assert np.array_equal(pre[i], f["pre"][i]) and np.array_equal(A[i], f["A"][i])
    assert np.array_equal(fp8.row_fwd_fp8(A, W2s, b2, X), f["Y"])
    dA, dW2, db2 = fp8.row_bwd_fp8(dY, A, W2s)
    for i in range(T):
        assert np.array_equal(dW2[i], g["dW2"][i])
        assert np.array_equal(fp8.round_bf16(oracle.act_bwd(f["pre"][i], dA[i], "gelu_tanh")), g["dPre"][i])
    assert np.array_equal(db2, g["db2"])
    dX, dW1, db1 = fp8.column_bwd_fp8(g["dPre"], X, W1s)
    assert np.array_equal(dX + dY, g["dX"])
    for i in range(T):
        assert np.array_equal(dW1[i], g["dW1"][i]) and np.array_equal(db1[i], g["db1"][i])


def test_sampled_fp8_layers_agree_with_full():
    """The sampled FP8 layer evaluators give the full functions' values at
    the sampled rows and units."""
    _, r, M, H, F, T = _layer_inputs(8, M=40, H=32, F=64, T=2)
    Fs = F // T
    X, W, dO = r(M, H), [r(Fs, H, sc=0.1) for _ in range(T)], [r(M, Fs) for _ in range(T)]
    rows, units = [0, 7, 39], [[0, 5, Fs - 1], [3, Fs - 1]]
    s = fp8.column_sampled_fp8(rows, units, X, W, dO)
    pre, _ = fp8.column_fwd_fp8(X, W, None, "none")
    dX, dW, _ = fp8.column_bwd_fp8(dO, X, W)
    assert np.allclose(s["dX"], dX[rows], rtol=1e-12, atol=1e-12)
    for i in range(T):
        assert np.array_equal(s["pre"][i], pre[i][rows])
        assert np.allclose(s["dW"][i], dW[i][units[i]], rtol=1e-12, atol=1e-12)
    Xs, W2, dY = [r(M, Fs) for _ in range(T)], [r(H, Fs, sc=0.1) for _ in range(T)], r(M, H)
    s = fp8.row_sampled_fp8(rows, units, Xs, W2, dY)
    assert np.allclose(s["Y"], fp8.row_fwd_fp8(Xs, W2)[rows], rtol=1e-12, atol=1e-12)
    rdX, rdW, _ = fp8.row_bwd_fp8(dY, Xs, W2)
    for i in range(T):
        assert np.allclose(s["dX"][i], rdX[i][rows], rtol=1e-12, atol=1e-12)
        assert np.allclose(s["dW"][i], rdW[i][:, units[i]], rtol=1e-12, atol=1e-12)
