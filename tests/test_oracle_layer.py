"""Pins of the TransformerLayer MLP sub-block oracle (oracle/layer.py):
Philox4x32-10 known-answer vectors of its publication, LayerNorm against
torch, and the whole sub-block against torch fp64 autograd with the same
dropout mask."""
import numpy as np
import pytest
import torch
import torch.nn.functional as F

import oracle
from oracle import layer


def test_philox_known_answers():
    """Known-answer vectors published with Philox4x32-10 (Salmon et al., SC 2011;
    Random123 distribution): (counter, key) -> output."""
    kat = [
        ((0, 0, 0, 0), (0, 0), (0x6627E8D5, 0xE169C58D, 0xBC57AC4C, 0x9B00DBD8)),
        ((0xFFFFFFFF,) * 4, (0xFFFFFFFF, 0xFFFFFFFF), (0x408F276D, 0x41C83B0E, 0xA20BC7C6, 0x6D5451FD)),
        ((0x243F6A88, 0x85A308D3, 0x13198A2E, 0x03707344), (0xA4093822, 0x299F31D0),
         (0xD16CFE09, 0x94FDCCEB, 0x5001E420, 0x24126EA1)),
    ]
    for ctr, key, want in kat:
        got = layer.philox4x32_10(*[[c] for c in ctr], *key)
        assert tuple(int(g[0]) for g in got) == want


def test_dropout_mask_statistics_and_row_independence():
    M, H, p, seed = 512, 256, 0.3, 1234
    keep = layer.dropout_keep(seed, np.arange(M), H, p)
    assert abs(keep.mean() - (1 - p)) < 0.005
    # rows are independent: a slice of rows equals the corresponding rows
    assert np.array_equal(layer.dropout_keep(seed, np.arange(100, 164), H, p), keep[100:164])
    assert layer.dropout_keep(seed, np.arange(8), H, 0.0).all()
    assert not np.array_equal(layer.dropout_keep(seed + 1, np.arange(M), H, p), keep)
    with pytest.raises(ValueError):
        layer.dropout_threshold(1.0)


def test_layernorm_matches_torch():
    rng = np.random.default_rng(0)
    X = rng.standard_normal((16, 24)) * 3 + 1
    gamma, beta = rng.standard_normal(24), rng.standard_normal(24)
    dXn = rng.standard_normal((16, 24))
    Xt = torch.tensor(X, requires_grad=True)
    gt = torch.tensor(gamma, requires_grad=True)
    bt = torch.tensor(beta, requires_grad=True)
    y = F.layer_norm(Xt, (24,), gt, bt, eps=layer.LN_EPS)
    (y * torch.tensor(dXn)).sum().backward()
    Xn, mean, rstd = layer.layernorm_fwd(X, gamma, beta)
    assert np.max(np.abs(Xn - y.detach().numpy())) < 1e-12
    dX, dg, db = layer.layernorm_bwd(dXn, X, gamma, mean, rstd)
    assert np.max(np.abs(dX - Xt.grad.numpy())) < 1e-12
    assert np.max(np.abs(dg - gt.grad.numpy())) < 1e-12
    assert np.max(np.abs(db - bt.grad.numpy())) < 1e-12


@pytest.mark.parametrize("act", ["gelu_tanh", "swiglu"])
def test_sub_block_matches_torch_autograd(act):
    rng = np.random.default_rng(4)
    M, H, Fw, T, p, seed = 12, 16, 32, 2, 0.25, 77
    g = 2 if act == "swiglu" else 1
    X = rng.standard_normal((M, H))
    gamma, beta = 1 + 0.1 * rng.standard_normal(H), 0.1 * rng.standard_normal(H)
    W1 = rng.standard_normal((g * Fw, H)) * 0.3
    W2 = rng.standard_normal((H, Fw)) * 0.3
    b1, b2 = rng.standard_normal(g * Fw) * 0.1, rng.standard_normal(H) * 0.1
    dY = rng.standard_normal((M, H))
    W1s, b1s = oracle.shard_column_weight(W1, T, act), oracle.shard_column_bias(b1, T, act)
    W2s = oracle.shard_row_weight(W2, T)
    f = layer.layer_fwd(X, gamma, beta, W1s, b1s, W2s, b2, act, p, seed)
    gr = layer.layer_bwd(dY, X, gamma, W1s, W2s, f, act, p)
    t = lambda a: torch.tensor(a, dtype=torch.float64, requires_grad=True)
    Xt, gt, bt, W1t, b1t, W2t, b2t = map(t, (X, gamma, beta, W1, b1, W2, b2))
    xn = F.layer_norm(Xt, (H,), gt, bt, eps=layer.LN_EPS)
    pre = F.linear(xn, W1t, b1t)
    if act == "swiglu":
        G, U = pre.chunk(2, dim=1)
        A = F.silu(G) * U
    else:
        A = F.gelu(pre, approximate="tanh")
    Z = F.linear(A, W2t, b2t)
    keep = torch.tensor(f["keep"])
    Y = Xt + torch.where(keep, Z / (1 - p), torch.zeros_like(Z))
    (Y * torch.tensor(dY)).sum().backward()
    rel = lambda a, b: np.max(np.abs(np.asarray(a) - np.asarray(b))) / np.max(np.abs(b))
    assert rel(f["Y"], Y.detach().numpy()) < 1e-13
    assert rel(gr["dX"], Xt.grad.numpy()) < 1e-12
    assert rel(gr["dgamma"], gt.grad.numpy()) < 1e-12
    assert rel(gr["dbeta"], bt.grad.numpy()) < 1e-12
    assert rel(oracle.unshard_column(gr["dW1"], act), W1t.grad.numpy()) < 1e-12
    assert rel(oracle.unshard_column(gr["db1"], act), b1t.grad.numpy()) < 1e-12
    assert rel(np.concatenate(gr["dW2"], axis=1), W2t.grad.numpy()) < 1e-12
    assert rel(gr["db2"], b2t.grad.numpy()) < 1e-12
    assert 0 < f["keep"].mean() < 1


def test_fp8_sub_block_stays_within_the_fp8_error_of_the_exact_one():
    """layer_fwd_fp8 / layer_bwd_fp8 differ from the exact sub-block only by
    the FP8 rounding of the MLP's operands (a few percent of max |ref|), and
    share its dropout flags and LayerNorm statistics exactly.  Forward bound:
    E4M3's relative half-step 2^-4 plus margin; backward bound: E5M2's
    relative half-step 2^-3 (dZ and dPre are E5M2 operands)."""
    rng = np.random.default_rng(11)
    M, H, F, T, p, seed = 64, 64, 256, 2, 0.2, 99
    X = rng.normal(size=(M, H)) * 2 + 0.5
    gamma, beta = 1 + 0.1 * rng.normal(size=H), 0.05 * rng.normal(size=H)
    W1s = [0.1 * rng.normal(size=(F // T, H)) for _ in range(T)]
    b1s = [0.02 * rng.normal(size=F // T) for _ in range(T)]
    W2s = [0.1 * rng.normal(size=(H, F // T)) for _ in range(T)]
    b2 = 0.02 * rng.normal(size=H)
    dY = rng.normal(size=(M, H))
    e = layer.layer_fwd(X, gamma, beta, W1s, b1s, W2s, b2, "gelu_tanh", p, seed)
    q = layer.layer_fwd_fp8(X, gamma, beta, W1s, b1s, W2s, b2, "gelu_tanh", p, seed)
    assert np.array_equal(e["keep"], q["keep"])
    assert np.array_equal(e["mean"], q["mean"]) and np.array_equal(e["rstd"], q["rstd"])
    dz = e["Y"] - X
    assert 0 < np.max(np.abs((q["Y"] - X) - dz)) / np.max(np.abs(dz)) < 0.08
    ge = layer.layer_bwd(dY, X, gamma, W1s, W2s, e, "gelu_tanh", p)
    gq = layer.layer_bwd_fp8(dY, X, gamma, "gelu_tanh", p, q)
    for k in ("dgamma", "dbeta", "db2"):
        r = np.max(np.abs(gq[k] - ge[k])) / np.max(np.abs(ge[k]))
        assert r < 0.125, (k, r)
