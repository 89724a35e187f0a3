"""TransformerLayer MLP sub-block -- oracle, TEST INFRASTRUCTURE ONLY.

Only ``tests/`` and ``bench.py``'s CPU legs import this module; it shares no
code with the CUDA path.

Source: the gitcode.csdn.net Megatron Core walk-through, s03 TransformerLayer:
hidden -> LayerNorm -> ... -> LayerNorm -> MLP -> bias/dropout/residual add ->
hidden; "Megatron-LM 源码精读" s3.5 (sequence parallelism keeps the
LayerNorm's activations split along the sequence).  This module computes the
MLP half of that layer:

    Xn = LayerNorm(X; gamma, beta)            per token, over H
    Z  = MLP(Xn) = sum_i A_i W2_i^T + b2      (mlp.py)
    Y  = X + dropout_p(Z)                     bias-dropout-add: the bias is
                                              inside the dropout, the residual
                                              is the block's input X

Readings:
  L1 LayerNorm with the population variance, eps = 1e-5, affine gamma/beta;
  L2 dropout keeps an element when its 24-bit uniform draw u24 satisfies
     u24 >= floor(p * 2^24) and scales kept elements by 1/(1-p);
  L3 the draw for element (m, h) (m the global token index, so sequence
     sharding does not change it) comes from Philox4x32-10 (Salmon, Moraes,
     Dror & Shaw, "Parallel random numbers: as easy as 1, 2, 3", SC 2011) with
     key (seed mod 2^32, seed div 2^32) and counter (q mod 2^32, q div 2^32, 0,
     0), q = (m*H + h) div 4, taking output word (m*H + h) mod 4 and its top 24
     bits;
  L4 backward: dZ = dY * keep / (1-p); the MLP backward runs on dZ; the
     LayerNorm backward adds the residual gradient dY.
"""
from __future__ import annotations

import numpy as np

from . import fp8 as _fp8
from . import mlp as _mlp

LN_EPS = 1e-5

_M0, _M1 = np.uint64(0xD2511F53), np.uint64(0xCD9E8D57)
_W0, _W1 = np.uint32(0x9E3779B9), np.uint32(0xBB67AE85)
_MASK32 = np.uint64(0xFFFFFFFF)


def philox4x32_10(c0, c1, c2, c3, k0, k1):
    """Philox4x32 with 10 rounds on uint32 arrays (counter words c0..c3, key
    words k0, k1).  One round: (hi0, lo0) = M0 * c0, (hi1, lo1) = M1 * c2,
    then (c0, c1, c2, c3) = (hi1 ^ c1 ^ k0, lo1, hi0 ^ c3 ^ k1, lo0); the key
    is bumped by the Weyl constants between rounds."""
    c0, c1, c2, c3 = (np.asarray(v, dtype=np.uint32) for v in (c0, c1, c2, c3))
    k0 = np.uint32(k0)
    k1 = np.uint32(k1)
    for r in range(10):
        p0 = _M0 * c0.astype(np.uint64)
        p1 = _M1 * c2.astype(np.uint64)
        hi0, lo0 = (p0 >> np.uint64(32)).astype(np.uint32), (p0 & _MASK32).astype(np.uint32)
        hi1, lo1 = (p1 >> np.uint64(32)).astype(np.uint32), (p1 & _MASK32).astype(np.uint32)
        c0, c1, c2, c3 = hi1 ^ c1 ^ k0, lo1, hi0 ^ c3 ^ k1, lo0
        if r < 9:
            with np.errstate(over="ignore"):
                k0 = np.uint32((int(k0) + int(_W0)) & 0xFFFFFFFF)
                k1 = np.uint32((int(k1) + int(_W1)) & 0xFFFFFFFF)
    return c0, c1, c2, c3


def dropout_threshold(p: float) -> int:
    """24-bit threshold: an element is kept when its draw is >= this (L2)."""
    if not 0.0 <= p < 1.0:
        raise ValueError("dropout probability must be in [0, 1)")
    return int(np.floor(p * 2.0 ** 24))


def dropout_keep(seed: int, rows, H: int, p: float):
    """Keep mask [len(rows), H] for the given global token rows (L2, L3)."""
    rows = np.asarray(rows, dtype=np.int64)
    t = dropout_threshold(p)
    idx = rows[:, None] * H + np.arange(H, dtype=np.int64)[None, :]
    q = idx // 4
    w = idx % 4
    k0, k1 = seed & 0xFFFFFFFF, (seed >> 32) & 0xFFFFFFFF
    zeros = np.zeros(q.shape, np.uint32)
    out = philox4x32_10((q & 0xFFFFFFFF).astype(np.uint32), (q >> 32).astype(np.uint32), zeros, zeros, k0, k1)
    word = np.choose(w, out)
    return (word >> np.uint32(8)) >= np.uint32(t)


def layernorm_fwd(X, gamma, beta, eps: float = LN_EPS):
    """Per-token LayerNorm (L1).  Returns (Xn, mean, rstd)."""
    X = np.asarray(X, np.float64)
    mean = X.mean(axis=1)
    var = ((X - mean[:, None]) ** 2).mean(axis=1)
    rstd = 1.0 / np.sqrt(var + eps)
    xhat = (X - mean[:, None]) * rstd[:, None]
    return xhat * np.asarray(gamma, np.float64) + np.asarray(beta, np.float64), mean, rstd


def layernorm_bwd(dXn, X, gamma, mean, rstd):
    """Gradients of layernorm_fwd: (dX, dgamma, dbeta).  With
    g = dXn * gamma and xhat = (X - mean) * rstd:
    dX = rstd * (g - mean_h(g) - xhat * mean_h(g * xhat))."""
    dXn = np.asarray(dXn, np.float64)
    X = np.asarray(X, np.float64)
    xhat = (X - mean[:, None]) * rstd[:, None]
    g = dXn * np.asarray(gamma, np.float64)
    dX = rstd[:, None] * (g - g.mean(axis=1, keepdims=True) - xhat * (g * xhat).mean(axis=1, keepdims=True))
    return dX, (dXn * xhat).sum(axis=0), dXn.sum(axis=0)


def layer_fwd(X, gamma, beta, W1s, b1s, W2s, b2, act: str, p: float, seed: int, eps: float = LN_EPS):
    """Forward of the sub-block on the full [M, H] input X."""
    Xn, mean, rstd = layernorm_fwd(X, gamma, beta, eps)
    pre, A, Z = _mlp.mlp_fwd(Xn, W1s, b1s, W2s, b2, act, False)
    keep = dropout_keep(seed, np.arange(Z.shape[0]), Z.shape[1], p)
    Y = np.asarray(X, np.float64) + np.where(keep, Z / (1.0 - p), 0.0)
    return {"Xn": Xn, "mean": mean, "rstd": rstd, "pre": pre, "A": A, "Z": Z, "keep": keep, "Y": Y}


def layer_bwd(dY, X, gamma, W1s, W2s, f, act: str, p: float):
    """Backward given the forward's dict ``f`` (L4)."""
    dY = np.asarray(dY, np.float64)
    dZ = np.where(f["keep"], dY / (1.0 - p), 0.0)
    g = _mlp.mlp_bwd(dZ, f["Xn"], W1s, W2s, f["pre"], f["A"], act, False)
    dXln, dgamma, dbeta = layernorm_bwd(g["dX"], X, gamma, f["mean"], f["rstd"])
    g.update(dZ=dZ, dXn=g["dX"], dX=dY + dXln, dgamma=dgamma, dbeta=dbeta)
    return g


def layer_fwd_fp8(X, gamma, beta, W1s, b1s, W2s, b2, act: str, p: float, seed: int, eps: float = LN_EPS,
                  history=None):
    """The sub-block with the MLP in the FP8 variant (fp8.py): the LayerNorm
    output is stored in bf16 and that bf16 tensor is the MLP's input (reading
    F4 of fp8.py applied to Xn).  ``history``: delayed scaling (fp8.py F6)."""
    Xn, mean, rstd = layernorm_fwd(X, gamma, beta, eps)
    Xn_b = _fp8.round_bf16(Xn)
    f = _fp8.mlp_fwd_fp8(Xn_b, W1s, b1s, W2s, b2, act, False, history)
    Z = f["Y"]
    keep = dropout_keep(seed, np.arange(Z.shape[0]), Z.shape[1], p)
    Y = np.asarray(X, np.float64) + np.where(keep, Z / (1.0 - p), 0.0)
    return {"Xn": Xn_b, "mean": mean, "rstd": rstd, "pre": f["pre"], "A": f["A"], "Z": Z, "keep": keep, "Y": Y,
            "mlp": f}


def layer_bwd_fp8(dY, X, gamma, act: str, p: float, f, history=None):
    """Backward of layer_fwd_fp8: dZ and dXn are stored in bf16 (F4), the MLP
    backward is fp8.mlp_bwd_fp8 on dZ."""
    dY = np.asarray(dY, np.float64)
    dZ = _fp8.round_bf16(np.where(f["keep"], dY / (1.0 - p), 0.0))
    g = _fp8.mlp_bwd_fp8(dZ, f["mlp"], act, False, history)
    dXn = _fp8.round_bf16(g["dX"])
    dXln, dgamma, dbeta = layernorm_bwd(dXn, X, gamma, f["mean"], f["rstd"])
    g.update(dZ=dZ, dXn=dXn, dX=dY + dXln, dgamma=dgamma, dbeta=dbeta)
    return g
