"""CPU oracle of the tensor-parallel MLP -- TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline
leg may import this module.  It shares no code with the CUDA path.

Plain fp64 numpy: every shard is computed on its own and the cross-shard sums
("all-reduces") are written out as explicit loops over shards in the order
i = 0..T-1.  A matrix product is the only library primitive used.

Sources (page titles; sections / figures on them):
  [P1] "Megatron-LM 源码精读——大模型并行训练全景" (roger-lv.github.io)
       s3.1 ColumnParallelLinear, s3.2 RowParallelLinear, s3.3 MLP pairing
       figure, s3.4 mapping functions, s3.5 sequence parallelism,
       s5.2 gradient-accumulation fusion, s7 (SwiGLU, three matrices),
       s8.2 mixed precision.
  [P3] the "no-code" Megatron walk-through (gitcode.csdn.net):
       s02 Tensor Parallel shapes, s03 TransformerLayer (bias/dropout/residual
       add), s06 Sequence Parallel.
  [P4] "megatron-docs" table of contents: "f-g 共轭算子", "SwiGLU MLP".

Readings of points the pages leave open:
  R1 weights use the PyTorch [out, in] layout and Y = X W^T ([P1] s3.1 note on
     the stored shape; s3.2's W_i in R^{out x in/T} is only consistent with it).
  R2 GeLU is the tanh form 0.5x(1+tanh(sqrt(2/pi)(x+0.044715x^3))).
  R3 b1 is sharded with the column layer; b2 is added once, after the sum.
  R4 residual: Y = X + MLP(X) ([P3] s03 "bias/dropout/residual add"), so the
     input gradient gains + dY.
  R5 SwiGLU shard i of W1 is [gate rows of shard i ; up rows of shard i], each
     F/T rows; A = SiLU(G) * U with SiLU(x) = x * sigmoid(x).
  R6 sequence parallelism: the full [M, H] activation is the concatenation of
     T row blocks of M/T tokens; it changes storage, not the result.
"""
from __future__ import annotations

import math

import numpy as np

GELU_K0 = math.sqrt(2.0 / math.pi)
GELU_K1 = 0.044715

ACTS = ("none", "gelu_tanh", "swiglu")


def _f64(a):
    return None if a is None else np.asarray(a, dtype=np.float64)


def divide(numerator: int, denominator: int) -> int:
    """Exact division used for every shard size ([P1] s3.1:
    output_size_per_partition = divide(output_size, world_size)); a size that
    does not divide is an error."""
    if denominator <= 0 or numerator % denominator != 0:
        raise ValueError(f"{numerator} is not divisible by {denominator}")
    return numerator // denominator


# ----------------------------------------------------------------------------
# activations (R2, R5)
# ----------------------------------------------------------------------------
def gelu_tanh(x):
    u = GELU_K0 * (x + GELU_K1 * x * x * x)
    return 0.5 * x * (1.0 + np.tanh(u))


def gelu_tanh_grad(x):
    """d/dx of gelu_tanh: 0.5(1+t) + 0.5 x (1-t^2) sqrt(2/pi)(1+3*0.044715 x^2)."""
    t = np.tanh(GELU_K0 * (x + GELU_K1 * x * x * x))
    return 0.5 * (1.0 + t) + 0.5 * x * (1.0 - t * t) * GELU_K0 * (1.0 + 3.0 * GELU_K1 * x * x)


def sigmoid(x):
    return 1.0 / (1.0 + np.exp(-x))


def silu(x):
    return x * sigmoid(x)


def act_fwd(pre, act: str):
    """A_i = act(pre_i).  For SwiGLU pre_i = [G_i | U_i] along columns (R5)."""
    if act == "none":
        return pre.copy()
    if act == "gelu_tanh":
        return gelu_tanh(pre)
    if act == "swiglu":
        f = pre.shape[1] // 2
        return silu(pre[:, :f]) * pre[:, f:]
    raise ValueError(act)


def act_bwd(pre, dA, act: str):
    """dPre_i = dA_i (.) act'(pre_i).  SwiGLU: dG = dA U s (1 + G (1 - s)) with
    s = sigmoid(G), dU = dA SiLU(G)."""
    if act == "none":
        return dA.copy()
    if act == "gelu_tanh":
        return dA * gelu_tanh_grad(pre)
    if act == "swiglu":
        f = pre.shape[1] // 2
        G, U = pre[:, :f], pre[:, f:]
        s = sigmoid(G)
        dG = dA * U * s * (1.0 + G * (1.0 - s))
        dU = dA * G * s
        return np.concatenate([dG, dU], axis=1)
    raise ValueError(act)


# ----------------------------------------------------------------------------
# shard layout ([P1] s3.1, s3.2; R1, R5)
# ----------------------------------------------------------------------------
def shard_column_weight(W, T: int, act: str = "none"):
    """Split a column-parallel weight [out, in] into T shards along the output
    dimension.  With SwiGLU the full weight is [gate; up] (2F rows) and shard i
    stacks its gate rows over its up rows (R5)."""
    W = np.asarray(W)
    if act == "swiglu":
        F = W.shape[0] // 2
        fs = divide(F, T)
        return [np.concatenate([W[i * fs:(i + 1) * fs], W[F + i * fs:F + (i + 1) * fs]], axis=0)
                for i in range(T)]
    fs = divide(W.shape[0], T)
    return [W[i * fs:(i + 1) * fs] for i in range(T)]


def shard_column_bias(b, T: int, act: str = "none"):
    if b is None:
        return [None] * T
    b = np.asarray(b)
    if act == "swiglu":
        F = b.shape[0] // 2
        fs = divide(F, T)
        return [np.concatenate([b[i * fs:(i + 1) * fs], b[F + i * fs:F + (i + 1) * fs]]) for i in range(T)]
    fs = divide(b.shape[0], T)
    return [b[i * fs:(i + 1) * fs] for i in range(T)]


def unshard_column(parts, act: str = "none"):
    """Inverse of shard_column_weight / shard_column_bias (axis 0)."""
    if act == "swiglu":
        fs = parts[0].shape[0] // 2
        return np.concatenate([p[:fs] for p in parts] + [p[fs:] for p in parts], axis=0)
    return np.concatenate(parts, axis=0)


def shard_row_weight(W, T: int):
    """Split a row-parallel weight [out, in] into T shards along the input
    dimension: W_i = W[:, i*in/T:(i+1)*in/T] ([P1] s3.2)."""
    W = np.asarray(W)
    ks = divide(W.shape[1], T)
    return [W[:, i * ks:(i + 1) * ks] for i in range(T)]


def sp_split(X, T: int):
    """Sequence-parallel storage: T row blocks of M/T tokens ([P1] s3.5,
    [P3] s06: [S,B,H] -> [S/T,B,H] per rank)."""
    ms = divide(X.shape[0], T)
    return [X[j * ms:(j + 1) * ms] for j in range(T)]


def sp_gather(shards):
    """All-gather of the sequence shards (concatenate along tokens)."""
    return np.concatenate(list(shards), axis=0)


# ----------------------------------------------------------------------------
# layers
# ----------------------------------------------------------------------------
def column_fwd(X, W_shards, b_shards, act: str):
    """ColumnParallelLinear + activation ([P1] s3.1, s3.3): X is replicated;
    shard i computes pre_i = X W_i^T + b_i and A_i = act(pre_i) with no
    communication."""
    X = _f64(X)
    pre, A = [], []
    for i, W in enumerate(W_shards):
        p = X @ _f64(W).T
        if b_shards is not None and b_shards[i] is not None:
            p = p + _f64(b_shards[i])
        pre.append(p)
        A.append(act_fwd(p, act))
    return pre, A


def row_fwd(X_shards, W_shards, b=None, R=None):
    """RowParallelLinear ([P1] s3.2, [P3] s02): shard i computes the partial
    output X_i W_i^T of full width; the forward all-reduce is the explicit
    sum over i = 0..T-1; the bias is added once after it (R3) and the
    residual R after that (R4)."""
    Y = None
    for i, W in enumerate(W_shards):
        part = _f64(X_shards[i]) @ _f64(W).T
        Y = part if Y is None else Y + part
    if b is not None:
        Y = Y + _f64(b)
    if R is not None:
        Y = Y + _f64(R)
    return Y


def column_bwd(dOut_shards, X, W_shards):
    """Backward of ColumnParallelLinear with respect to its (pre-activation)
    outputs: dX = sum_i dOut_i W_i (the backward all-reduce, [P1] s3.1),
    dW_i = dOut_i^T X, db_i = sum over tokens of dOut_i."""
    X = _f64(X)
    dX = None
    dW, db = [], []
    for i, W in enumerate(W_shards):
        d = _f64(dOut_shards[i])
        part = d @ _f64(W)
        dX = part if dX is None else dX + part
        dW.append(d.T @ X)
        db.append(d.sum(axis=0))
    return dX, dW, db


def row_bwd(dY, X_shards, W_shards):
    """Backward of RowParallelLinear: no communication ([P1] s3.2).
    dX_i = dY W_i, dW_i = dY^T X_i, db = sum over tokens of dY."""
    dY = _f64(dY)
    dX = [dY @ _f64(W) for W in W_shards]
    dW = [dY.T @ _f64(Xi) for Xi in X_shards]
    return dX, dW, dY.sum(axis=0)


# ----------------------------------------------------------------------------
# the MLP ([P1] s3.3 figure: X -> Column -> GeLU -> Row -> all-reduce -> Y)
# ----------------------------------------------------------------------------
def mlp_fwd(X, W1s, b1s, W2s, b2, act: str, residual: bool):
    """Returns (pre list, A list, Y), all fp64.  X is the full [M, H] input
    (gather sequence shards first with :func:`sp_gather`)."""
    pre, A = column_fwd(X, W1s, b1s, act)
    Y = row_fwd(A, W2s, b2, X if residual else None)
    return pre, A, Y


def mlp_bwd(dY, X, W1s, W2s, pre, A, act: str, residual: bool):
    """Backward of :func:`mlp_fwd` given the upstream gradient dY [M, H].

    Row layer (no communication): dA_i = dY W2_i, dW2_i = dY^T A_i,
    db2 = sum_m dY.  Activation: dPre_i = dA_i (.) act'(pre_i).  Column layer:
    dW1_i = dPre_i^T X, db1_i = sum_m dPre_i and dX = sum_i dPre_i W1_i (the
    backward all-reduce), plus dY with the residual.  Returns a dict."""
    dY = _f64(dY)
    dA, dW2, db2 = row_bwd(dY, A, W2s)
    dPre = [act_bwd(pre[i], dA[i], act) for i in range(len(W1s))]
    dX, dW1, db1 = column_bwd(dPre, X, W1s)
    if residual:
        dX = dX + dY
    return {"dA": dA, "dPre": dPre, "dX": dX, "dW1": dW1, "db1": db1, "dW2": dW2, "db2": db2}


def mlp_loss(X, W1s, b1s, W2s, b2, dY, act: str, residual: bool) -> float:
    """<dY, Y>: the scalar whose gradient :func:`mlp_bwd` returns."""
    _, _, Y = mlp_fwd(X, W1s, b1s, W2s, b2, act, residual)
    return float(np.sum(_f64(dY) * Y))


# ----------------------------------------------------------------------------
# sampled evaluation for full-size problems
# ----------------------------------------------------------------------------
def mlp_rows(rows, X, W1s, b1s, W2s, b2, dY, act: str, residual: bool):
    """Y, dX, pre_i, A_i and dPre_i at the given token rows only.  Exact,
    because every token row is independent in both passes."""
    rows = np.asarray(rows)
    Xr = _f64(X)[rows]
    dYr = _f64(dY)[rows]
    pre, A, Y = mlp_fwd(Xr, W1s, b1s, W2s, b2, act, residual)
    g = mlp_bwd(dYr, Xr, W1s, W2s, pre, A, act, residual)
    return {"Y": Y, "dX": g["dX"], "pre": pre, "A": A, "dPre": g["dPre"]}


def mlp_units(units, X, W1s, b1s, W2s, dY, act: str):
    """Weight and bias gradients of the given hidden units of every shard.

    ``units[i]`` lists unit indices u in [0, F/T) of shard i.  Returns, per
    shard, dW1 rows (for SwiGLU the gate row u and the up row F/T + u,
    stacked), dW2 columns [H, len(u)] and db1 entries (same stacking as dW1).
    Exact: a hidden unit's gradients depend only on its own pre-activation
    column over all tokens."""
    X = _f64(X)
    dY = _f64(dY)
    out = {"dW1": [], "dW2": [], "db1": []}
    for i, W1 in enumerate(W1s):
        u = np.asarray(units[i])
        W1 = _f64(W1)
        fs = W2s[i].shape[1]
        rows1 = np.concatenate([u, fs + u]) if act == "swiglu" else u
        pre = X @ W1[rows1].T
        if b1s is not None and b1s[i] is not None:
            pre = pre + _f64(b1s[i])[rows1]
        A = act_fwd(pre, act)
        W2u = _f64(W2s[i])[:, u]
        dA = dY @ W2u
        dPre = act_bwd(pre, dA, act)
        out["dW1"].append(dPre.T @ X)
        out["dW2"].append(dY.T @ A)
        out["db1"].append(dPre.sum(axis=0))
    return out
