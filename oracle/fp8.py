"""FP8 variant of the tensor-parallel MLP -- oracle, TEST INFRASTRUCTURE ONLY.

Only ``tests/`` and ``bench.py``'s CPU legs import this module; it shares no
code with the CUDA path.

Source: "Megatron-LM 源码精读——大模型并行训练全景" (roger-lv.github.io), s8.2
(mixed precision / FP8): E4M3 in the forward, E5M2 in the backward, per-tensor
scaling from the tensor's amax, with the amax reduced across the tensor- and
data-parallel group.  Readings:
  F1 one scale per logical tensor: the amax is the maximum over all T shards
     (the cross-shard amax all-reduce), scale = fmax / amax computed in fp32
     (1 when amax is 0), fmax = 448 (E4M3) or 57344 (E5M2);
  F2 quantisation q = fp8(x * scale): the product is rounded to fp32, then to
     the FP8 format with round-to-nearest-even, saturating to +-fmax;
  F3 a GEMM of quantised operands is dequantised by 1 / (scale_a * scale_b)
     (fp32), applied to the fp32/fp64 sum before bias, activation or residual;
  F4 the forward quantises X, W1, W2 (E4M3) and the stored bf16 activation A
     (E4M3); the backward quantises dY (E5M2) and the stored bf16 dPre (E5M2);
     pre, A, dPre, Y and dX are stored in bf16 (round-to-nearest-even), as in
     the bf16 variant, and act' uses the stored bf16 pre;
  F5 bias gradients sum the unquantised bf16 dPre and dY.
  F6 delayed scaling (the pages' "amax history"): a tensor's scale may come
     from the maximum of the amaxes its last n quantisations recorded (n = 1
     is the previous step's amax) instead of from its own amax; while its
     history is empty (the first step) it uses its own amax.  Every
     quantisation records the tensor's own amax.  No margin.

FP8 formats (OCP 8-bit floating point): E4M3 -- 1 sign, 4 exponent bits
(bias 7), 3 mantissa bits, largest finite 448, smallest normal 2^-6, smallest
subnormal 2^-9, no infinities; E5M2 -- 1 sign, 5 exponent bits (bias 15),
2 mantissa bits, largest finite 57344, smallest normal 2^-14, smallest
subnormal 2^-16.
"""
from __future__ import annotations

import numpy as np

from . import mlp as _mlp

FORMATS = {
    # name: (mantissa bits, minimum normal exponent, largest finite)
    "e4m3": (3, -6, 448.0),
    "e5m2": (2, -14, 57344.0),
}


def fmax(fmt: str) -> float:
    return FORMATS[fmt][2]


def round_fp8(v, fmt: str):
    """Round values (exact in fp64) to the FP8 format: nearest, ties to even,
    saturating to the largest finite value (F2).  Returns fp64 values."""
    mbits, emin, top = FORMATS[fmt]
    v = np.asarray(v, dtype=np.float64)
    a = np.abs(v)
    _, ex = np.frexp(np.where(a > 0, a, 1.0))   # a = m * 2^ex with m in [0.5, 1)
    e = (ex - 1).astype(np.float64)
    e = np.maximum(e, emin)               # subnormals share the minimum exponent's quantum
    quantum = np.exp2(e - mbits)
    q = np.rint(a / quantum) * quantum    # np.rint: round half to even
    q = np.minimum(q, top)
    return np.copysign(q, v) * (a > 0)


def round_bf16(x):
    """Round to bf16 (nearest, ties to even) through the fp32 bit pattern."""
    f = np.asarray(x, dtype=np.float32)
    u = f.view(np.uint32).astype(np.uint64)
    r = ((u + 0x7FFF + ((u >> 16) & 1)) >> 16) << 16
    return r.astype(np.uint32).view(np.float32).astype(np.float64)


def scale_of(amax, fmt: str) -> np.float32:
    """Per-tensor scale fmax / amax in fp32 (F1); 1 when amax is 0."""
    amax = np.float32(amax)
    if amax == 0 or not np.isfinite(amax):
        return np.float32(1.0)
    return np.float32(np.float32(fmax(fmt)) / amax)


def amax_of(parts) -> np.float32:
    """Maximum |x| over all shards of one logical tensor (F1)."""
    return np.float32(max(float(np.max(np.abs(np.asarray(p, np.float64)))) if np.size(p) else 0.0
                          for p in parts))


class AmaxHistory:
    """Delayed scaling (F6): per tensor name, the amaxes of its last n
    quantisations."""

    def __init__(self, n: int):
        if n < 1:
            raise ValueError("history length must be >= 1")
        self.n = n
        self.hist = {}

    def amax_for(self, name: str, amax):
        """The amax the scale derives from: the history's maximum, or the
        tensor's own amax while the history is empty."""
        h = self.hist.get(name)
        return np.float32(max(h)) if h else np.float32(amax)

    def record(self, name: str, amax):
        h = self.hist.setdefault(name, [])
        h.append(np.float32(amax))
        del h[:-self.n]


def quantize(parts, fmt: str, name: str = None, history: "AmaxHistory" = None):
    """Quantise every shard of one tensor with the tensor's scale (F1, F2),
    or with the scale its amax history gives (F6) when ``history`` is set.
    Returns (list of quantised values as fp64, scale)."""
    a = amax_of(parts)
    s = scale_of(history.amax_for(name, a) if history is not None else a, fmt)
    out = [round_fp8((np.asarray(p, np.float32) * s).astype(np.float32), fmt) for p in parts]
    if history is not None:
        history.record(name, a)
    return out, s


def dequant(sa, sb) -> float:
    """Dequantisation factor of a product of two quantised operands (F3)."""
    return float(np.float32(1.0) / np.float32(np.float32(sa) * np.float32(sb)))


def mlp_fwd_fp8(X, W1s, b1s, W2s, b2, act: str, residual: bool, history: AmaxHistory = None):
    """Forward of the FP8 variant.  X is the full [M, H] input (bf16 values).
    Returns a dict with pre, A (bf16-rounded, per shard), Y (fp64, before the
    bf16 store), and the quantised operands and scales the backward reuses.
    ``history``: delayed scaling (F6) with this state, updated in place."""
    T = len(W1s)
    (Xq,), sx = quantize([X], "e4m3", "X", history)
    W1q, sw1 = quantize(W1s, "e4m3", "W1", history)
    W2q, sw2 = quantize(W2s, "e4m3", "W2", history)
    d1 = dequant(sx, sw1)
    pre, A = [], []
    for i in range(T):
        p = (Xq @ W1q[i].T) * d1
        if b1s is not None and b1s[i] is not None:
            p = p + np.asarray(b1s[i], np.float64)
        pre.append(round_bf16(p))
        A.append(round_bf16(_mlp.act_fwd(p, act)))
    Aq, sa = quantize(A, "e4m3", "A", history)
    d2 = dequant(sa, sw2)
    Y = None
    for i in range(T):
        part = Aq[i] @ W2q[i].T
        Y = part if Y is None else Y + part
    Y = Y * d2
    if b2 is not None:
        Y = Y + np.asarray(b2, np.float64)
    if residual:
        Y = Y + np.asarray(X, np.float64)
    return {"pre": pre, "A": A, "Y": Y, "Xq": Xq, "W1q": W1q, "W2q": W2q, "Aq": Aq,
            "sx": sx, "sw1": sw1, "sw2": sw2, "sa": sa}


def mlp_bwd_fp8(dY, f, act: str, residual: bool, history: AmaxHistory = None):
    """Backward of the FP8 variant given the forward's dict ``f``
    (``history`` as in mlp_fwd_fp8)."""
    T = len(f["W1q"])
    (dYq,), sdy = quantize([dY], "e5m2", "dY", history)
    d = dequant(sdy, f["sw2"])
    dPre = []
    for i in range(T):
        dA = (dYq @ f["W2q"][i]) * d
        dPre.append(round_bf16(_mlp.act_bwd(f["pre"][i], dA, act)))
    dPq, sdp = quantize(dPre, "e5m2", "dPre", history)
    dW2 = [(dYq.T @ f["Aq"][i]) * dequant(sdy, f["sa"]) for i in range(T)]
    dW1 = [(dPq[i].T @ f["Xq"]) * dequant(sdp, f["sx"]) for i in range(T)]
    dX = None
    for i in range(T):
        part = dPq[i] @ f["W1q"][i]
        dX = part if dX is None else dX + part
    dX = dX * dequant(sdp, f["sw1"])
    if residual:
        dX = dX + np.asarray(dY, np.float64)
    db1 = [p.sum(axis=0) for p in dPre]
    db2 = np.asarray(dY, np.float64).sum(axis=0)
    return {"dPre": dPre, "dX": dX, "dW1": dW1, "dW2": dW2, "db1": db1, "db2": db2, "sdy": sdy, "sdp": sdp}


def mlp_sampled_fp8(rows, units, X, W1s, b1s, W2s, b2, dY, act: str, residual: bool):
    """The FP8 variant's Y and dX at the given token rows and its dW1 rows,
    dW2 columns and db1 entries at the given hidden units of every shard
    (``units[i]`` indexes [0, F/T) of shard i; for SwiGLU both the gate and the
    up row of a unit), plus db2 in full.

    The per-tensor scales of A and dPre depend on every token, so A and dPre
    are formed in full (two GEMMs); every other product is evaluated only where
    sampled.  Same arithmetic as mlp_fwd_fp8 / mlp_bwd_fp8."""
    rows = np.asarray(rows)
    T = len(W1s)
    fs = np.asarray(W2s[0]).shape[1]
    (Xq,), sx = quantize([X], "e4m3")
    W1q, sw1 = quantize(W1s, "e4m3")
    W2q, sw2 = quantize(W2s, "e4m3")
    d1 = dequant(sx, sw1)
    pre, A = [], []
    for i in range(T):
        p = (Xq @ W1q[i].T) * d1
        if b1s is not None and b1s[i] is not None:
            p = p + np.asarray(b1s[i], np.float64)
        pre.append(round_bf16(p))
        A.append(round_bf16(_mlp.act_fwd(p, act)))
        del p
    Aq, sa = quantize(A, "e4m3")
    Y = sum(Aq[i][rows] @ W2q[i].T for i in range(T)) * dequant(sa, sw2)
    if b2 is not None:
        Y = Y + np.asarray(b2, np.float64)
    if residual:
        Y = Y + np.asarray(X, np.float64)[rows]
    (dYq,), sdy = quantize([dY], "e5m2")
    d = dequant(sdy, sw2)
    dPre = [round_bf16(_mlp.act_bwd(pre[i], (dYq @ W2q[i]) * d, act)) for i in range(T)]
    dPq, sdp = quantize(dPre, "e5m2")
    dX = sum(dPq[i][rows] @ W1q[i] for i in range(T)) * dequant(sdp, sw1)
    if residual:
        dX = dX + np.asarray(dY, np.float64)[rows]
    out = {"Y": Y, "dX": dX, "dW1": [], "dW2": [], "db1": [],
           "db2": np.asarray(dY, np.float64).sum(axis=0)}
    for i in range(T):
        u = np.asarray(units[i])
        sel = np.concatenate([u, fs + u]) if act == "swiglu" else u
        out["dW1"].append((dPq[i][:, sel].T @ Xq) * dequant(sdp, sx))
        out["dW2"].append((dYq.T @ Aq[i][:, u]) * dequant(sdy, sa))
        out["db1"].append(dPre[i][:, sel].sum(axis=0))
    return out


# ----------------------------------------------------------------------------
# the single layers in FP8 (the same readings F1-F5 applied to one
# ColumnParallelLinear or RowParallelLinear): the layer's input activation and
# weight are quantised E4M3 in the forward, its upstream gradient E5M2 in the
# backward, each with one scale over all its shards; current scaling.
# ----------------------------------------------------------------------------
def column_fwd_fp8(X, W_shards, b_shards, act: str):
    """ColumnParallelLinear + activation: pre_i = Xq Wq_i^T / (s_x s_w) + b_i,
    out_i = act(pre_i); pre and out stored in bf16.  X is the full [M, H]
    input.  Returns (pre list, out list), bf16 values as fp64."""
    (Xq,), sx = quantize([X], "e4m3")
    Wq, sw = quantize(W_shards, "e4m3")
    d = dequant(sx, sw)
    pre, out = [], []
    for i in range(len(Wq)):
        p = (Xq @ Wq[i].T) * d
        if b_shards is not None and b_shards[i] is not None:
            p = p + np.asarray(b_shards[i], np.float64)
        pre.append(round_bf16(p))
        out.append(round_bf16(_mlp.act_fwd(p, act)))
    return pre, out


def row_fwd_fp8(X_shards, W_shards, b=None, R=None):
    """RowParallelLinear: Y = (sum_i Xq_i Wq_i^T) / (s_x s_w) + b (+ R), the
    shard sum explicit in shard order, one scale over all shards of X and of
    W.  Returns Y in fp64 (before the bf16 store)."""
    Xq, sx = quantize(X_shards, "e4m3")
    Wq, sw = quantize(W_shards, "e4m3")
    Y = None
    for i in range(len(Wq)):
        part = Xq[i] @ Wq[i].T
        Y = part if Y is None else Y + part
    Y = Y * dequant(sx, sw)
    if b is not None:
        Y = Y + np.asarray(b, np.float64)
    if R is not None:
        Y = Y + np.asarray(R, np.float64)
    return Y


def column_bwd_fp8(dOut_shards, X, W_shards):
    """Backward of ColumnParallelLinear (no activation): dOut quantised E5M2
    over all shards, X and W as in the forward (E4M3):
    dX = (sum_i dOq_i Wq_i) / (s_do s_w), dW_i = dOq_i^T Xq / (s_do s_x),
    db_i = sum over tokens of the unquantised dOut_i (F5)."""
    (Xq,), sx = quantize([X], "e4m3")
    Wq, sw = quantize(W_shards, "e4m3")
    dOq, sdo = quantize(dOut_shards, "e5m2")
    dX = None
    for i in range(len(Wq)):
        part = dOq[i] @ Wq[i]
        dX = part if dX is None else dX + part
    dX = dX * dequant(sdo, sw)
    dW = [(dOq[i].T @ Xq) * dequant(sdo, sx) for i in range(len(Wq))]
    db = [np.asarray(d, np.float64).sum(axis=0) for d in dOut_shards]
    return dX, dW, db


def row_bwd_fp8(dY, X_shards, W_shards):
    """Backward of RowParallelLinear: dY quantised E5M2, X and W as in the
    forward (E4M3): dX_i = dYq Wq_i / (s_dy s_w), dW_i = dYq^T Xq_i /
    (s_dy s_x), db = sum over tokens of the unquantised dY (F5)."""
    Xq, sx = quantize(X_shards, "e4m3")
    Wq, sw = quantize(W_shards, "e4m3")
    (dYq,), sdy = quantize([dY], "e5m2")
    dX = [(dYq @ Wq[i]) * dequant(sdy, sw) for i in range(len(Wq))]
    dW = [(dYq.T @ Xq[i]) * dequant(sdy, sx) for i in range(len(Wq))]
    return dX, dW, np.asarray(dY, np.float64).sum(axis=0)


def column_sampled_fp8(rows, units, X, W_shards, dOut_shards):
    """column_fwd_fp8 (act none) and column_bwd_fp8 evaluated only at the
    given token rows (pre and dX) and at the given output units of every
    shard (``units[i]`` indexes [0, Fs): rows of dW_i); the per-tensor scales
    still come from the full tensors.  Returns {"pre": [...], "dX", "dW"}."""
    rows = np.asarray(rows)
    (Xq,), sx = quantize([X], "e4m3")
    Wq, sw = quantize(W_shards, "e4m3")
    dOq, sdo = quantize(dOut_shards, "e5m2")
    d = dequant(sx, sw)
    pre = [round_bf16((Xq[rows] @ Wq[i].T) * d) for i in range(len(Wq))]
    dX = sum(dOq[i][rows] @ Wq[i] for i in range(len(Wq))) * dequant(sdo, sw)
    dW = [(dOq[i][:, np.asarray(units[i])].T @ Xq) * dequant(sdo, sx) for i in range(len(Wq))]
    return {"pre": pre, "dX": dX, "dW": dW}


def row_sampled_fp8(rows, units, X_shards, W_shards, dY):
    """row_fwd_fp8 (no bias or residual) and row_bwd_fp8 evaluated only at
    the given token rows (Y and dX_i) and at the given input units of every
    shard (``units[i]`` indexes [0, Fs): columns of dW_i); the scales come
    from the full tensors.  Returns {"Y", "dX": [...], "dW": [...]}."""
    rows = np.asarray(rows)
    Xq, sx = quantize(X_shards, "e4m3")
    Wq, sw = quantize(W_shards, "e4m3")
    (dYq,), sdy = quantize([dY], "e5m2")
    Y = sum(Xq[i][rows] @ Wq[i].T for i in range(len(Wq))) * dequant(sx, sw)
    dX = [(dYq[rows] @ Wq[i]) * dequant(sdy, sw) for i in range(len(Wq))]
    dW = [(dYq.T @ Xq[i][:, np.asarray(units[i])]) * dequant(sdy, sx) for i in range(len(Wq))]
    return {"Y": Y, "dX": dX, "dW": dW}
