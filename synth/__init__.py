"""Seeded synthetic inputs for the tensor-parallel MLP.

This module is shared by the CPU oracle and the CUDA path and holds none of
the MLP's arithmetic.  It draws full (unsharded) tensors from a counter-based
generator (SplitMix64 output function + Box-Muller, see ``synth.c``) and
rounds them to bf16 with round-to-nearest-even.  Splitting the tensors into
shards is left to the callers.

Workload recipes (shapes, distributions, seeds) for the five measured problems
are in :data:`WORKLOADS`.  Every tensor of a workload has its own seed,
``SEED_BASE + tensor id``.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import tempfile
from dataclasses import dataclass, field

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "synth.c")
_LIB = os.path.join(_HERE, "libtpsynth.so")
_lib = None

SEED_BASE = 20261202

# tensor ids (seed = SEED_BASE + id)
TID_X, TID_W1, TID_B1, TID_W2, TID_B2, TID_DY = 1, 2, 3, 4, 5, 6
TID_Z, TID_DY_QKV, TID_DY_O, TID_WQKV, TID_WO = 7, 8, 9, 10, 11
TID_GAMMA, TID_BETA, TID_ROW_SHIFT, TID_ROW_SCALE = 12, 13, 14, 15


def build(force: bool = False) -> str:
    """Compile synth.c into libtpsynth.so (gcc, OpenMP) if missing or stale."""
    if (not force and os.path.exists(_LIB)
            and os.path.getmtime(_LIB) >= os.path.getmtime(_SRC)):
        return _LIB
    fd, tmp = tempfile.mkstemp(suffix=".so", dir=_HERE)
    os.close(fd)
    cmd = ["gcc", "-O2", "-fPIC", "-shared", "-fopenmp", "-o", tmp, _SRC, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    if _lib is None:
        lib = ctypes.CDLL(build())
        lib.synth_normal_f32.argtypes = [ctypes.c_uint64, ctypes.c_int64, ctypes.c_int64,
                                         ctypes.c_double, ctypes.c_double, ctypes.c_void_p]
        lib.synth_normal_f32.restype = None
        lib.synth_f32_to_bf16.argtypes = [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int64]
        lib.synth_f32_to_bf16.restype = None
        lib.synth_bf16_to_f32.argtypes = [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int64]
        lib.synth_bf16_to_f32.restype = None
        lib.synth_num_threads.argtypes = []
        lib.synth_num_threads.restype = ctypes.c_int
        _lib = lib
    return _lib


def normal(seed: int, shape, std: float = 1.0, mean: float = 0.0, offset: int = 0) -> np.ndarray:
    """fp32 array of N(mean, std^2) draws; element i uses counter offset + i."""
    shape = tuple(int(s) for s in shape)
    out = np.empty(shape, dtype=np.float32)
    n = out.size
    if n:
        _load().synth_normal_f32(ctypes.c_uint64(seed & (2**64 - 1)), offset, n,
                                 float(mean), float(std), out.ctypes.data)
    return out


def to_bf16_bits(a: np.ndarray) -> np.ndarray:
    """Round an fp32 array to bf16 (RNE); returns the bit patterns as uint16."""
    a = np.ascontiguousarray(a, dtype=np.float32)
    out = np.empty(a.shape, dtype=np.uint16)
    if a.size:
        _load().synth_f32_to_bf16(a.ctypes.data, out.ctypes.data, a.size)
    return out


def bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    """Widen bf16 bit patterns (uint16) to fp32 exactly."""
    b = np.ascontiguousarray(b, dtype=np.uint16)
    out = np.empty(b.shape, dtype=np.float32)
    if b.size:
        _load().synth_bf16_to_f32(b.ctypes.data, out.ctypes.data, b.size)
    return out


def round_bf16(a: np.ndarray) -> np.ndarray:
    """fp32 values exactly representable in bf16 (RNE of ``a``)."""
    return bf16_bits_to_f32(to_bf16_bits(a))


def num_threads() -> int:
    return int(_load().synth_num_threads())


@dataclass(frozen=True)
class Workload:
    """Shapes and input distributions of one measured problem.

    M = S*B tokens stored row-major as [S, B, H] (token m = s*B + b).  ``kind``
    is ``"mlp"`` (column -> activation -> row) or ``"attn_proj"`` (QKV column
    layer with no activation plus the output row layer, fed an independent
    input Z)."""
    name: str
    kind: str
    S: int
    B: int
    H: int
    F: int
    T: int
    act: str          # "gelu_tanh" | "swiglu" | "none"
    dtype: str        # "f32" | "bf16" | "fp8" (bf16 buffers, FP8 products)
    has_bias: bool
    bias_std: float
    residual: bool
    seq_parallel: bool
    x_std: float = 1.0
    w_std: float = 0.02
    dy_std: float = 1.0
    F_o: int = 0      # attn_proj: input width of the output projection
    notes: str = ""
    extra: dict = field(default_factory=dict)

    @property
    def M(self) -> int:
        return self.S * self.B

    @property
    def g(self) -> int:
        return 2 if self.act == "swiglu" else 1

    def flops(self) -> float:
        """Algorithmic fwd+bwd FLOP (multiply-add = 2), elementwise excluded."""
        M, H = self.M, self.H
        if self.kind == "attn_proj":
            return 3.0 * (2.0 * M * H * self.F + 2.0 * M * self.F_o * H)
        return 3.0 * (2.0 * M * H * self.F * self.g + 2.0 * M * self.F * H)


WORKLOADS = {
    "tiny": Workload("tiny", "mlp", S=128, B=2, H=256, F=1024, T=2, act="gelu_tanh",
                     dtype="f32", has_bias=True, bias_std=0.0, residual=False,
                     seq_parallel=False, notes="biases present and zero"),
    "gpt": Workload("gpt", "mlp", S=2048, B=4, H=4096, F=16384, T=8, act="gelu_tanh",
                    dtype="bf16", has_bias=True, bias_std=0.02, residual=True,
                    seq_parallel=False),
    "attn_proj": Workload("attn_proj", "attn_proj", S=4096, B=2, H=4096, F=3 * 4096, T=8,
                          act="none", dtype="bf16", has_bias=False, bias_std=0.0,
                          residual=False, seq_parallel=False, F_o=4096,
                          notes="QKV 32 heads x 128 split over T=8; O projection 4096->4096"),
    "swiglu": Workload("swiglu", "mlp", S=4096, B=1, H=8192, F=28672, T=8, act="swiglu",
                       dtype="bf16", has_bias=False, bias_std=0.0, residual=False,
                       seq_parallel=False),
    "narrow": Workload("narrow", "mlp", S=4096, B=16, H=256, F=1024, T=2, act="gelu_tanh",
                       dtype="bf16", has_bias=True, bias_std=0.02, residual=True,
                       seq_parallel=False,
                       notes="the tiny configuration's widths in bf16 with 65536 tokens: a memory-bound MLP"),
    "narrow_swiglu": Workload("narrow_swiglu", "mlp", S=4096, B=16, H=256, F=1024, T=2, act="swiglu",
                              dtype="bf16", has_bias=True, bias_std=0.02, residual=True,
                              seq_parallel=False,
                              notes="the narrow workload with a SwiGLU activation (gate and up rows in W1)"),
    "sp": Workload("sp", "mlp", S=4096, B=4, H=6144, F=24576, T=8, act="gelu_tanh",
                   dtype="bf16", has_bias=False, bias_std=0.0, residual=False,
                   seq_parallel=True, notes="input/output stored as 8 shards [512,4,6144]"),
}


def mlp_tensors(w: Workload, M: int | None = None):
    """Full (unsharded) fp32 tensors of an MLP workload, rounded to bf16 when
    the workload is bf16.  W1 is [g*F, H] (for SwiGLU: gate rows then up
    rows), W2 is [H, F], X and dY are [M, H].  Biases are None when absent."""
    M = w.M if M is None else M
    g = w.g
    rnd = (lambda a: a) if w.dtype == "f32" else round_bf16
    t = {
        "X": rnd(normal(SEED_BASE + TID_X, (M, w.H), w.x_std)),
        "W1": rnd(normal(SEED_BASE + TID_W1, (g * w.F, w.H), w.w_std)),
        "W2": rnd(normal(SEED_BASE + TID_W2, (w.H, w.F), w.w_std)),
        "dY": rnd(normal(SEED_BASE + TID_DY, (M, w.H), w.dy_std)),
        "b1": None,
        "b2": None,
    }
    if w.has_bias:
        t["b1"] = rnd(normal(SEED_BASE + TID_B1, (g * w.F,), w.bias_std)) if w.bias_std else np.zeros(g * w.F, np.float32)
        t["b2"] = rnd(normal(SEED_BASE + TID_B2, (w.H,), w.bias_std)) if w.bias_std else np.zeros(w.H, np.float32)
    return t


def attn_tensors(w: Workload, M: int | None = None):
    """Full fp32 (bf16-rounded) tensors of the attention-projection workload:
    X [M,H], Wqkv [F,H], Z [M,F_o] (the attention core's output, drawn
    independently), Wo [H,F_o], upstream gradients dYqkv [M,F] and dYo [M,H]."""
    M = w.M if M is None else M
    rnd = round_bf16 if w.dtype == "bf16" else (lambda a: a)
    return {
        "X": rnd(normal(SEED_BASE + TID_X, (M, w.H), w.x_std)),
        "Wqkv": rnd(normal(SEED_BASE + TID_WQKV, (w.F, w.H), w.w_std)),
        "Z": rnd(normal(SEED_BASE + TID_Z, (M, w.F_o), w.x_std)),
        "Wo": rnd(normal(SEED_BASE + TID_WO, (w.H, w.F_o), w.w_std)),
        "dYqkv": rnd(normal(SEED_BASE + TID_DY_QKV, (M, w.F), w.dy_std)),
        "dYo": rnd(normal(SEED_BASE + TID_DY_O, (M, w.H), w.dy_std)),
    }


def layer_tensors(M: int, H: int, dtype: str, seed_off: int = 0):
    """LayerNorm parameters and a residual-stream-like input for the
    TransformerLayer MLP sub-block: gamma ~ 1 + 0.1 N(0,1), beta ~ 0.05 N(0,1)
    ([H]), and X [M, H] whose rows have their own offset (N(0,1)) and scale
    (0.5 + |N(0,1)|) around a N(0,1) body, so that the LayerNorm's mean and
    variance differ per token.  Rounded to bf16 unless dtype is "f32"."""
    rnd = (lambda a: a) if dtype == "f32" else round_bf16
    base = SEED_BASE + 1000 * seed_off
    shift = normal(base + TID_ROW_SHIFT, (M, 1), 1.0)
    scale = 0.5 + np.abs(normal(base + TID_ROW_SCALE, (M, 1), 1.0))
    X = normal(base + TID_X, (M, H), 1.0) * scale + shift
    return {
        "X": rnd(X.astype(np.float32)),
        "gamma": rnd(normal(base + TID_GAMMA, (H,), 0.1, mean=1.0)),
        "beta": rnd(normal(base + TID_BETA, (H,), 0.05)),
    }
