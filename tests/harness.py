"""Helpers shared by the parity tests: build seeded inputs, shard them with the
oracle's shard layout, upload them, run the CUDA library through the C ABI and
compare element by element with the oracle."""
from __future__ import annotations

import numpy as np
import torch

import oracle
import synth

TOL = {"f32": 1e-5, "bf16": 1e-2}


def status_ok(tp, *handles) -> bool:
    """Synchronise and read (clearing them) the status word of the calls
    without a handle and the words of the given MLP / sub-block handles:
    True when none of them recorded a device-side error."""
    ok = tp.sync_status() == 0
    for h in handles:
        ok = (h.sync_status() == 0) and ok
    return ok


def rel_err(gpu, ref) -> float:
    """max |gpu - ref| / max |ref| over all elements (fp64)."""
    g = np.asarray(gpu, dtype=np.float64)
    r = np.asarray(ref, dtype=np.float64)
    assert g.shape == r.shape, (g.shape, r.shape)
    if r.size == 0:
        return 0.0
    den = np.max(np.abs(r))
    return float(np.max(np.abs(g - r)) / (den if den > 0 else 1.0))


def host(t: torch.Tensor) -> np.ndarray:
    return t.detach().float().cpu().numpy()


def dev(a, dtype: str, device="cuda"):
    td = torch.float32 if dtype == "f32" else torch.bfloat16
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32)).to(device=device, dtype=td)


def mlp_inputs(M, H, F, T, act, dtype, has_bias=True, bias_std=0.02, seed_off=0, x_std=1.0, w_std=0.02):
    """Seeded full tensors (synth) and their shards (oracle layout)."""
    g = 2 if act == "swiglu" else 1
    rnd = (lambda a: a) if dtype == "f32" else synth.round_bf16
    base = synth.SEED_BASE + 1000 * seed_off
    t = {
        "X": rnd(synth.normal(base + synth.TID_X, (M, H), x_std)),
        "W1": rnd(synth.normal(base + synth.TID_W1, (g * F, H), w_std)),
        "W2": rnd(synth.normal(base + synth.TID_W2, (H, F), w_std)),
        "dY": rnd(synth.normal(base + synth.TID_DY, (M, H), 1.0)),
        "b1": rnd(synth.normal(base + synth.TID_B1, (g * F,), bias_std)) if has_bias else None,
        "b2": rnd(synth.normal(base + synth.TID_B2, (H,), bias_std)) if has_bias else None,
    }
    t["W1s"] = [np.ascontiguousarray(w) for w in oracle.shard_column_weight(t["W1"], T, act)]
    t["b1s"] = [np.ascontiguousarray(b) for b in oracle.shard_column_bias(t["b1"], T, act)] if has_bias else None
    t["W2s"] = [np.ascontiguousarray(w) for w in oracle.shard_row_weight(t["W2"], T)]
    return t


def split_tokens(a, T, sp):
    return [np.ascontiguousarray(x) for x in oracle.sp_split(a, T)] if sp else [a]


class MlpRun:
    """Device buffers + one fwd/bwd of the library for a layout and inputs."""

    def __init__(self, lay, t, device="cuda"):
        import tensor_transformer_mlp_shard_gb300 as tp
        self.tp, self.lay, self.t = tp, lay, t
        dt = lay.dtype
        T, M, H, Fs, g = lay.T, lay.M, lay.H, lay.Fs, lay.g
        sp = lay.seq_parallel
        self.X = [dev(x, dt) for x in split_tokens(t["X"], T, sp)]
        self.dY = [dev(x, dt) for x in split_tokens(t["dY"], T, sp)]
        self.W1 = [dev(w, dt) for w in t["W1s"]]
        self.W2 = [dev(w, dt) for w in t["W2s"]]
        self.b1 = [dev(b, dt) for b in t["b1s"]] if lay.has_bias else None
        self.b2 = dev(t["b2"], dt) if lay.has_bias else None
        td = torch.float32 if dt == "f32" else torch.bfloat16
        rows = lay.xrows
        self.Y = [torch.full((rows, H), float("nan"), dtype=td, device=device) for _ in range(lay.nx)]
        self.dX = [torch.full((rows, H), float("nan"), dtype=td, device=device) for _ in range(lay.nx)]
        self.pre = [torch.full((M, g * Fs), float("nan"), dtype=td, device=device) for _ in range(T)]
        self.A = [torch.full((M, Fs), float("nan"), dtype=td, device=device) for _ in range(T)]
        f32 = torch.float32
        self.dW1 = [torch.full((g * Fs, H), float("nan"), dtype=f32, device=device) for _ in range(T)]
        self.dW2 = [torch.full((H, Fs), float("nan"), dtype=f32, device=device) for _ in range(T)]
        self.db1 = [torch.full((g * Fs,), float("nan"), dtype=f32, device=device) for _ in range(T)] \
            if lay.has_bias else None
        self.db2 = torch.full((H,), float("nan"), dtype=f32, device=device) if lay.has_bias else None
        self.ws = tp.alloc_workspace(lay.workspace_bytes()) if isinstance(lay, tp.TPMLP) else None

    def fwd(self, with_workspace=True):
        """tp_mlp_fwd_ws with the run's workspace (for bf16 it holds only the
        scratch of the row GEMM's tail split and of the fused forward's even
        split), or plain tp_mlp_fwd."""
        ws = self.ws if with_workspace or self.lay.dtype == "fp8" else None
        self.lay.fwd(self.X, self.W1, self.b1, self.W2, self.b2, self.Y, self.pre, self.A, workspace=ws)

    def bwd(self):
        self.lay.bwd(self.dY, self.X, self.W1, self.W2, self.pre, self.A, self.dX, self.dW1, self.db1,
                     self.dW2, self.db2, self.ws)

    def gathered(self, bufs):
        return np.concatenate([host(b) for b in bufs], axis=0)


def oracle_full(lay, t):
    """Full fp64 oracle of the MLP on the same (sharded) inputs."""
    pre, A, Y = oracle.mlp_fwd(t["X"], t["W1s"], t["b1s"], t["W2s"], t["b2"], lay.act, lay.residual)
    g = oracle.mlp_bwd(t["dY"], t["X"], t["W1s"], t["W2s"], pre, A, lay.act, lay.residual)
    g.update(pre=pre, A=A, Y=Y)
    return g
