"""ctypes binding of libtpmlp (include/tp_mlp.h).

Argument marshalling only: every computation runs in the library's CUDA
kernels.  Besides turning torch tensors into the pointer arrays of the C ABI,
the binding checks what the C side cannot see from raw pointers -- each
buffer's device, dtype, contiguity and shape -- so that no kernel is ever
handed a buffer smaller than the descriptor implies.

There is no fallback: if the library is missing, :func:`lib` raises.
"""
from __future__ import annotations

import ctypes
import os

import torch

from . import build as _build

ACT = {"none": 0, "gelu_tanh": 1, "swiglu": 2}
DTYPE = {"f32": 0, "bf16": 1, "fp8": 2}
TORCH_DTYPE = {"f32": torch.float32, "bf16": torch.bfloat16, "fp8": torch.bfloat16}  # fp8: bf16 buffers
STATUS = {0: "TP_OK", 1: "TP_ERR_ARG", 2: "TP_ERR_SHAPE", 3: "TP_ERR_UNSUPPORTED", 4: "TP_ERR_CUDA",
          5: "TP_ERR_TIMEOUT"}
MAX_SHARDS = 16


class TpError(RuntimeError):
    def __init__(self, status: int, msg: str):
        super().__init__(f"{STATUS.get(status, status)}: {msg}")
        self.status = status


class Desc(ctypes.Structure):
    _fields_ = [("S", ctypes.c_int), ("B", ctypes.c_int), ("H", ctypes.c_int), ("F", ctypes.c_int),
                ("T", ctypes.c_int), ("act", ctypes.c_int), ("dtype", ctypes.c_int), ("has_bias", ctypes.c_int),
                ("residual", ctypes.c_int), ("seq_parallel", ctypes.c_int), ("wgrad_accumulate", ctypes.c_int)]


class LayerDesc(ctypes.Structure):
    _fields_ = [("mlp", Desc), ("dropout_p", ctypes.c_float), ("ln_eps", ctypes.c_float)]


class ProfEntry(ctypes.Structure):
    _fields_ = [("name", ctypes.c_char * 48), ("launches", ctypes.c_int), ("total_ms", ctypes.c_double),
                ("sm_cycles", ctypes.c_uint64), ("sm_ns", ctypes.c_uint64)]


_lib = None
VP = ctypes.c_void_p
PP = ctypes.POINTER(ctypes.c_void_p)

# exported symbol -> (restype, argtypes)
SIGNATURES = {
    "tp_abi_version": (ctypes.c_int, []),
    "tp_status_str": (ctypes.c_char_p, [ctypes.c_int]),
    "tp_last_error": (ctypes.c_char_p, []),
    "tp_mlp_create": (ctypes.c_int, [ctypes.POINTER(Desc), ctypes.POINTER(VP)]),
    "tp_mlp_destroy": (None, [VP]),
    "tp_mlp_workspace_bytes": (ctypes.c_size_t, [VP]),
    "tp_mlp_fwd": (ctypes.c_int, [VP, PP, PP, PP, PP, VP, PP, PP, PP, VP]),
    "tp_mlp_fwd_ws": (ctypes.c_int, [VP, PP, PP, PP, PP, VP, PP, PP, PP, VP, ctypes.c_size_t, VP]),
    "tp_mlp_set_fp8_history": (ctypes.c_int, [VP, ctypes.c_int]),
    "tp_mlp_fp8_amax": (ctypes.c_int, [VP, VP, ctypes.c_size_t, VP, VP]),
    "tp_layer_fp8_amax": (ctypes.c_int, [VP, VP, ctypes.c_size_t, VP, VP]),
    "tp_mlp_bwd": (ctypes.c_int, [VP, PP, PP, PP, PP, PP, PP, PP, PP, PP, PP, VP, VP, ctypes.c_size_t, VP]),
    "tp_linear_col": (ctypes.c_int, [ctypes.POINTER(Desc), PP, PP, PP, PP, PP, VP]),
    "tp_linear_row": (ctypes.c_int, [ctypes.POINTER(Desc), PP, PP, VP, PP, PP, VP]),
    "tp_linear_col_ws": (ctypes.c_int, [ctypes.POINTER(Desc), PP, PP, PP, PP, PP, VP, ctypes.c_size_t, VP]),
    "tp_linear_row_ws": (ctypes.c_int, [ctypes.POINTER(Desc), PP, PP, VP, PP, PP, VP, ctypes.c_size_t, VP]),
    "tp_linear_workspace_bytes": (ctypes.c_size_t, [ctypes.POINTER(Desc)]),
    "tp_linear_col_bwd": (ctypes.c_int, [ctypes.POINTER(Desc), PP, PP, PP, PP, PP, PP, VP, ctypes.c_size_t, VP]),
    "tp_linear_row_bwd": (ctypes.c_int, [ctypes.POINTER(Desc), PP, PP, PP, PP, PP, VP, VP, ctypes.c_size_t, VP]),
    "tp_linear_row_bwd_noalloc": (ctypes.c_int, [ctypes.POINTER(Desc), PP, PP, PP, PP, PP, VP, VP]),
    "tp_layer_create": (ctypes.c_int, [ctypes.POINTER(LayerDesc), ctypes.POINTER(VP)]),
    "tp_layer_destroy": (None, [VP]),
    "tp_layer_workspace_bytes": (ctypes.c_size_t, [VP]),
    "tp_layer_set_fp8_history": (ctypes.c_int, [VP, ctypes.c_int]),
    "tp_layer_fwd": (ctypes.c_int, [VP, PP, VP, VP, PP, PP, PP, VP, ctypes.c_uint64, PP, VP, VP, VP, PP, PP, VP,
                                    ctypes.c_size_t, VP]),
    "tp_layer_bwd": (ctypes.c_int, [VP, PP, PP, VP, VP, VP, VP, PP, PP, PP, PP, ctypes.c_uint64, PP, VP, VP, PP,
                                    PP, PP, VP, VP, ctypes.c_size_t, VP]),
    "tp_fp8_quantize": (ctypes.c_int, [PP, PP, ctypes.POINTER(ctypes.c_int64), ctypes.c_int, ctypes.c_int, VP, VP]),
    "tp_sync_status": (ctypes.c_int, [VP]),
    "tp_mlp_sync_status": (ctypes.c_int, [VP, VP]),
    "tp_layer_sync_status": (ctypes.c_int, [VP, VP]),
    "tp_mlp_debug_wait_timeout": (ctypes.c_int, [VP, ctypes.c_uint64, VP]),
    "tp_set_wait_limit_ns": (None, [ctypes.c_uint64]),
    "tp_debug_wait_timeout": (ctypes.c_int, [ctypes.c_uint64, VP]),
    "tp_launch_count": (ctypes.c_uint64, []),
    "tp_tail_split_count": (ctypes.c_uint64, []),
    "tp_set_tail_split": (ctypes.c_int, [ctypes.c_int]),
    "tp_set_max_gemm_pairs": (ctypes.c_int, [ctypes.c_int]),
    "tp_set_k_order": (ctypes.c_int, [ctypes.c_int]),
    "tp_set_band_rows": (ctypes.c_int, [ctypes.c_int]),
    "tp_set_launch_overlap": (ctypes.c_int, [ctypes.c_int]),
    "tp_set_tile_mode": (ctypes.c_int, [ctypes.c_int]),
    "tp_set_fused_fwd": (ctypes.c_int, [ctypes.c_int]),
    "tp_prof_enable": (None, [ctypes.c_int]),
    "tp_prof_collect": (ctypes.c_int, [ctypes.POINTER(ProfEntry), ctypes.c_int]),
    "tp_prof_select": (None, [ctypes.c_char_p]),
}


def library_path() -> str:
    return _build.LIB


def lib():
    """Load libtpmlp.so (raises if it has not been built)."""
    global _lib
    if _lib is None:
        path = library_path()
        if not os.path.exists(path):
            raise RuntimeError(f"{path} is missing: build it with __graft_entry__.build() "
                               "(the CUDA library is required; there is no fallback)")
        L = ctypes.CDLL(path)
        for name, (res, args) in SIGNATURES.items():
            f = getattr(L, name)
            f.restype = res
            f.argtypes = args
        _lib = L
    return _lib


def _check(status: int):
    if status != 0:
        raise TpError(status, lib().tp_last_error().decode(errors="replace"))


def _stream(stream):
    if stream is None:
        return VP(torch.cuda.current_stream().cuda_stream)
    if isinstance(stream, torch.cuda.Stream):
        return VP(stream.cuda_stream)
    return VP(int(stream))


def _arr(ptrs):
    """Host array of device pointers (None for a missing array)."""
    if ptrs is None:
        return None
    a = (VP * max(1, len(ptrs)))()
    for i, p in enumerate(ptrs):
        a[i] = p
    return ctypes.cast(a, PP)


class _Checker:
    def __init__(self, dtype: str):
        self.dt = TORCH_DTYPE[dtype]

    def tensors(self, name, ts, n, shape, dtype=None):
        dtype = dtype or self.dt
        if ts is None:
            raise ValueError(f"{name}: required")
        if isinstance(ts, torch.Tensor):
            ts = [ts]
        ts = list(ts)
        if len(ts) != n:
            raise ValueError(f"{name}: expected {n} tensors, got {len(ts)}")
        for i, t in enumerate(ts):
            if not isinstance(t, torch.Tensor) or not t.is_cuda:
                raise ValueError(f"{name}[{i}]: must be a CUDA tensor")
            if t.dtype != dtype:
                raise ValueError(f"{name}[{i}]: dtype {t.dtype}, expected {dtype}")
            if not t.is_contiguous():
                raise ValueError(f"{name}[{i}]: must be contiguous")
            if t.numel() != _prod(shape):
                raise ValueError(f"{name}[{i}]: {tuple(t.shape)} has {t.numel()} elements, expected {shape}")
        return [t.data_ptr() for t in ts]

    def optional(self, name, ts, n, shape, dtype=None):
        return None if ts is None else self.tensors(name, ts, n, shape, dtype)


def _prod(shape):
    p = 1
    for s in shape:
        p *= int(s)
    return p


def make_desc(S, B, H, F, T, act="gelu_tanh", dtype="bf16", has_bias=False, residual=False,
              seq_parallel=False, wgrad_accumulate=False) -> Desc:
    return Desc(int(S), int(B), int(H), int(F), int(T), ACT[act], DTYPE[dtype], int(bool(has_bias)),
                int(bool(residual)), int(bool(seq_parallel)), int(bool(wgrad_accumulate)))


class Layout:
    """Buffer shapes implied by a descriptor (see include/tp_mlp.h)."""

    def __init__(self, S, B, H, F, T, act="gelu_tanh", dtype="bf16", has_bias=False, residual=False,
                 seq_parallel=False, wgrad_accumulate=False):
        self.S, self.B, self.H, self.F, self.T = S, B, H, F, T
        self.act, self.dtype = act, dtype
        self.has_bias, self.residual = has_bias, residual
        self.seq_parallel, self.wgrad_accumulate = seq_parallel, wgrad_accumulate
        self.M = S * B
        self.g = 2 if act == "swiglu" else 1
        self.Fs = F // T if T else 0
        self.nx = T if seq_parallel else 1
        self.xrows = self.M // T if seq_parallel else self.M

    def desc(self) -> Desc:
        return make_desc(self.S, self.B, self.H, self.F, self.T, self.act, self.dtype, self.has_bias,
                         self.residual, self.seq_parallel, self.wgrad_accumulate)


class TPMLP(Layout):
    """Handle for one tensor-parallel MLP shape (tp_mlp_create)."""

    def __init__(self, *args, **kw):
        super().__init__(*args, **kw)
        self._d = self.desc()
        h = VP()
        _check(lib().tp_mlp_create(ctypes.byref(self._d), ctypes.byref(h)))
        self._h = h
        self._c = _Checker(self.dtype)

    def __del__(self):
        h = getattr(self, "_h", None)
        if h is not None and _lib is not None:
            _lib.tp_mlp_destroy(h)
            self._h = None

    def workspace_bytes(self) -> int:
        return int(lib().tp_mlp_workspace_bytes(self._h))

    def sync_status(self, stream=None) -> int:
        """Synchronise the stream and return (and clear) this handle's device
        status word (TP_ERR_TIMEOUT when one of its kernels' waits ran out)."""
        return int(lib().tp_mlp_sync_status(self._h, _stream(stream)))

    def debug_wait_timeout(self, limit_ns: int, stream=None):
        """A kernel that waits on a flag nothing sets, reporting its timeout to
        this handle's status word."""
        _check(lib().tp_mlp_debug_wait_timeout(self._h, int(limit_ns), _stream(stream)))

    def set_fp8_history(self, n: int):
        """FP8 delayed scaling over the last n amaxes of every operand (0:
        current scaling).  Clears the history; pass the same workspace to
        every later fwd / bwd."""
        _check(lib().tp_mlp_set_fp8_history(self._h, int(n)))

    FP8_AMAX_NAMES = ("X", "W1", "W2", "A", "dY", "dPre")

    def fp8_amax(self, workspace, stream=None):
        """The per-tensor amaxes the last fwd / bwd recorded in `workspace`, as
        a CUDA float32 tensor in the order of FP8_AMAX_NAMES (dtype "fp8")."""
        ws_ptr, ws_bytes = _workspace(workspace)
        out = torch.empty(len(self.FP8_AMAX_NAMES), dtype=torch.float32, device=workspace.device)
        _check(lib().tp_mlp_fp8_amax(self._h, ws_ptr, ws_bytes, out.data_ptr(), _stream(stream)))
        return out

    def fwd(self, X, W1, b1, W2, b2, Y, pre, A, stream=None, workspace=None):
        """Forward; `workspace` (required for dtype "fp8") must then be passed,
        unchanged, to the following bwd."""
        c, T, H, Fs, g = self._c, self.T, self.H, self.Fs, self.g
        px = c.tensors("X", X, self.nx, (self.xrows, H))
        pw1 = c.tensors("W1", W1, T, (g * Fs, H))
        pw2 = c.tensors("W2", W2, T, (H, Fs))
        pb1 = c.tensors("b1", b1, T, (g * Fs,)) if self.has_bias else None
        pb2 = c.tensors("b2", b2, 1, (H,))[0] if self.has_bias else None
        py = c.tensors("Y", Y, self.nx, (self.xrows, H))
        pp = c.optional("pre", pre, T, (self.M, g * Fs))
        pa = c.tensors("A", A, T, (self.M, Fs))
        if workspace is None:
            _check(lib().tp_mlp_fwd(self._h, _arr(px), _arr(pw1), _arr(pb1), _arr(pw2), pb2, _arr(py), _arr(pp),
                                    _arr(pa), _stream(stream)))
        else:
            ws_ptr, ws_bytes = _workspace(workspace, self.workspace_bytes())
            _check(lib().tp_mlp_fwd_ws(self._h, _arr(px), _arr(pw1), _arr(pb1), _arr(pw2), pb2, _arr(py),
                                       _arr(pp), _arr(pa), ws_ptr, ws_bytes, _stream(stream)))

    def bwd(self, dY, X, W1, W2, pre, A, dX, dW1, db1, dW2, db2, workspace, stream=None):
        c, T, H, Fs, g = self._c, self.T, self.H, self.Fs, self.g
        f32 = torch.float32
        pdy = c.tensors("dY", dY, self.nx, (self.xrows, H))
        px = c.tensors("X", X, self.nx, (self.xrows, H))
        pw1 = c.tensors("W1", W1, T, (g * Fs, H))
        pw2 = c.tensors("W2", W2, T, (H, Fs))
        pp = c.optional("pre", pre, T, (self.M, g * Fs))
        pa = c.tensors("A", A, T, (self.M, Fs))
        pdx = c.tensors("dX", dX, self.nx, (self.xrows, H))
        pdw1 = c.tensors("dW1", dW1, T, (g * Fs, H), f32)
        pdw2 = c.tensors("dW2", dW2, T, (H, Fs), f32)
        pdb1 = c.tensors("db1", db1, T, (g * Fs,), f32) if self.has_bias else None
        pdb2 = c.tensors("db2", db2, 1, (H,), f32)[0] if self.has_bias else None
        nws = self.workspace_bytes()
        ws_ptr, ws_bytes = _workspace(workspace, nws)
        _check(lib().tp_mlp_bwd(self._h, _arr(pdy), _arr(px), _arr(pw1), _arr(pw2), _arr(pp), _arr(pa),
                                _arr(pdx), _arr(pdw1), _arr(pdb1), _arr(pdw2), pdb2, ws_ptr, ws_bytes,
                                _stream(stream)))


class TPLayer(Layout):
    """Handle for the TransformerLayer MLP sub-block
    Y = X + dropout_p(MLP(LayerNorm(X))) (tp_layer_create).  The MLP keyword
    arguments are those of TPMLP (residual must stay False)."""

    def __init__(self, *args, dropout_p: float = 0.0, ln_eps: float = 1e-5, **kw):
        super().__init__(*args, **kw)
        self.dropout_p, self.ln_eps = float(dropout_p), float(ln_eps)
        self._d = LayerDesc(self.desc(), self.dropout_p, self.ln_eps)
        h = VP()
        _check(lib().tp_layer_create(ctypes.byref(self._d), ctypes.byref(h)))
        self._h = h
        self._c = _Checker(self.dtype)

    def __del__(self):
        h = getattr(self, "_h", None)
        if h is not None and _lib is not None:
            _lib.tp_layer_destroy(h)
            self._h = None

    def workspace_bytes(self) -> int:
        return int(lib().tp_layer_workspace_bytes(self._h))

    def sync_status(self, stream=None) -> int:
        """Synchronise the stream and return (and clear) this handle's device
        status word."""
        return int(lib().tp_layer_sync_status(self._h, _stream(stream)))

    FP8_AMAX_NAMES = ("X", "W1", "W2", "A", "dY", "dPre")

    def fp8_amax(self, workspace, stream=None):
        """The per-tensor amaxes of the MLP inside the block, as TPMLP.fp8_amax
        (X: the LayerNorm output, dY: the gradient at the MLP's output)."""
        ws_ptr, ws_bytes = _workspace(workspace)
        out = torch.empty(len(self.FP8_AMAX_NAMES), dtype=torch.float32, device=workspace.device)
        _check(lib().tp_layer_fp8_amax(self._h, ws_ptr, ws_bytes, out.data_ptr(), _stream(stream)))
        return out

    def set_fp8_history(self, n: int):
        """FP8 delayed scaling over the last n amaxes (0: current scaling); as
        TPMLP.set_fp8_history."""
        _check(lib().tp_layer_set_fp8_history(self._h, int(n)))

    def fwd(self, X, gamma, beta, W1, b1, W2, b2, seed, Y, Xn, mean, rstd, pre, A, workspace=None, stream=None):
        c, T, H, Fs, g, M = self._c, self.T, self.H, self.Fs, self.g, self.M
        f32 = torch.float32
        px = c.tensors("X", X, self.nx, (self.xrows, H))
        pg = c.tensors("gamma", gamma, 1, (H,))[0]
        pbt = c.tensors("beta", beta, 1, (H,))[0]
        pw1 = c.tensors("W1", W1, T, (g * Fs, H))
        pw2 = c.tensors("W2", W2, T, (H, Fs))
        pb1 = c.tensors("b1", b1, T, (g * Fs,)) if self.has_bias else None
        pb2 = c.tensors("b2", b2, 1, (H,))[0] if self.has_bias else None
        py = c.tensors("Y", Y, self.nx, (self.xrows, H))
        pxn = c.tensors("Xn", Xn, 1, (M, H))[0]
        pm = c.tensors("mean", mean, 1, (M,), f32)[0]
        pr = c.tensors("rstd", rstd, 1, (M,), f32)[0]
        pp = c.optional("pre", pre, T, (M, g * Fs))
        pa = c.tensors("A", A, T, (M, Fs))
        ws_ptr, ws_bytes = (None, 0) if workspace is None else _workspace(workspace, self.workspace_bytes())
        _check(lib().tp_layer_fwd(self._h, _arr(px), pg, pbt, _arr(pw1), _arr(pb1), _arr(pw2), pb2,
                                  int(seed) & (2 ** 64 - 1), _arr(py), pxn, pm, pr, _arr(pp), _arr(pa), ws_ptr,
                                  ws_bytes, _stream(stream)))

    def bwd(self, dY, X, gamma, Xn, mean, rstd, W1, W2, pre, A, seed, dX, dgamma, dbeta, dW1, db1, dW2, db2,
            workspace, stream=None):
        c, T, H, Fs, g, M = self._c, self.T, self.H, self.Fs, self.g, self.M
        f32 = torch.float32
        pdy = c.tensors("dY", dY, self.nx, (self.xrows, H))
        px = c.tensors("X", X, self.nx, (self.xrows, H))
        pg = c.tensors("gamma", gamma, 1, (H,))[0]
        pxn = c.tensors("Xn", Xn, 1, (M, H))[0]
        pm = c.tensors("mean", mean, 1, (M,), f32)[0]
        pr = c.tensors("rstd", rstd, 1, (M,), f32)[0]
        pw1 = c.tensors("W1", W1, T, (g * Fs, H))
        pw2 = c.tensors("W2", W2, T, (H, Fs))
        pp = c.optional("pre", pre, T, (M, g * Fs))
        pa = c.tensors("A", A, T, (M, Fs))
        pdx = c.tensors("dX", dX, self.nx, (self.xrows, H))
        pdg = c.tensors("dgamma", dgamma, 1, (H,), f32)[0]
        pdb = c.tensors("dbeta", dbeta, 1, (H,), f32)[0]
        pdw1 = c.tensors("dW1", dW1, T, (g * Fs, H), f32)
        pdw2 = c.tensors("dW2", dW2, T, (H, Fs), f32)
        pdb1 = c.tensors("db1", db1, T, (g * Fs,), f32) if self.has_bias else None
        pdb2 = c.tensors("db2", db2, 1, (H,), f32)[0] if self.has_bias else None
        ws_ptr, ws_bytes = _workspace(workspace, self.workspace_bytes())
        _check(lib().tp_layer_bwd(self._h, _arr(pdy), _arr(px), pg, pxn, pm, pr, _arr(pw1), _arr(pw2), _arr(pp),
                                  _arr(pa), int(seed) & (2 ** 64 - 1), _arr(pdx), pdg, pdb, _arr(pdw1), _arr(pdb1),
                                  _arr(pdw2), pdb2, ws_ptr, ws_bytes, _stream(stream)))


def _workspace(workspace, need=None):
    """(pointer, bytes) of a workspace tensor, (None, 0) for None.  The library
    checks the size: the part a call requires can be smaller than the queried
    size `need`, whose end is the optional tail-split scratch."""
    if workspace is None:
        return None, 0
    if not (isinstance(workspace, torch.Tensor) and workspace.is_cuda and workspace.is_contiguous()):
        raise ValueError("workspace must be a contiguous CUDA tensor")
    return workspace.data_ptr(), workspace.numel() * workspace.element_size()


def alloc_workspace(nbytes: int, device="cuda"):
    """A 256-byte aligned byte buffer (torch allocations are 512-aligned)."""
    return torch.empty(max(1, nbytes), dtype=torch.uint8, device=device)


# ---------------------------------------------------------------------------
# single layers
# ---------------------------------------------------------------------------
def linear_col(layout: Layout, X, W, b, out, pre=None, stream=None, workspace=None):
    """Column layer forward; with `workspace` (required for dtype "fp8",
    which then needs it, unchanged, in linear_col_bwd) tp_linear_col_ws."""
    c, T, H, Fs, g = _Checker(layout.dtype), layout.T, layout.H, layout.Fs, layout.g
    d = layout.desc()
    px = c.tensors("X", X, layout.nx, (layout.xrows, H))
    pw = c.tensors("W", W, T, (g * Fs, H))
    pb = c.tensors("b", b, T, (g * Fs,)) if layout.has_bias else None
    po = c.tensors("out", out, T, (layout.M, Fs))
    pp = c.optional("pre", pre, T, (layout.M, g * Fs))
    if workspace is None:
        _check(lib().tp_linear_col(ctypes.byref(d), _arr(px), _arr(pw), _arr(pb), _arr(po), _arr(pp),
                                   _stream(stream)))
    else:
        ws, nws = _workspace(workspace)
        _check(lib().tp_linear_col_ws(ctypes.byref(d), _arr(px), _arr(pw), _arr(pb), _arr(po), _arr(pp), ws, nws,
                                      _stream(stream)))


def linear_row(layout: Layout, X, W, b, R, Y, stream=None, workspace=None):
    """Row layer forward; with `workspace` (required for dtype "fp8", which
    then needs it, unchanged, in linear_row_bwd) tp_linear_row_ws."""
    c, T, H, Fs = _Checker(layout.dtype), layout.T, layout.H, layout.Fs
    d = layout.desc()
    px = c.tensors("X", X, T, (layout.M, Fs))
    pw = c.tensors("W", W, T, (H, Fs))
    pb = c.tensors("b", b, 1, (H,))[0] if layout.has_bias else None
    pr = c.tensors("R", R, layout.nx, (layout.xrows, H)) if layout.residual else None
    py = c.tensors("Y", Y, layout.nx, (layout.xrows, H))
    if workspace is None:
        _check(lib().tp_linear_row(ctypes.byref(d), _arr(px), _arr(pw), pb, _arr(pr), _arr(py), _stream(stream)))
    else:
        ws, nws = _workspace(workspace)
        _check(lib().tp_linear_row_ws(ctypes.byref(d), _arr(px), _arr(pw), pb, _arr(pr), _arr(py), ws, nws,
                                      _stream(stream)))


def linear_workspace_bytes(layout: Layout) -> int:
    d = layout.desc()
    return int(lib().tp_linear_workspace_bytes(ctypes.byref(d)))


def linear_col_bwd(layout: Layout, dOut, X, W, dX, dW, db, workspace=None, stream=None):
    c, T, H, Fs = _Checker(layout.dtype), layout.T, layout.H, layout.Fs
    f32 = torch.float32
    d = layout.desc()
    pdo = c.tensors("dOut", dOut, T, (layout.M, Fs))
    px = c.tensors("X", X, layout.nx, (layout.xrows, H))
    pw = c.tensors("W", W, T, (Fs, H))
    pdx = c.tensors("dX", dX, layout.nx, (layout.xrows, H))
    pdw = c.tensors("dW", dW, T, (Fs, H), f32)
    pdb = c.tensors("db", db, T, (Fs,), f32) if layout.has_bias else None
    ws, nws = _workspace(workspace, linear_workspace_bytes(layout))
    _check(lib().tp_linear_col_bwd(ctypes.byref(d), _arr(pdo), _arr(px), _arr(pw), _arr(pdx), _arr(pdw),
                                   _arr(pdb), ws, nws, _stream(stream)))


def linear_row_bwd(layout: Layout, dY, X, W, dX, dW, db, workspace=None, stream=None):
    c, T, H, Fs = _Checker(layout.dtype), layout.T, layout.H, layout.Fs
    f32 = torch.float32
    d = layout.desc()
    pdy = c.tensors("dY", dY, layout.nx, (layout.xrows, H))
    px = c.tensors("X", X, T, (layout.M, Fs))
    pw = c.tensors("W", W, T, (H, Fs))
    pdx = c.tensors("dX", dX, T, (layout.M, Fs))
    pdw = c.tensors("dW", dW, T, (H, Fs), f32)
    pdb = c.tensors("db", db, 1, (H,), f32)[0] if layout.has_bias else None
    ws, nws = _workspace(workspace, linear_workspace_bytes(layout))
    _check(lib().tp_linear_row_bwd(ctypes.byref(d), _arr(pdy), _arr(px), _arr(pw), _arr(pdx), _arr(pdw), pdb,
                                   ws, nws, _stream(stream)))


def linear_row_bwd_noalloc(layout: Layout, dY, X, W, dX, dW, db, stream=None):
    """tp_linear_row_bwd for callers that cannot allocate device memory: the
    bias-gradient scratch comes from a fixed 4 MiB array inside the library
    instead of a caller workspace (see include/tp_mlp.h for the limits and
    for why overlapping calls race)."""
    c, T, H, Fs = _Checker(layout.dtype), layout.T, layout.H, layout.Fs
    f32 = torch.float32
    d = layout.desc()
    pdy = c.tensors("dY", dY, layout.nx, (layout.xrows, H))
    px = c.tensors("X", X, T, (layout.M, Fs))
    pw = c.tensors("W", W, T, (H, Fs))
    pdx = c.tensors("dX", dX, T, (layout.M, Fs))
    pdw = c.tensors("dW", dW, T, (H, Fs), f32)
    pdb = c.tensors("db", db, 1, (H,), f32)[0] if layout.has_bias else None
    _check(lib().tp_linear_row_bwd_noalloc(ctypes.byref(d), _arr(pdy), _arr(px), _arr(pw), _arr(pdx), _arr(pdw),
                                           pdb, _stream(stream)))


FP8_FORMATS = {"e4m3": 0, "e5m2": 1}


def fp8_quantize(inputs, outputs, fmt: str, amax, stream=None):
    """Quantise one tensor split over bf16 buffers `inputs` into uint8 buffers
    `outputs` (same element counts) with one per-tensor scale; the amax lands
    in the one-element fp32 CUDA tensor `amax`."""
    inputs, outputs = list(inputs), list(outputs)
    if len(inputs) != len(outputs):
        raise ValueError("inputs and outputs differ in length")
    for a, b in zip(inputs, outputs):
        if not (a.is_cuda and b.is_cuda and a.is_contiguous() and b.is_contiguous()):
            raise ValueError("contiguous CUDA tensors required")
        if a.dtype != torch.bfloat16 or b.dtype != torch.uint8 or a.numel() != b.numel():
            raise ValueError("bf16 inputs and uint8 outputs of equal sizes required")
    if not (amax.is_cuda and amax.dtype == torch.float32 and amax.numel() >= 1):
        raise ValueError("amax must be a CUDA float32 tensor")
    n = (ctypes.c_int64 * len(inputs))(*[t.numel() for t in inputs])
    _check(lib().tp_fp8_quantize(_arr([t.data_ptr() for t in inputs]), _arr([t.data_ptr() for t in outputs]), n,
                                 len(inputs), FP8_FORMATS[fmt], amax.data_ptr(), _stream(stream)))


# ---------------------------------------------------------------------------
# status / diagnostics
# ---------------------------------------------------------------------------
def sync_status(stream=None) -> int:
    """Synchronise the stream and return (and clear) the status word of the
    calls without a handle (single layers, FP8 quantiser); MLP and sub-block
    handles report through their own sync_status()."""
    return int(lib().tp_sync_status(_stream(stream)))


def set_wait_limit_ns(ns: int):
    lib().tp_set_wait_limit_ns(int(ns))


def debug_wait_timeout(limit_ns: int, stream=None):
    _check(lib().tp_debug_wait_timeout(int(limit_ns), _stream(stream)))


TILE_MODES = {"auto": 0, "single": 1, "pair": 2}


def set_tile_mode(mode: str):
    """GEMM tiling of the bf16 engine: "auto", "single" (128-row tiles, one
    CTA) or "pair" (256-row tiles on a CTA pair)."""
    _check(lib().tp_set_tile_mode(TILE_MODES[mode]))


def set_tail_split(on: bool):
    """Tail split of the pair-tile GEMMs (on by default): the last,
    part-filled round of tiles is cut along K over all CTA pairs."""
    _check(lib().tp_set_tail_split(1 if on else 0))


def set_k_order(alternate: bool):
    """Every other persistent round of the pair GEMMs (row forward, column
    dgrad, weight gradients) walks K backwards (True, the default) so that
    it starts on what the previous round left in L2; False: always forwards."""
    _check(lib().tp_set_k_order(1 if alternate else 0))


def set_launch_overlap(on: bool):
    """Programmatic dependent launch of the pair GEMMs (on by default): a
    GEMM's CTAs set up while the previous kernel finishes and wait for it
    before touching memory; False: plain stream order."""
    _check(lib().tp_set_launch_overlap(1 if on else 0))


def set_band_rows(rows: int):
    """Rows of 256-row tiles per raster band of the pair GEMMs' tile order
    (0: the library's choice)."""
    _check(lib().tp_set_band_rows(int(rows)))


def set_max_gemm_pairs(n: int):
    """Upper bound on the CTA pairs of the pair-tile GEMMs (0: all that fit)."""
    _check(lib().tp_set_max_gemm_pairs(int(n)))


def tail_split_count() -> int:
    """GEMM launches since load that split their last round's tiles."""
    return int(lib().tp_tail_split_count())


FUSED_MODES = {"auto": 0, "off": 1, "on": 2}


def set_fused_fwd(mode: str):
    """Forward as one fused kernel for narrow bf16 MLPs (H <= 256): "auto"
    (default) and "on" run it whenever the shape allows it (it measures faster
    than the two GEMMs there), "off" runs the column and row GEMM kernels;
    see include/tp_mlp.h."""
    _check(lib().tp_set_fused_fwd(FUSED_MODES[mode]))


def launch_count() -> int:
    return int(lib().tp_launch_count())


def prof_enable(on: bool = True):
    lib().tp_prof_enable(1 if on else 0)


def prof_select(kernel=None):
    """Time only the launches of `kernel` with events (None: every launch);
    the GEMMs' clock counters keep counting for all kernels."""
    lib().tp_prof_select(kernel.encode() if kernel else None)


def prof_collect(clocks: bool = False):
    """{kernel name: (launches, total device ms)} since the last collect;
    with clocks=True {name: (launches, total ms, SM cycles, SM ns)}, the last
    two summed over the CTAs of GEMM launches (0 for other kernels)."""
    buf = (ProfEntry * 64)()
    n = lib().tp_prof_collect(buf, 64)
    if n < 0:
        raise TpError(4, lib().tp_last_error().decode(errors="replace"))
    if clocks:
        return {buf[i].name.decode(): (buf[i].launches, buf[i].total_ms, buf[i].sm_cycles, buf[i].sm_ns)
                for i in range(n)}
    return {buf[i].name.decode(): (buf[i].launches, buf[i].total_ms) for i in range(n)}


def status_str(s: int) -> str:
    return lib().tp_status_str(int(s)).decode()
