"""Host-side checks of the C ABI (no GPU): the library loads, exports every
symbol include/tp_mlp.h declares, and rejects bad descriptors and pointers
before anything is enqueued."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "tp_mlp.h")


@pytest.fixture(scope="module")
def tp():
    from tensor_transformer_mlp_shard_gb300 import build
    build.build()
    import tensor_transformer_mlp_shard_gb300 as tp
    return tp


def declared_symbols():
    names = []
    for path in (HEADER,):
        with open(path) as f:
            for line in f:
                m = re.match(r"^TP_API\s+[\w\s\*]+?\b(tp_\w+)\(", line)
                if m:
                    names.append(m.group(1))
    return names


def test_every_declared_symbol_is_exported(tp):
    names = declared_symbols()
    assert len(names) >= 19
    L = ctypes.CDLL(tp.library_path())
    for n in names:
        assert hasattr(L, n), n
    # and the binding knows every one of them
    from tensor_transformer_mlp_shard_gb300.binding import SIGNATURES
    assert set(names) == set(SIGNATURES)


def test_abi_version_and_status_strings(tp):
    L = tp.lib()
    assert L.tp_abi_version() == 1
    assert L.tp_status_str(0) == b"TP_OK"
    assert L.tp_status_str(2) == b"TP_ERR_SHAPE"
    assert L.tp_status_str(5) == b"TP_ERR_TIMEOUT"


def test_gemm_setting_validation(tp):
    L = tp.lib()
    assert L.tp_set_tail_split(2) == 1 and L.tp_set_tail_split(-1) == 1
    assert L.tp_set_max_gemm_pairs(-1) == 1
    assert L.tp_set_k_order(2) == 1 and L.tp_set_k_order(-1) == 1
    assert L.tp_set_k_order(0) == 0 and L.tp_set_k_order(1) == 0
    assert L.tp_set_band_rows(-1) == 1 and L.tp_set_band_rows(5000) == 1
    assert L.tp_set_band_rows(16) == 0 and L.tp_set_band_rows(0) == 0
    assert L.tp_set_launch_overlap(2) == 1 and L.tp_set_launch_overlap(-1) == 1
    assert L.tp_set_launch_overlap(0) == 0 and L.tp_set_launch_overlap(1) == 0
    assert L.tp_set_tail_split(0) == 0 and L.tp_set_tail_split(1) == 0
    assert L.tp_set_max_gemm_pairs(4) == 0 and L.tp_set_max_gemm_pairs(0) == 0
    assert L.tp_tail_split_count() == 0  # nothing launched on a host without a GPU


def _create(tp, **kw):
    base = dict(S=128, B=2, H=256, F=1024, T=2, act="gelu_tanh", dtype="bf16")
    base.update(kw)
    d = tp.make_desc(**base)
    h = ctypes.c_void_p()
    s = tp.lib().tp_mlp_create(ctypes.byref(d), ctypes.byref(h))
    if s == 0:
        tp.lib().tp_mlp_destroy(h)
    return s


@pytest.mark.parametrize("kw,expect", [
    ({}, 0),
    ({"F": 1000, "T": 3}, 2),           # divide(): F % T != 0
    ({"T": 0}, 2),
    ({"T": 17}, 2),
    ({"H": 260}, 2),                    # H % 8
    ({"F": 1028, "T": 2}, 2),           # F/T = 514, not a multiple of 8
    ({"S": 100, "T": 8, "F": 1024, "seq_parallel": True}, 2),   # S % T
    ({"S": 8 * 100, "B": 1, "T": 8, "F": 1024, "seq_parallel": True}, 2),  # bf16 SP: M/T % 128
    ({"S": 8 * 100, "B": 1, "T": 8, "F": 1024, "seq_parallel": True, "dtype": "f32"}, 0),
    ({"S": 0}, 0),                      # empty problem is valid
    ({"act": "swiglu"}, 0),
])
def test_create_validation(tp, kw, expect):
    assert _create(tp, **kw) == expect


def test_bad_enum_and_flags(tp):
    d = tp.make_desc(128, 2, 256, 1024, 2)
    d.act = 7
    h = ctypes.c_void_p()
    assert tp.lib().tp_mlp_create(ctypes.byref(d), ctypes.byref(h)) == 1
    d = tp.make_desc(128, 2, 256, 1024, 2)
    d.residual = 2
    assert tp.lib().tp_mlp_create(ctypes.byref(d), ctypes.byref(h)) == 1
    assert tp.lib().tp_mlp_create(None, ctypes.byref(h)) == 1


def test_null_and_misaligned_pointers_rejected_before_launch(tp):
    L = tp.lib()
    d = tp.make_desc(128, 2, 256, 1024, 2, act="gelu_tanh", dtype="bf16")
    h = ctypes.c_void_p()
    assert L.tp_mlp_create(ctypes.byref(d), ctypes.byref(h)) == 0
    from tensor_transformer_mlp_shard_gb300.binding import _arr
    good = [0x10000 * (i + 1) for i in range(2)]
    # X array missing
    assert L.tp_mlp_fwd(h, None, _arr(good), None, _arr(good), None, _arr(good[:1]), _arr(good), _arr(good),
                        None) == 1
    # misaligned W1[1]
    bad = [0x10000, 0x20008]
    assert L.tp_mlp_fwd(h, _arr(good[:1]), _arr(bad), None, _arr(good), None, _arr(good[:1]), _arr(good),
                        _arr(good), None) == 1
    assert b"W1[1]" in L.tp_last_error()
    # workspace too small
    ws_need = L.tp_mlp_workspace_bytes(h)
    assert ws_need >= 2 * 256 * 512 * 2
    assert L.tp_mlp_bwd(h, _arr(good[:1]), _arr(good[:1]), _arr(good), _arr(good), _arr(good), _arr(good),
                        _arr(good[:1]), _arr(good), None, _arr(good), None, ctypes.c_void_p(0x100000), 16,
                        None) == 1
    assert b"workspace" in L.tp_last_error()
    L.tp_mlp_destroy(h)


def test_fp8_amax_validation(tp):
    """tp_mlp_fp8_amax rejects a NULL handle or out, a non-FP8 handle and a
    workspace too small for the FP8 region, before any copy."""
    L = tp.lib()
    out = ctypes.c_void_p(0x10000)
    assert L.tp_mlp_fp8_amax(None, ctypes.c_void_p(0x100000), 1 << 30, out, None) == 1
    assert L.tp_layer_fp8_amax(None, ctypes.c_void_p(0x100000), 1 << 30, out, None) == 1
    for dtype, expect_msg in (("bf16", b"TP_DT_FP8"), ("fp8", b"workspace")):
        d = tp.make_desc(128, 2, 256, 1024, 2, act="gelu_tanh", dtype=dtype)
        h = ctypes.c_void_p()
        assert L.tp_mlp_create(ctypes.byref(d), ctypes.byref(h)) == 0
        assert L.tp_mlp_fp8_amax(h, ctypes.c_void_p(0x100000), 256, None, None) == 1
        assert L.tp_mlp_fp8_amax(h, ctypes.c_void_p(0x100000), 256, out, None) == 1
        assert expect_msg in L.tp_last_error()
        L.tp_mlp_destroy(h)


def test_linear_col_bwd_rejects_activation(tp):
    from tensor_transformer_mlp_shard_gb300.binding import _arr
    L = tp.lib()
    d = tp.make_desc(128, 2, 256, 1024, 2, act="gelu_tanh")
    p = [0x10000, 0x20000]
    assert L.tp_linear_col_bwd(ctypes.byref(d), _arr(p), _arr(p[:1]), _arr(p), _arr(p[:1]), _arr(p), None,
                               None, 0, None) == 3


def test_workspace_sizes(tp):
    # dPre (T * M * g*Fs * 2 bytes, each shard 256-aligned) + bias partials
    lay = tp.Layout(S=2048, B=4, H=4096, F=16384, T=8, act="gelu_tanh", dtype="bf16", has_bias=True)
    d = lay.desc()
    h = ctypes.c_void_p()
    L = tp.lib()
    assert L.tp_mlp_create(ctypes.byref(d), ctypes.byref(h)) == 0
    tp.set_tail_split(False)
    ws = L.tp_mlp_workspace_bytes(h)
    tp.set_tail_split(True)
    dpre = 8 * 8192 * 2048 * 2
    # db1 partials: one fp32 row of column sums per 32-token block and shard
    partials = 4 * 8 * (8192 // 32) * 2048
    assert ws == dpre + partials
    # the tail-split scratch (sized from the device's SM count) only adds at the end
    assert L.tp_mlp_workspace_bytes(h) >= ws
    L.tp_mlp_destroy(h)
    lay2 = tp.Layout(S=2048, B=4, H=4096, F=16384, T=8, act="none", has_bias=False)
    assert tp.linear_workspace_bytes(lay2) == 0


def _layer_create(tp, p=0.1, eps=1e-5, **kw):
    from tensor_transformer_mlp_shard_gb300.binding import LayerDesc
    base = dict(S=128, B=2, H=256, F=1024, T=2, act="gelu_tanh", dtype="bf16")
    base.update(kw)
    d = LayerDesc(tp.make_desc(**base), p, eps)
    h = ctypes.c_void_p()
    s = tp.lib().tp_layer_create(ctypes.byref(d), ctypes.byref(h))
    ws = 0
    if s == 0:
        ws = tp.lib().tp_layer_workspace_bytes(h)
        tp.lib().tp_layer_destroy(h)
    return s, ws


@pytest.mark.parametrize("kw,expect", [
    ({}, 0),
    ({"p": 0.0}, 0),
    ({"p": 0.999}, 0),
    ({"p": 1.0}, 1),                      # dropout probability outside [0, 1)
    ({"p": -0.1}, 1),
    ({"p": float("nan")}, 1),
    ({"eps": 0.0}, 1),
    ({"residual": True}, 1),              # the block adds X itself
    ({"H": 8192}, 0),
    ({"H": 8200}, 3),                     # above the LayerNorm kernels' row capacity (bf16)
    ({"H": 4096, "dtype": "f32"}, 0),
    ({"H": 4104, "dtype": "f32"}, 3),
    ({"F": 1000, "T": 3}, 2),             # the MLP's own shape checks still apply
    ({"dtype": "fp8"}, 0),
])
def test_layer_create_validation(tp, kw, expect):
    assert _layer_create(tp, **kw)[0] == expect


def test_layer_workspace_holds_mlp_workspace_dz_and_dxn(tp):
    s, ws = _layer_create(tp)
    assert s == 0
    d = tp.make_desc(128, 2, 256, 1024, 2, act="gelu_tanh", dtype="bf16")
    h = ctypes.c_void_p()
    assert tp.lib().tp_mlp_create(ctypes.byref(d), ctypes.byref(h)) == 0
    mlp_ws = tp.lib().tp_mlp_workspace_bytes(h)
    tp.lib().tp_mlp_destroy(h)
    M, H = 256, 256
    assert ws >= mlp_ws + 2 * M * H * 2
    # M = 0: nothing but alignment padding
    s0, ws0 = _layer_create(tp, S=0)
    assert s0 == 0 and ws0 <= 4096


def test_layer_null_pointers_rejected_before_launch(tp):
    from tensor_transformer_mlp_shard_gb300.binding import LayerDesc, _arr
    L = tp.lib()
    d = LayerDesc(tp.make_desc(128, 2, 256, 1024, 2, act="gelu_tanh", dtype="bf16"), 0.1, 1e-5)
    h = ctypes.c_void_p()
    assert L.tp_layer_create(ctypes.byref(d), ctypes.byref(h)) == 0
    good = [0x10000 * (i + 1) for i in range(2)]
    one = _arr(good[:1])
    # gamma missing
    assert L.tp_layer_fwd(h, one, None, 0x10000, _arr(good), None, _arr(good), None, 7, one, 0x10000, 0x10000,
                          0x10000, _arr(good), _arr(good), None, 0, None) == 1
    assert b"gamma" in L.tp_last_error()
    # Xn misaligned
    assert L.tp_layer_fwd(h, one, 0x10000, 0x10000, _arr(good), None, _arr(good), None, 7, one, 0x10008, 0x10000,
                          0x10000, _arr(good), _arr(good), None, 0, None) == 1
    assert b"Xn" in L.tp_last_error()
    # backward: workspace too small
    assert L.tp_layer_bwd(h, one, one, 0x10000, 0x10000, 0x10000, 0x10000, _arr(good), _arr(good), _arr(good),
                          _arr(good), 7, one, 0x10000, 0x10000, _arr(good), None, _arr(good), None,
                          ctypes.c_void_p(0x100000), 16, None) == 1
    assert b"workspace" in L.tp_last_error()
    L.tp_layer_destroy(h)


def test_handles_take_status_slots_until_exhausted(tp):
    """Every MLP / sub-block handle owns one of 1023 device status words; the
    1024th live handle is refused (TP_ERR_UNSUPPORTED) before any CUDA call,
    and destroying a handle returns its word."""
    L = tp.lib()
    d = tp.make_desc(128, 2, 256, 1024, 2)
    hs = []
    try:
        while True:
            h = ctypes.c_void_p()
            s = L.tp_mlp_create(ctypes.byref(d), ctypes.byref(h))
            if s != 0:
                break
            hs.append(h)
            assert len(hs) <= 1023
        assert s == 3 and 1000 <= len(hs) <= 1023  # other live handles of this process hold the rest
        assert b"live handles" in L.tp_last_error()
        L.tp_mlp_destroy(hs.pop())
        h = ctypes.c_void_p()
        assert L.tp_mlp_create(ctypes.byref(d), ctypes.byref(h)) == 0
        hs.append(h)
    finally:
        for h in hs:
            L.tp_mlp_destroy(h)
    h = ctypes.c_void_p()
    assert L.tp_mlp_create(ctypes.byref(d), ctypes.byref(h)) == 0
    L.tp_mlp_destroy(h)
    assert L.tp_mlp_sync_status(None, None) == 1 and L.tp_layer_sync_status(None, None) == 1


def test_fp8_single_layers_need_a_workspace_and_no_alloc_refuses_fp8(tp):
    """The FP8 single-layer forward without a workspace is TP_ERR_ARG, and the
    allocation-free row backward refuses FP8 (its backward reads the
    forward's codes from the forward's workspace): both before any launch."""
    L = tp.lib()
    from tensor_transformer_mlp_shard_gb300.binding import _arr
    d = tp.make_desc(128, 2, 256, 1024, 2, act="none", dtype="fp8")
    p = [0x10000 * (i + 1) for i in range(2)]
    assert L.tp_linear_col(ctypes.byref(d), _arr(p[:1]), _arr(p), None, _arr(p), None, None) == 1
    assert L.tp_linear_row(ctypes.byref(d), _arr(p), _arr(p), None, None, _arr(p[:1]), None) == 1
    assert L.tp_linear_row_bwd_noalloc(ctypes.byref(d), _arr(p[:1]), _arr(p), _arr(p), _arr(p), _arr(p), None,
                                       None) == 3
    need = L.tp_linear_workspace_bytes(ctypes.byref(d))
    nb = tp.make_desc(128, 2, 256, 1024, 2, act="none", dtype="bf16")
    assert need > L.tp_linear_workspace_bytes(ctypes.byref(nb))  # the FP8 region: amax slots and codes
    # a workspace smaller than that is refused
    assert L.tp_linear_col_ws(ctypes.byref(d), _arr(p[:1]), _arr(p), None, _arr(p), None,
                              ctypes.c_void_p(0x100000), need - 256, None) == 1
