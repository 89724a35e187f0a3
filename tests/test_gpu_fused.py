"""GPU parity of the fused MLP forward (one kernel: column GEMM, bias,
activation, row GEMM with A passed through shared memory; Megatron's
FlashFusedMLP, "Megatron-LM 源码精读" s7, the fusions/ entry) through the
C ABI.

* Against the fp64 oracle, element by element, on ragged multi-tile sizes,
  sequence parallelism, odd T, every H the kernel takes (64..256), GeLU,
  no activation and SwiGLU, and more token tiles than SMs (the persistent
  loop): tolerance 1e-2 * max|ref| (bf16 storage of pre and A, fp32 sums),
  the MLP's bf16 bound.
* Against the two-kernel path on the same inputs: both accumulate the same
  products in fp32 in 64-element K steps, so pre and A agree bit for bit and
  Y to within fp32 reassociation of the chunk sums.
* The even split of the work over the SMs (taken when the token tiles spill
  over whole rounds of the SMs by at most a quarter of a round, and the
  workspace's scratch is there) against the whole-tile schedule of the same
  kernel (no workspace).
"""
import numpy as np
import pytest
import torch

import oracle
from harness import MlpRun, host, mlp_inputs, oracle_full, rel_err, status_ok
from oracle import layer as olayer

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def tp():
    import tensor_transformer_mlp_shard_gb300 as tp
    from tensor_transformer_mlp_shard_gb300 import build
    build.build()
    yield tp
    tp.set_fused_fwd("auto")


CASES = [
    # M, H, F, T, act, bias, residual, sp
    (300, 256, 1024, 2, "gelu_tanh", True, True, False),
    (300, 64, 512, 4, "none", False, False, False),
    (517, 128, 768, 3, "gelu_tanh", True, False, False),
    (1024, 192, 1024, 4, "gelu_tanh", True, True, True),
    (128, 256, 256, 1, "gelu_tanh", False, True, False),
    (40000, 256, 1024, 2, "gelu_tanh", True, True, False),
    # a few token tiles more than a whole number of rounds: the work is cut
    # evenly over the CTAs and a cut tile is finished by the second of its two
    (20736, 128, 768, 3, "gelu_tanh", True, True, True),
    (20485, 64, 512, 4, "none", False, False, False),
    # the most shards the kernel's tensor maps take (16), and 8 token shards
    (600, 128, 2048, 16, "gelu_tanh", True, True, False),
    (1024, 64, 1024, 8, "gelu_tanh", True, True, True),
    # SwiGLU: 64 gate and 64 up units per chunk
    (300, 256, 512, 2, "swiglu", True, True, False),
    (1024, 128, 768, 2, "swiglu", False, False, True),
    (517, 192, 320, 5, "swiglu", True, False, False),
    (20736, 64, 384, 3, "swiglu", True, True, True),
]


def _fwd(tp, lay, t, mode):
    tp.set_fused_fwd(mode)
    run = MlpRun(lay, t)
    n0 = tp.launch_count()
    run.fwd()
    launches = tp.launch_count() - n0
    assert status_ok(tp, lay)
    return run, launches


@pytest.mark.parametrize("M,H,F,T,act,bias,residual,sp", CASES)
def test_fused_forward_matches_oracle_and_two_kernel_path(tp, M, H, F, T, act, bias, residual, sp):
    S, B = (M // 2, 2) if M % 2 == 0 else (M, 1)
    lay = tp.TPMLP(S=S, B=B, H=H, F=F, T=T, act=act, dtype="bf16", has_bias=bias, residual=residual,
                   seq_parallel=sp)
    t = mlp_inputs(M, H, F, T, act, "bf16", has_bias=bias)
    fused, n_fused = _fwd(tp, lay, t, "on")
    split, n_split = _fwd(tp, lay, t, "off")
    assert n_fused == 1 and n_split == 2
    pre, A, Y = oracle.mlp_fwd(t["X"], t["W1s"], t["b1s"], t["W2s"], t["b2"], act, residual)
    errs = {"Y": rel_err(fused.gathered(fused.Y), Y)}
    for i in range(T):
        errs[f"pre{i}"] = rel_err(host(fused.pre[i]), pre[i])
        errs[f"A{i}"] = rel_err(host(fused.A[i]), A[i])
    bad = {k: v for k, v in errs.items() if not v <= 1e-2}
    assert not bad, bad
    for i in range(T):
        assert torch.equal(fused.pre[i], split.pre[i]), i
        assert torch.equal(fused.A[i], split.A[i]), i
    d = rel_err(fused.gathered(fused.Y), split.gathered(split.Y).astype(np.float64))
    assert d <= 2 ** -7, d


@pytest.mark.parametrize("M,H,F,T,sp", [(40000, 256, 1024, 2, False), (20736, 128, 768, 3, True)])
def test_fused_even_split_matches_whole_tiles(tp, M, H, F, T, sp):
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    tiles = (M + 127) // 128
    assert tiles > sms and 0 < tiles % sms <= sms // 4, "the case must cut tiles"
    lay = tp.TPMLP(S=M // T if sp else M, B=T if sp else 1, H=H, F=F, T=T, act="gelu_tanh", dtype="bf16",
                   has_bias=True, residual=True, seq_parallel=sp)
    t = mlp_inputs(M, H, F, T, "gelu_tanh", "bf16", has_bias=True)
    tp.set_fused_fwd("on")
    runs = []
    for ws in (True, False):
        run = MlpRun(lay, t)
        run.fwd(with_workspace=ws)
        assert status_ok(tp, lay)
        runs.append(run)
    split, whole = runs
    for i in range(T):
        assert torch.equal(split.pre[i], whole.pre[i]), i
        assert torch.equal(split.A[i], whole.A[i]), i
    d = rel_err(split.gathered(split.Y), whole.gathered(whole.Y).astype(np.float64))
    assert d <= 2 ** -7, d
    tp.set_fused_fwd("auto")


def test_fused_forward_pre_buffers_16_byte_aligned(tp):
    """pre buffers 16- but not 32-byte aligned take the 16-byte stores instead
    of the 32-byte ones, with the same results."""
    M, H, F, T = 1000, 256, 1024, 2
    lay = tp.TPMLP(S=M // 2, B=2, H=H, F=F, T=T, act="gelu_tanh", dtype="bf16", has_bias=True, residual=True)
    t = mlp_inputs(M, H, F, T, "gelu_tanh", "bf16", has_bias=True)
    tp.set_fused_fwd("on")
    aligned, _ = _fwd(tp, lay, t, "on")
    run = MlpRun(lay, t)
    Fs = F // T
    backing = [torch.empty(M * Fs + 8, dtype=torch.bfloat16, device="cuda") for _ in range(T)]
    run.pre = [b[8:].view(M, Fs) for b in backing]  # 16 bytes past a 256-byte boundary
    assert all(x.data_ptr() % 32 == 16 for x in run.pre)
    run.fwd()
    assert status_ok(tp, lay)
    for i in range(T):
        assert torch.equal(run.pre[i], aligned.pre[i]), i
        assert torch.equal(run.A[i], aligned.A[i]), i
    for a, b in zip(run.Y, aligned.Y):
        assert torch.equal(a, b)
    tp.set_fused_fwd("auto")


def test_narrow_workload_full_size_against_oracle(tp):
    """The narrow workload as bench.py times it (65536 tokens, H = 256, F = 1024,
    T = 2, bias, residual; the fused forward by default, whole tiles), forward
    and backward against the fp64 oracle element by element: the bias
    gradients' 2048 partial rows go through the finalize's clusters of 8
    blocks and the weight gradients through the 16-way split-K reduction."""
    M, H, F, T = 65536, 256, 1024, 2
    lay = tp.TPMLP(S=4096, B=16, H=H, F=F, T=T, act="gelu_tanh", dtype="bf16", has_bias=True, residual=True)
    t = mlp_inputs(M, H, F, T, "gelu_tanh", "bf16", has_bias=True)
    tp.set_fused_fwd("auto")
    run = MlpRun(lay, t)
    n0 = tp.launch_count()
    run.fwd()
    assert tp.launch_count() - n0 == 1
    run.bwd()
    assert status_ok(tp, lay)
    ref = oracle_full(lay, t)
    errs = {"Y": rel_err(run.gathered(run.Y), ref["Y"]), "dX": rel_err(run.gathered(run.dX), ref["dX"]),
            "db2": rel_err(host(run.db2), ref["db2"])}
    for i in range(T):
        errs[f"pre{i}"] = rel_err(host(run.pre[i]), ref["pre"][i])
        errs[f"A{i}"] = rel_err(host(run.A[i]), ref["A"][i])
        errs[f"dW1_{i}"] = rel_err(host(run.dW1[i]), ref["dW1"][i])
        errs[f"dW2_{i}"] = rel_err(host(run.dW2[i]), ref["dW2"][i])
        errs[f"db1_{i}"] = rel_err(host(run.db1[i]), ref["db1"][i])
    bad = {k: v for k, v in errs.items() if not v <= 1e-2}
    assert not bad, bad


def test_fused_forward_feeds_the_backward(tp):
    """The backward after a fused forward equals the backward after the
    two-kernel forward (it reads pre and A, which are bit-identical)."""
    M, H, F, T = 384, 256, 1024, 2
    lay = tp.TPMLP(S=M // 2, B=2, H=H, F=F, T=T, act="gelu_tanh", dtype="bf16", has_bias=True, residual=True)
    t = mlp_inputs(M, H, F, T, "gelu_tanh", "bf16", has_bias=True)
    outs = []
    for mode in ("on", "off"):
        run, _ = _fwd(tp, lay, t, mode)
        run.bwd()
        assert status_ok(tp, lay)
        outs.append(run)
    a, b = outs
    for x, y in zip(a.dW1 + a.dW2 + [a.db2] + a.db1 + a.dX, b.dW1 + b.dW2 + [b.db2] + b.db1 + b.dX):
        assert torch.equal(x, y)


def test_fused_forward_not_taken_outside_its_shapes(tp):
    tp.set_fused_fwd("on")
    for kw in (dict(H=320, F=1024), dict(H=256, F=96 * 2, act="swiglu"), dict(H=256, F=96 * 2)):
        act = kw.pop("act", "gelu_tanh")
        lay = tp.TPMLP(S=64, B=2, T=2, act=act, dtype="bf16", **kw)
        t = mlp_inputs(128, lay.H, lay.F, 2, act, "bf16", has_bias=False)
        run = MlpRun(lay, t)
        n0 = tp.launch_count()
        run.fwd()
        assert tp.launch_count() - n0 == 2, kw
    assert status_ok(tp, lay)
    tp.set_fused_fwd("auto")


def test_fused_forward_by_default(tp):
    """TP_FUSED_AUTO takes the fused kernel for the shapes it takes, at any
    token count, and the two GEMMs for the shapes it does not take."""
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    tp.set_fused_fwd("auto")
    for M, H, F, fused in ((4096, 256, 1024, True), (128 * (10 * sms + 1), 128, 512, True),
                           (4096, 512, 1024, False), (4096, 256, 96 * 2, False)):
        lay = tp.TPMLP(S=M, B=1, H=H, F=F, T=2, act="gelu_tanh", dtype="bf16", has_bias=True, residual=True)
        t = mlp_inputs(M, H, F, 2, "gelu_tanh", "bf16", has_bias=True)
        run = MlpRun(lay, t)
        n0 = tp.launch_count()
        run.fwd()
        assert tp.launch_count() - n0 == (1 if fused else 2), (M, H)
        assert status_ok(tp, lay)


@pytest.mark.parametrize("M", [300, 20000])
def test_fused_layer_forward_with_dropout(tp, M):
    """The sub-block's forward on the fused kernel (dropout in its output
    epilogue) against the layer oracle; at 20000 tokens the work is cut
    evenly over the SMs, so the cut tiles' dropout runs in the CTA that
    finishes them."""
    from test_gpu_layer import LayerRun, layer_inputs, SEED, _p32
    H, F, T, p = 256, 1024, 2, 0.1
    lay = tp.TPLayer(S=M // 2, B=2, H=H, F=F, T=T, act="gelu_tanh", dtype="bf16", has_bias=True, dropout_p=p)
    t = layer_inputs(M, H, F, T, "gelu_tanh", "bf16", True)
    tp.set_fused_fwd("on")
    run = LayerRun(lay, t)
    n0 = tp.launch_count()
    run.fwd(SEED)
    assert tp.launch_count() - n0 == 2  # LayerNorm + fused MLP
    run.bwd(SEED)
    assert status_ok(tp, lay)
    f = olayer.layer_fwd(t["X"], t["gamma"], t["beta"], t["W1s"], t["b1s"], t["W2s"], t["b2"], "gelu_tanh",
                         _p32(p), SEED)
    gr = olayer.layer_bwd(t["dY"], t["X"], t["gamma"], t["W1s"], t["W2s"], f, "gelu_tanh", _p32(p))
    errs = {"Y": rel_err(run.gathered(run.Y), f["Y"]), "dX": rel_err(run.gathered(run.dX), gr["dX"]),
            "dgamma": rel_err(host(run.dgamma), gr["dgamma"]), "db2": rel_err(host(run.db2), gr["db2"])}
    bad = {k: v for k, v in errs.items() if not v <= 1e-2}
    assert not bad, bad
    tp.set_fused_fwd("auto")
