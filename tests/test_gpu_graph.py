"""CUDA-graph capture of the library's calls: after one eager call (which
sets the per-device kernel attributes and looks up the status words), a
forward + backward step records into a graph through the caller's stream,
and replaying it gives bit-identical results to eager calls -- the library
enqueues only kernels and memsets on that stream and does no host sync.
(Under FP8 delayed scaling the history column a call writes is fixed when the
call is captured; the test uses current scaling there.)"""
import pytest
import torch

from harness import MlpRun, mlp_inputs, status_ok

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def tp():
    import tensor_transformer_mlp_shard_gb300 as tp
    from tensor_transformer_mlp_shard_gb300 import build
    build.build()
    return tp


@pytest.mark.parametrize("dtype,act,sp", [("bf16", "gelu_tanh", False), ("bf16", "swiglu", True),
                                          ("f32", "gelu_tanh", False), ("fp8", "gelu_tanh", False)])
def test_mlp_step_replays_bitwise(tp, dtype, act, sp):
    M, H, F, T = 512, 256, 1024, 4
    lay = tp.TPMLP(S=M // 2, B=2, H=H, F=F, T=T, act=act, dtype=dtype, has_bias=True, residual=True,
                   seq_parallel=sp)
    t = mlp_inputs(M, H, F, T, act, dtype, has_bias=True)
    run = MlpRun(lay, t)
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        run.fwd()  # eager warm-up call
        run.bwd()
    s.synchronize()
    assert status_ok(tp, lay)
    ref = [x.clone() for x in run.Y + run.dX + run.pre + run.A + run.dW1 + run.dW2 + run.db1 + [run.db2]]
    for x in run.Y + run.dX + run.dW1 + run.dW2:
        x.fill_(float("nan"))
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        run.fwd()
        run.bwd()
    for _ in range(2):
        g.replay()
    torch.cuda.synchronize()
    assert status_ok(tp, lay)
    out = run.Y + run.dX + run.pre + run.A + run.dW1 + run.dW2 + run.db1 + [run.db2]
    for a, b in zip(ref, out):
        assert torch.equal(a, b)


def test_fused_split_forward_replays_bitwise(tp):
    """The fused forward with its work split evenly over the SMs (a few token
    tiles past a whole round): the flag memset and the kernel record into the
    graph, and every replay gives the eager result bit for bit (a cut tile's
    two parts are added in either arrival order to the same sum)."""
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    M, H, F, T = 128 * (sms + 3), 256, 1024, 2
    lay = tp.TPMLP(S=M, B=1, H=H, F=F, T=T, act="gelu_tanh", dtype="bf16", has_bias=True, residual=True)
    t = mlp_inputs(M, H, F, T, "gelu_tanh", "bf16", has_bias=True)
    run = MlpRun(lay, t)
    tp.set_fused_fwd("on")
    try:
        s = torch.cuda.Stream()
        with torch.cuda.stream(s):
            run.fwd()
        s.synchronize()
        assert status_ok(tp, lay)
        ref = [x.clone() for x in run.Y + run.pre + run.A]
        for x in run.Y:
            x.fill_(float("nan"))
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=s):
            run.fwd()
        for _ in range(3):
            g.replay()
            torch.cuda.synchronize()
            assert status_ok(tp, lay)
            for a, b in zip(ref, run.Y + run.pre + run.A):
                assert torch.equal(a, b)
    finally:
        tp.set_fused_fwd("auto")


def test_layer_step_replays_bitwise(tp):
    from test_gpu_layer import LayerRun, layer_inputs, SEED
    M, H, F, T = 384, 256, 1024, 4
    lay = tp.TPLayer(S=M // 2, B=2, H=H, F=F, T=T, act="gelu_tanh", dtype="bf16", has_bias=True, dropout_p=0.1)
    t = layer_inputs(M, H, F, T, "gelu_tanh", "bf16", True)
    run = LayerRun(lay, t)
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        run.fwd(SEED)
        run.bwd(SEED)
    s.synchronize()
    ref = [x.clone() for x in run.Y + run.dX + [run.Xn, run.dgamma, run.dbeta, run.db2] + run.dW1]
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        run.fwd(SEED)
        run.bwd(SEED)
    g.replay()
    torch.cuda.synchronize()
    assert status_ok(tp, lay)
    for a, b in zip(ref, run.Y + run.dX + [run.Xn, run.dgamma, run.dbeta, run.db2] + run.dW1):
        assert torch.equal(a, b)
