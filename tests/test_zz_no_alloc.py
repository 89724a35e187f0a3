"""The allocation-free row-layer backward (tp_linear_row_bwd_noalloc).

Some callers cannot allocate device memory when they call: a plugin that is
handed only the op's tensors, a process whose device memory belongs to another
allocator, a latency-critical loop that cannot take cudaMalloc's implicit
synchronisation.  For them the library's bias-gradient scratch comes from a
fixed array compiled into it.  This test calls that entry point through the C
ABI twice in a row (the second time with different inputs, so stale scratch
from the first call would show) and checks each result against
tp_linear_row_bwd with a caller workspace.  The file sorts last so that a run
stopping at the first failure has already run every other test.
"""
import pytest
import torch

from harness import TOL, host, rel_err

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def tp():
    import tensor_transformer_mlp_shard_gb300 as tp
    from tensor_transformer_mlp_shard_gb300 import build
    build.build()
    return tp


def _buffers(lay, seed):
    g = torch.Generator(device="cuda").manual_seed(seed)
    bf = dict(dtype=torch.bfloat16, device="cuda")
    dY = [torch.randn(lay.xrows, lay.H, generator=g, device="cuda").to(torch.bfloat16) for _ in range(lay.nx)]
    X = [torch.randn(lay.M, lay.Fs, generator=g, device="cuda").to(torch.bfloat16) for _ in range(lay.T)]
    W = [(0.02 * torch.randn(lay.H, lay.Fs, generator=g, device="cuda")).to(torch.bfloat16) for _ in range(lay.T)]
    outs = lambda: ([torch.empty(lay.M, lay.Fs, **bf) for _ in range(lay.T)],
                    [torch.empty(lay.H, lay.Fs, dtype=torch.float32, device="cuda") for _ in range(lay.T)],
                    torch.empty(lay.H, dtype=torch.float32, device="cuda"))
    return dY, X, W, outs


@pytest.mark.parametrize("seq_parallel", [False, True])
def test_noalloc_matches_workspace_entry_point(tp, seq_parallel):
    lay = tp.Layout(S=512, B=2, H=520, F=1024, T=4, act="none", dtype="bf16", has_bias=True,
                    seq_parallel=seq_parallel)
    tol = TOL["bf16"]
    for call, seed in enumerate((11, 12)):
        dY, X, W, outs = _buffers(lay, seed)
        dX_ref, dW_ref, db_ref = outs()
        ws = tp.alloc_workspace(tp.linear_workspace_bytes(lay))
        tp.linear_row_bwd(lay, dY, X, W, dX_ref, dW_ref, db_ref, ws)
        dX, dW, db = outs()
        tp.linear_row_bwd_noalloc(lay, dY, X, W, dX, dW, db)
        assert tp.sync_status() == 0
        for a, b in zip(dX + dW + [db], dX_ref + dW_ref + [db_ref]):
            assert rel_err(host(a), host(b)) <= tol, f"call {call}"


def test_noalloc_rejects_oversized_scratch(tp):
    # bias partials: 4 * ceil(M/256) * H bytes; M = 65536, H = 8192 -> 8 MiB > 4 MiB
    lay = tp.Layout(S=65536, B=1, H=8192, F=64, T=8, act="none", dtype="bf16", has_bias=True)
    from tensor_transformer_mlp_shard_gb300.binding import TpError
    bf = dict(dtype=torch.bfloat16, device="cuda")
    with pytest.raises(TpError) as e:
        tp.linear_row_bwd_noalloc(lay, [torch.empty(lay.M, lay.H, **bf)],
                                  [torch.empty(lay.M, lay.Fs, **bf) for _ in range(lay.T)],
                                  [torch.empty(lay.H, lay.Fs, **bf) for _ in range(lay.T)],
                                  [torch.empty(lay.M, lay.Fs, **bf) for _ in range(lay.T)],
                                  [torch.empty(lay.H, lay.Fs, dtype=torch.float32, device="cuda")
                                   for _ in range(lay.T)],
                                  torch.empty(lay.H, dtype=torch.float32, device="cuda"))
    assert e.value.status == 3
    assert tp.sync_status() == 0
