"""CPU oracle of the tensor-parallel MLP -- test infrastructure only.

Imported only by ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline
leg of ``bench.py``.  The product path never imports it.
"""
from .mlp import *  # noqa: F401,F403
from .mlp import (ACTS, act_bwd, act_fwd, column_bwd, column_fwd, divide, gelu_tanh,  # noqa: F401
                  gelu_tanh_grad, mlp_bwd, mlp_fwd, mlp_loss, mlp_rows, mlp_units, row_bwd,
                  row_fwd, shard_column_bias, shard_column_weight, shard_row_weight, sigmoid, silu,
                  sp_gather, sp_split, unshard_column)
