"""Single-GPU tensor-parallel MLP for GB300 (sm_103a).

The Megatron ColumnParallelLinear -> activation -> RowParallelLinear block with
all T shards in one GPU's memory; the cross-shard all-reduces are fp32 sums
inside the tcgen05 GEMM kernels of ``libtpmlp.so`` (C ABI in
``include/tp_mlp.h``).  This package is the thin Python binding.
"""
from .binding import (ACT, DTYPE, Layout, TPLayer, TPMLP, TpError, alloc_workspace, debug_wait_timeout,  # noqa: F401
                      fp8_quantize,
                      launch_count, lib, library_path, linear_col, linear_col_bwd, linear_row, linear_row_bwd,
                      linear_row_bwd_noalloc,
                      linear_workspace_bytes, make_desc, prof_collect, prof_enable, prof_select, set_fused_fwd, set_max_gemm_pairs,
                      set_band_rows, set_k_order, set_launch_overlap, set_tail_split, set_tile_mode, tail_split_count,
                      set_wait_limit_ns,
                      status_str,
                      sync_status)
