"""GB300-native DTensor tensor-parallel linear and layout transforms.

The compute lives in ``libdt.so`` (CUDA kernels for sm_103a behind the C ABI
declared in ``include/dt.h``); this package is a thin ctypes binding over it.
The library is loaded on first use and a missing build raises immediately:
there is no CPU fallback.
"""
from .api import (  # noqa: F401
    ALL_REDUCE, PARTIAL, REDUCE_SCATTER, ColumnParallelLinear, ColumnParallelLinearWithReplicateInputOutput,
    ColumnParallelLinearWithReplicateOutput, DeviceMesh, DTensor, EmbeddingWithReplicateOutput, Linear, Partial,
    Replicate, ReplicateParallelLinear, RowParallelLinear, RowParallelLinearWithReplicateOutput, Shard,
    column_parallel_linear, column_parallel_linear_multi, column_parallel_linear_workspace_bytes,
    cuda_core_gemm_count, init_device_mesh, read_device_status, redistribute, redistribute_batch,
    row_parallel_linear, row_parallel_linear_workspace_bytes, tp_attention_projections, tp_embedding, tp_mlp,
    tp_mlp_output, tp_mlp_workspace_bytes)
from ._lib import DtError  # noqa: F401
