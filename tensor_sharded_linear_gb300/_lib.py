"""ctypes declarations of the C ABI in ``include/dt.h`` (argument marshalling only)."""
from __future__ import annotations

import ctypes as C
import os
import threading

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "libdt.so")

MAX_MESH_DIMS = 4
MAX_TENSOR_DIMS = 4
MAX_SLOTS = 64

# dt_status
OK, ERR_INVALID_ARG, ERR_SHAPE, ERR_PLACEMENT, ERR_UNSUPPORTED, ERR_ALIGNMENT, ERR_CUDA, ERR_CAPACITY = range(8)
DEV_ERR_INDEX = 0x1
DEV_ERR_TIMEOUT = 0x2
# dt_dtype
BF16, FP32, INT32 = 0, 1, 2
# dt_pkind
REPLICATE, SHARD, PARTIAL = 0, 1, 2
SUM, AVG, MAX = 0, 1, 2
# dt_tp_mode
TP_PARTIAL, TP_ALL_REDUCE, TP_REDUCE_SCATTER = 0, 1, 2
TP_MLP_STATIC_WORKSPACE_BYTES = 32 * 1024 * 1024


class Placement(C.Structure):
    _fields_ = [("kind", C.c_int32), ("dim", C.c_int32), ("op", C.c_int32)]


class Layout(C.Structure):
    _fields_ = [
        ("mesh_ndim", C.c_int32),
        ("mesh_shape", C.c_int32 * MAX_MESH_DIMS),
        ("placements", Placement * MAX_MESH_DIMS),
        ("ndim", C.c_int32),
        ("gshape", C.c_int64 * MAX_TENSOR_DIMS),
        ("dtype", C.c_int32),
        ("materialize_replicas", C.c_int32),
    ]


class DTensorDesc(C.Structure):
    _fields_ = [
        ("layout", Layout),
        ("nslots", C.c_int32),
        ("slots", C.POINTER(C.c_void_p)),
        ("strides", C.POINTER(C.c_int64)),
    ]


EXPORTS = [
    "dt_layout_nslots", "dt_layout_slot_of_rank", "dt_layout_slot_box", "dt_redistribute",
    "dt_redistribute_batch",
    "dt_tp_embedding", "dt_column_parallel_linear", "dt_column_parallel_linear_multi",
    "dt_row_parallel_linear", "dt_column_parallel_linear_workspace_size", "dt_row_parallel_linear_workspace_size",
    "dt_tp_mlp_workspace_size", "dt_tp_mlp", "dt_status_string",
    "dt_last_error", "dt_read_device_status", "dt_clear_cache", "dt_version", "dt_launch_count",
    "dt_cuda_core_gemm_count", "dt_tp_mlp_static_workspace",
]

_lib = None
_lock = threading.Lock()


class DtError(RuntimeError):
    def __init__(self, status: int, message: str):
        super().__init__(message)
        self.status = status


def load(path: str = LIB_PATH) -> C.CDLL:
    """Load libdt.so; raises if it has not been built (there is no fallback)."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        if not os.path.exists(path):
            raise RuntimeError(
                f"{path} is missing: build it with `python -m tensor_sharded_linear_gb300.build` "
                "(the CUDA library is required; there is no CPU path)")
        lib = C.CDLL(path)
        P = C.POINTER
        st = C.c_int
        D = P(DTensorDesc)
        sig = {
            "dt_layout_nslots": (st, [P(Layout), P(C.c_int32)]),
            "dt_layout_slot_of_rank": (st, [P(Layout), C.c_int32, P(C.c_int32)]),
            "dt_layout_slot_box": (st, [P(Layout), C.c_int32, P(C.c_int64), P(C.c_int64)]),
            "dt_redistribute": (st, [D, D, C.c_void_p, C.c_void_p]),
            "dt_redistribute_batch": (st, [C.c_int32, D, D, C.c_void_p, C.c_void_p]),
            "dt_tp_embedding": (st, [D, D, D, C.c_int32, C.c_void_p, C.c_void_p]),
            "dt_column_parallel_linear": (st, [D, D, D, D, C.c_int32, C.c_void_p, C.c_size_t, C.c_void_p,
                                               C.c_void_p]),
            "dt_column_parallel_linear_multi": (st, [D, C.c_int32, D, D, D, C.c_int32, C.c_void_p, C.c_size_t,
                                                     C.c_void_p, C.c_void_p]),
            "dt_row_parallel_linear": (st, [D, D, D, D, C.c_int32, C.c_int32, C.c_void_p, C.c_size_t, C.c_void_p,
                                            C.c_void_p]),
            "dt_column_parallel_linear_workspace_size": (st, [D, C.c_int32, D, D, C.c_int32, P(C.c_size_t)]),
            "dt_row_parallel_linear_workspace_size": (st, [D, D, D, C.c_int32, C.c_int32, P(C.c_size_t)]),
            "dt_tp_mlp_workspace_size": (st, [D, D, D, D, D, C.c_int32, C.c_int32, P(C.c_size_t)]),
            "dt_tp_mlp": (st, [D, D, D, D, D, C.c_int32, C.c_int32, C.c_void_p, C.c_size_t, C.c_void_p, C.c_void_p]),
            "dt_status_string": (C.c_char_p, [C.c_int]),
            "dt_last_error": (C.c_char_p, []),
            "dt_read_device_status": (st, [P(C.c_int32), C.c_int32]),
            "dt_clear_cache": (st, []),
            "dt_version": (C.c_int32, []),
            "dt_launch_count": (C.c_uint64, []),
            "dt_cuda_core_gemm_count": (C.c_uint64, []),
            "dt_tp_mlp_static_workspace": (st, [D, D, D, D, D, C.c_int32, C.c_int32, C.c_void_p, C.c_void_p]),
        }
        for name, (res, args) in sig.items():
            fn = getattr(lib, name)
            fn.restype = res
            fn.argtypes = args
        _lib = lib
        return lib


def check(status: int, what: str) -> None:
    if status != OK:
        lib = load()
        reason = lib.dt_last_error().decode()
        raise DtError(status, f"{what}: {lib.dt_status_string(status).decode()}: {reason}")
