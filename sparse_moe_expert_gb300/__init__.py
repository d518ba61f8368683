"""GB300-native forward of a quantized sparse-MoE SwitchGLU layer.

The compute lives in libmoe_gb300.so (CUDA for sm_103a, C ABI declared in
include/moe_gb300.h).  This package is its binding: ``binding`` has one
function per C entry point and ``MoELayer`` composes them.  Importing it
does not build anything; calling into it without the built library raises.
"""
from ._lib import (DEVERR_BAD_EXPERT, DEVERR_BAD_INDEX, DEVERR_TIMEOUT, DROPPED, DTYPE_BF16,
                   DTYPE_F32,
                   EPILOGUE_RAW, EPILOGUE_SWIGLU, EXPORTS, PATH_AUTO, PATH_FLAG_K_GATED,
                   PATH_FLAG_WEIGHTS_EARLY, PATH_GEMV, PATH_TC, path_k_range,
                   MoEError,
                   lib, lib_path)
from .binding import (moe_abi_version, moe_combine, moe_down_qmm, moe_expert_counts_accumulate,
                      moe_expert_health, moe_gate_up_qmm,
                      moe_get_device_error, moe_pack_gate_up, moe_permute, moe_permute_capped,
                      moe_permute_rows,
                      moe_route, moe_route_grouped, moe_router_topk, moe_selftest_wait_timeout,
                      moe_set_launch_overlap,
                      moe_router_workspace_size, moe_status_string, moe_swiglu, qdesc)
from .health import ExpertHealthMonitor, WindowHealth
from .layer import MoELayer, QTensor, bf16_from_bits, qtensor_from_numpy

__all__ = [
    "MoELayer", "QTensor", "MoEError", "ExpertHealthMonitor", "WindowHealth",
    "moe_expert_counts_accumulate", "moe_expert_health", "qtensor_from_numpy", "bf16_from_bits", "lib", "lib_path",
    "moe_abi_version", "moe_set_launch_overlap", "moe_status_string", "moe_pack_gate_up", "moe_router_workspace_size",
    "moe_router_topk", "moe_route", "moe_route_grouped", "moe_permute", "moe_permute_capped", "moe_permute_rows", "moe_gate_up_qmm", "moe_down_qmm", "moe_combine",
    "moe_swiglu", "moe_get_device_error", "moe_selftest_wait_timeout", "qdesc", "EXPORTS", "DTYPE_F32", "DTYPE_BF16",
    "EPILOGUE_RAW", "EPILOGUE_SWIGLU", "PATH_AUTO", "PATH_FLAG_K_GATED", "path_k_range", "PATH_FLAG_WEIGHTS_EARLY", "PATH_GEMV", "PATH_TC",
    "DEVERR_BAD_EXPERT", "DEVERR_TIMEOUT", "DEVERR_BAD_INDEX", "DROPPED",
]
