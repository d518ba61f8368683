"""ctypes declarations of libmoe_gb300.so (the C ABI in include/moe_gb300.h)."""
from __future__ import annotations

import ctypes
import os

from . import _build

MOE_OK = 0
STATUS_NAMES = {0: "MOE_OK", 1: "MOE_ERR_INVALID_ARG", 2: "MOE_ERR_UNSUPPORTED",
                3: "MOE_ERR_INCOMPATIBLE", 4: "MOE_ERR_CUDA", 5: "MOE_ERR_TIMEOUT",
                6: "MOE_ERR_DEVICE"}
DTYPE_F32, DTYPE_BF16 = 0, 1
EPILOGUE_RAW, EPILOGUE_SWIGLU = 0, 1
PATH_AUTO, PATH_GEMV, PATH_TC = 0, 1, 2
PATH_FLAG_WEIGHTS_EARLY = 0x100  # moe_down_qmm: offsets/weights read before the wait
PATH_FLAG_K_GATED = 0x200  # the product runs only for lo <= k <= hi (MOE_PATH_K_RANGE)


def path_k_range(lo: int, hi: int) -> int:
    """Flags of a k-gated launch: the product runs only if lo <= k <= hi."""
    return PATH_FLAG_K_GATED | (lo << 16) | (hi << 24)
DEVERR_BAD_EXPERT, DEVERR_TIMEOUT, DEVERR_BAD_INDEX = 1, 2, 4
DROPPED = -2  # inv_pos of an assignment dropped by its expert's capacity
QMODE_AFFINE = 0
SCALE_F16, SCALE_BF16, SCALE_F32 = 0, 1, 2

# every symbol the header declares
EXPORTS = (
    "moe_status_string", "moe_abi_version", "moe_set_launch_overlap", "moe_pack_gate_up", "moe_router_workspace_size",
    "moe_router_topk", "moe_router_topk_noalloc", "moe_route", "moe_route_grouped", "moe_permute", "moe_permute_capped", "moe_permute_rows", "moe_gate_up_qmm", "moe_down_qmm", "moe_combine",
    "moe_swiglu", "moe_get_device_error", "moe_selftest_wait_timeout",
    "moe_expert_counts_accumulate", "moe_expert_health",
)


class MoEError(RuntimeError):
    def __init__(self, func: str, status: int):
        self.status = status
        super().__init__(f"{func} returned {STATUS_NAMES.get(status, status)}")


class QDesc(ctypes.Structure):
    _fields_ = [("quantized", ctypes.c_int32), ("bits", ctypes.c_int32),
                ("group_size", ctypes.c_int32), ("mode", ctypes.c_int32),
                ("has_bias", ctypes.c_int32), ("rows", ctypes.c_int32),
                ("cols", ctypes.c_int32), ("scale_dtype", ctypes.c_int32)]


_LIB = None

vp = ctypes.c_void_p
i32 = ctypes.c_int
f32 = ctypes.c_float
sz = ctypes.c_size_t


def _declare(lib):
    lib.moe_status_string.argtypes = [i32]
    lib.moe_status_string.restype = ctypes.c_char_p
    lib.moe_abi_version.argtypes = []
    lib.moe_abi_version.restype = i32
    lib.moe_set_launch_overlap.argtypes = [i32]
    lib.moe_set_launch_overlap.restype = i32
    lib.moe_pack_gate_up.argtypes = [ctypes.POINTER(QDesc), ctypes.POINTER(QDesc), vp, vp, vp, vp,
                                     vp, vp, i32, vp, vp, vp, vp]
    lib.moe_router_workspace_size.argtypes = [i32]
    lib.moe_router_workspace_size.restype = sz
    lib.moe_router_topk.argtypes = [vp, vp, vp, f32, i32, i32, i32, i32, i32, f32, f32, i32, vp,
                                    vp, vp, vp, vp, sz, vp]
    lib.moe_router_topk_noalloc.argtypes = [vp, vp, vp, f32, i32, i32, i32, i32, i32, f32, f32,
                                            i32, vp, vp, vp, vp, vp]
    lib.moe_route.argtypes = [vp, vp, vp, f32, i32, i32, i32, i32, i32, f32, f32, i32, vp, vp, vp,
                              vp, vp, sz, vp, vp, vp, vp, vp]
    lib.moe_permute.argtypes = [vp, vp, i32, i32, i32, vp, vp, vp, vp, vp]
    lib.moe_permute_capped.argtypes = [vp, vp, i32, i32, i32, i32, vp, vp, vp, vp, vp]
    lib.moe_route_grouped.argtypes = [vp, vp, vp, f32, i32, i32, i32, i32, i32, i32, vp, vp, vp,
                                      vp, vp, sz, vp, vp, vp, vp, vp]
    lib.moe_permute_rows.argtypes = [vp, vp, vp, i32, i32, i32, vp, vp]
    lib.moe_gate_up_qmm.argtypes = [vp, vp, vp, vp, i32, i32, i32, i32, i32, vp, vp, vp, i32, i32,
                                    i32, vp, i32, vp]
    lib.moe_down_qmm.argtypes = [vp, i32, vp, vp, i32, i32, i32, i32, i32, vp, vp, vp, i32, vp,
                                 i32, i32, vp]
    lib.moe_combine.argtypes = [vp, i32, vp, vp, vp, i32, i32, i32, vp, vp]
    lib.moe_swiglu.argtypes = [vp, vp, vp, i32, i32, i32, i32, vp, vp]
    lib.moe_get_device_error.argtypes = [ctypes.POINTER(ctypes.c_uint32), i32, vp]
    lib.moe_selftest_wait_timeout.argtypes = [ctypes.c_uint32, vp]
    lib.moe_expert_counts_accumulate.argtypes = [vp, i32, vp, vp]
    lib.moe_expert_health.argtypes = [vp, i32, vp, vp, vp]
    for name in ("moe_pack_gate_up", "moe_router_topk", "moe_router_topk_noalloc", "moe_route",
                 "moe_route_grouped", "moe_permute_capped",
                 "moe_permute", "moe_permute_rows", "moe_gate_up_qmm",
                 "moe_down_qmm", "moe_combine", "moe_swiglu", "moe_get_device_error",
                 "moe_selftest_wait_timeout", "moe_expert_counts_accumulate",
                 "moe_expert_health"):
        getattr(lib, name).restype = i32


def lib_path() -> str:
    return _build.LIB


def lib():
    """The loaded library.  Raises if it has not been built: there is no
    fallback implementation of any step."""
    global _LIB
    if _LIB is None:
        path = _build.LIB
        if not os.path.exists(path):
            raise RuntimeError(
                f"{path} is missing: build it with sparse_moe_expert_gb300._build.build() "
                "(nvcc, sm_103a); the MoE layer has no other implementation")
        handle = ctypes.CDLL(path)
        _declare(handle)
        _LIB = handle
    return _LIB


def check(name: str, status: int) -> None:
    if status != MOE_OK:
        raise MoEError(name, status)
