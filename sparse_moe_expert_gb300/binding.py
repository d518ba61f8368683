"""Thin Python binding of the C ABI: one function per entry point, same names.

Each function checks tensor placement and dtypes, allocates missing outputs
with torch (device memory only), passes raw pointers and the current CUDA
stream to libmoe_gb300.so, and raises MoEError on a non-zero status.  No step
of the layer is computed here.
"""
from __future__ import annotations

import ctypes
from typing import Optional

import torch

from . import _lib
from ._lib import (DTYPE_BF16, DTYPE_F32, EPILOGUE_RAW, EPILOGUE_SWIGLU, PATH_AUTO, QDesc,
                   check, lib)

_DT = {torch.float32: DTYPE_F32, torch.bfloat16: DTYPE_BF16}


def _p(t: Optional[torch.Tensor]):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream=None):
    s = stream if stream is not None else torch.cuda.current_stream()
    return ctypes.c_void_p(s.cuda_stream)


def _need(t: torch.Tensor, dtype, name: str):
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if t.dtype != dtype:
        raise ValueError(f"{name} must be {dtype}, got {t.dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")


def moe_abi_version() -> int:
    return int(lib().moe_abi_version())


def moe_set_launch_overlap(enable: bool) -> bool:
    """Programmatic dependent launch on (default) or off for later launches;
    returns the previous setting."""
    return bool(lib().moe_set_launch_overlap(int(bool(enable))))


def moe_status_string(status: int) -> str:
    return lib().moe_status_string(status).decode()


def qdesc(rows: int, cols: int, bits: int, group_size: int = 64, quantized: bool = True,
          mode: int = _lib.QMODE_AFFINE, has_bias: bool = False,
          scale_dtype: int = _lib.SCALE_F16) -> QDesc:
    return QDesc(int(quantized), bits, group_size, mode, int(has_bias), rows, cols, scale_dtype)


def moe_pack_gate_up(gate_desc: QDesc, up_desc: QDesc, gate_q, gate_s, gate_b, up_q, up_s, up_b,
                     stream=None):
    """[gate; up] concatenation of codes, scales and biases -> (gu_q, gu_s, gu_b)."""
    E, I = gate_q.shape[0], gate_q.shape[1]
    gu_q = torch.empty((E, 2 * I, gate_q.shape[2]), dtype=gate_q.dtype, device=gate_q.device)
    gu_s = torch.empty((E, 2 * I, gate_s.shape[2]), dtype=gate_s.dtype, device=gate_s.device)
    gu_b = torch.empty_like(gu_s)
    st = lib().moe_pack_gate_up(ctypes.byref(gate_desc), ctypes.byref(up_desc), _p(gate_q),
                                _p(gate_s), _p(gate_b), _p(up_q), _p(up_s), _p(up_b), E, _p(gu_q),
                                _p(gu_s), _p(gu_b), _stream(stream))
    check("moe_pack_gate_up", st)
    return gu_q, gu_s, gu_b


def moe_router_workspace_size(T: int) -> int:
    return int(lib().moe_router_workspace_size(T))


def moe_router_topk(x, w_router, logit_bias=None, inv_temperature: float = 1.0, k_fixed: int = 2,
                    kmax: Optional[int] = None, thr1: float = 1.2, thr2: float = 2.5,
                    renormalize: bool = True, topk_ids=None, topk_w=None, k_dev=None,
                    mean_entropy=None, workspace=None, stream=None):
    """-> (topk_ids int32 [T,kmax], topk_w f32 [T,kmax], k_dev int32 [1], mean_entropy f32 [1])"""
    _need(x, torch.bfloat16, "x")
    _need(w_router, torch.float32, "w_router")
    T, H = x.shape
    E = w_router.shape[0]
    if kmax is None:
        kmax = k_fixed if k_fixed > 0 else 3
    dev = x.device
    if topk_ids is None:
        topk_ids = torch.empty((T, kmax), dtype=torch.int32, device=dev)
    if topk_w is None:
        topk_w = torch.empty((T, kmax), dtype=torch.float32, device=dev)
    if k_dev is None:
        k_dev = torch.empty(1, dtype=torch.int32, device=dev)
    if mean_entropy is None:
        mean_entropy = torch.empty(1, dtype=torch.float32, device=dev)
    wsb = moe_router_workspace_size(T)
    if workspace is None:
        workspace = torch.empty(wsb, dtype=torch.uint8, device=dev)
    st = lib().moe_router_topk(_p(x), _p(w_router), _p(logit_bias), ctypes.c_float(inv_temperature),
                               T, H, E, k_fixed, kmax, ctypes.c_float(thr1), ctypes.c_float(thr2),
                               int(renormalize), _p(topk_ids), _p(topk_w), _p(k_dev),
                               _p(mean_entropy), _p(workspace), workspace.numel(), _stream(stream))
    check("moe_router_topk", st)
    return topk_ids, topk_w, k_dev, mean_entropy


def moe_route(x, w_router, logit_bias, inv_temperature: float, k_fixed: int, kmax: int,
              thr1: float, thr2: float, renormalize: bool, topk_ids, topk_w, k_dev, mean_entropy,
              workspace, expert_counts, expert_offsets, sorted_assign, inv_pos, stream=None):
    """moe_router_topk then moe_permute in one call (one launch for small
    batches); every output buffer is given."""
    _need(x, torch.bfloat16, "x")
    _need(w_router, torch.float32, "w_router")
    T, H = x.shape
    E = w_router.shape[0]
    st = lib().moe_route(_p(x), _p(w_router), _p(logit_bias), ctypes.c_float(inv_temperature),
                         T, H, E, k_fixed, kmax, ctypes.c_float(thr1), ctypes.c_float(thr2),
                         int(renormalize), _p(topk_ids), _p(topk_w), _p(k_dev), _p(mean_entropy),
                         _p(workspace), workspace.numel(), _p(expert_counts), _p(expert_offsets),
                         _p(sorted_assign), _p(inv_pos), _stream(stream))
    check("moe_route", st)
    return topk_ids, topk_w, k_dev, mean_entropy, expert_counts, expert_offsets, sorted_assign, inv_pos


def moe_route_grouped(x, w_router, logit_bias, inv_temperature: float, n_groups: int, kmax: int,
                      renormalize: bool, topk_ids, topk_w, k_dev, mean_entropy, workspace,
                      expert_counts, expert_offsets, sorted_assign, inv_pos, stream=None):
    """moe_route with group-limited selection (the best expert of each of
    n_groups groups of consecutive ids, k = n_groups)."""
    _need(x, torch.bfloat16, "x")
    _need(w_router, torch.float32, "w_router")
    T, H = x.shape
    E = w_router.shape[0]
    st = lib().moe_route_grouped(_p(x), _p(w_router), _p(logit_bias),
                                 ctypes.c_float(inv_temperature), T, H, E, n_groups, kmax,
                                 int(renormalize), _p(topk_ids), _p(topk_w), _p(k_dev),
                                 _p(mean_entropy), _p(workspace), workspace.numel(),
                                 _p(expert_counts), _p(expert_offsets), _p(sorted_assign),
                                 _p(inv_pos), _stream(stream))
    check("moe_route_grouped", st)
    return topk_ids, topk_w, k_dev, mean_entropy, expert_counts, expert_offsets, sorted_assign, inv_pos


def moe_permute(topk_ids, k_dev, E: int, expert_counts=None, expert_offsets=None,
                sorted_assign=None, inv_pos=None, stream=None):
    """-> (expert_counts [E], expert_offsets [E+1], sorted_assign [T*kmax], inv_pos [T*kmax])"""
    _need(topk_ids, torch.int32, "topk_ids")
    T, kmax = topk_ids.shape
    dev = topk_ids.device
    if expert_counts is None:
        expert_counts = torch.empty(E, dtype=torch.int32, device=dev)
    if expert_offsets is None:
        expert_offsets = torch.empty(E + 1, dtype=torch.int32, device=dev)
    if sorted_assign is None:
        sorted_assign = torch.empty(max(T * kmax, 1), dtype=torch.int32, device=dev)
    if inv_pos is None:
        inv_pos = torch.empty(max(T * kmax, 1), dtype=torch.int32, device=dev)
    st = lib().moe_permute(_p(topk_ids), _p(k_dev), T, kmax, E, _p(expert_counts),
                           _p(expert_offsets), _p(sorted_assign), _p(inv_pos), _stream(stream))
    check("moe_permute", st)
    return expert_counts, expert_offsets, sorted_assign, inv_pos


def moe_permute_capped(topk_ids, k_dev, E: int, capacity: int, expert_counts, expert_offsets,
                       sorted_assign, inv_pos, stream=None):
    """moe_permute keeping at most `capacity` assignments per expert (the
    lowest a = t*kmax + j); dropped ones get inv_pos = DROPPED."""
    _need(topk_ids, torch.int32, "topk_ids")
    T, kmax = topk_ids.shape
    st = lib().moe_permute_capped(_p(topk_ids), _p(k_dev), T, kmax, E, int(capacity),
                                  _p(expert_counts), _p(expert_offsets), _p(sorted_assign),
                                  _p(inv_pos), _stream(stream))
    check("moe_permute_capped", st)
    return expert_counts, expert_offsets, sorted_assign, inv_pos


def moe_permute_rows(x, sorted_assign, k_dev, kmax: int, x_sorted=None, stream=None):
    """-> x_sorted bf16 [T*kmax, H]: row r = x[sorted_assign[r] // kmax] for r < T*k."""
    _need(x, torch.bfloat16, "x")
    _need(sorted_assign, torch.int32, "sorted_assign")
    T, H = x.shape
    if x_sorted is None:
        x_sorted = torch.empty((max(T * kmax, 1), H), dtype=torch.bfloat16, device=x.device)
    st = lib().moe_permute_rows(_p(x), _p(sorted_assign), _p(k_dev), T, kmax, H, _p(x_sorted),
                                _stream(stream))
    check("moe_permute_rows", st)
    return x_sorted


def moe_gate_up_qmm(x, sorted_assign, expert_offsets, k_dev, kmax: int, w_q, w_s, w_b, bits: int,
                    epilogue: int = EPILOGUE_SWIGLU, out_dtype=torch.float32, out=None,
                    path: int = PATH_AUTO, stream=None, T: Optional[int] = None):
    """x bf16 [T, H] read through sorted_assign, or (sorted_assign None) the
    rows already in sorted order, [T*kmax, H]; then T must be given."""
    _need(x, torch.bfloat16, "x")
    if sorted_assign is None:
        if T is None:
            raise ValueError("T is required when x is already in sorted row order")
        H = x.shape[1]
    else:
        T, H = x.shape
    E, n_rows = w_q.shape[0], w_q.shape[1]
    cols = n_rows // 2 if epilogue == EPILOGUE_SWIGLU else n_rows
    if out is None:
        out = torch.empty((max(T * kmax, 1), cols), dtype=out_dtype, device=x.device)
    st = lib().moe_gate_up_qmm(_p(x), _p(sorted_assign), _p(expert_offsets), _p(k_dev), T, kmax, E,
                               H, n_rows, _p(w_q), _p(w_s), _p(w_b), bits, epilogue,
                               _DT[out.dtype], _p(out), path, _stream(stream))
    check("moe_gate_up_qmm", st)
    return out


def moe_down_qmm(h, expert_offsets, k_dev, T: int, kmax: int, w_q, w_s, w_b, bits: int, y=None,
                 path: int = PATH_AUTO, stream=None, y_dtype=torch.float32):
    """y: fp32 or bf16 [T*kmax, H] (allocated as ``y_dtype`` when not given)."""
    E, H = w_q.shape[0], w_q.shape[1]
    I = h.shape[1]
    if y is None:
        y = torch.empty((max(T * kmax, 1), H), dtype=y_dtype, device=h.device)
    st = lib().moe_down_qmm(_p(h), _DT[h.dtype], _p(expert_offsets), _p(k_dev), T, kmax, E, I, H,
                            _p(w_q), _p(w_s), _p(w_b), bits, _p(y), _DT[y.dtype], path,
                            _stream(stream))
    check("moe_down_qmm", st)
    return y


def moe_combine(y, inv_pos, topk_w, k_dev, T: int, kmax: int, out=None, stream=None):
    H = y.shape[1]
    if out is None:
        out = torch.empty((T, H), dtype=torch.bfloat16, device=y.device)
    st = lib().moe_combine(_p(y), _DT[y.dtype], _p(inv_pos), _p(topk_w), _p(k_dev), T, kmax, H,
                           _p(out), _stream(stream))
    check("moe_combine", st)
    return out


def moe_swiglu(gate, up, k_dev, T: int, kmax: int, out_dtype=torch.float32, out=None,
               stream=None):
    I = gate.shape[1]
    if out is None:
        out = torch.empty((max(T * kmax, 1), I), dtype=out_dtype, device=gate.device)
    st = lib().moe_swiglu(_p(gate), _p(up), _p(k_dev), T, kmax, I, _DT[out.dtype], _p(out),
                          _stream(stream))
    check("moe_swiglu", st)
    return out


def moe_selftest_wait_timeout(budget_cycles: int = 2_000_000, stream=None) -> None:
    """Launch the bounded-wait self-test (a wait that runs out on purpose)."""
    check("moe_selftest_wait_timeout",
          lib().moe_selftest_wait_timeout(int(budget_cycles), _stream(stream)))


def moe_expert_counts_accumulate(expert_counts, window_counts, stream=None):
    """window_counts (int64 [E]) += expert_counts (int32 [E]), on the device."""
    _need(expert_counts, torch.int32, "expert_counts")
    _need(window_counts, torch.int64, "window_counts")
    E = window_counts.numel()
    if expert_counts.numel() != E:
        raise ValueError("expert_counts and window_counts differ in length")
    check("moe_expert_counts_accumulate",
          lib().moe_expert_counts_accumulate(_p(expert_counts), E, _p(window_counts),
                                             _stream(stream)))
    return window_counts


def moe_expert_health(window_counts, least=None, mean_std=None, stream=None):
    """Least-activated expert (int32 [1]) and (mean, population std) of the
    window's counts (float64 [2]), both left on the device."""
    _need(window_counts, torch.int64, "window_counts")
    dev = window_counts.device
    if least is None:
        least = torch.empty(1, dtype=torch.int32, device=dev)
    if mean_std is None:
        mean_std = torch.empty(2, dtype=torch.float64, device=dev)
    check("moe_expert_health",
          lib().moe_expert_health(_p(window_counts), window_counts.numel(), _p(least),
                                  _p(mean_std), _stream(stream)))
    return least, mean_std


def moe_get_device_error(clear: bool = True, stream=None) -> int:
    v = ctypes.c_uint32(0)
    st = lib().moe_get_device_error(ctypes.byref(v), int(clear), _stream(stream))
    check("moe_get_device_error", st)
    return int(v.value)
