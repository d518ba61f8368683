"""MoELayer: the six C-ABI calls composed into one quantized SwitchGLU MoE layer.

Pages: "Qwen3.5 Block在llama.cpp中的映射与优化原理" section 4 (router, then
only the chosen experts' FFN, then the weighted sum); "oMLX MoE gate/up 融合
优化：qwen35_moe_gate_up 实现剖析" (gate and up fused once at load, one
gate_up product per layer; the environment switch turns fusion off).
"""
from __future__ import annotations

import dataclasses
import os
from typing import Optional

import numpy as np
import torch

from . import binding as B
from ._lib import (EPILOGUE_RAW, EPILOGUE_SWIGLU, PATH_AUTO, PATH_FLAG_WEIGHTS_EARLY, PATH_GEMV,
                   PATH_TC, MoEError, path_k_range)

FUSE_ENV = "MOE_GB300_FUSE_GATE_UP"
TC_MIN_TOKENS_PER_EXPERT = 24  # mirrors the library's automatic path choice
TC_BUILT = True                # the tensor-core grouped GEMM (tcgen05) is available


@dataclasses.dataclass
class QTensor:
    """Affine-quantized weights of E experts on the device."""
    q: torch.Tensor  # uint32 [E, rows, cols*bits/32]
    s: torch.Tensor  # float16 [E, rows, cols/64]
    b: torch.Tensor  # float16 [E, rows, cols/64]
    bits: int

    @property
    def rows(self) -> int:
        return self.q.shape[1]

    @property
    def cols(self) -> int:
        return self.q.shape[2] * 32 // self.bits


def qtensor_from_numpy(m, device) -> QTensor:
    """Upload a workloads.QuantMatrix (numpy) to the device."""
    q = torch.from_numpy(np.ascontiguousarray(m.q)).to(device)
    s = torch.from_numpy(np.ascontiguousarray(m.s)).to(device)
    b = torch.from_numpy(np.ascontiguousarray(m.b)).to(device)
    return QTensor(q, s, b, m.bits)


def bf16_from_bits(x_bits: np.ndarray, device=None, pin: bool = False) -> torch.Tensor:
    t = torch.from_numpy(np.ascontiguousarray(x_bits, dtype=np.uint16)).view(torch.bfloat16)
    if pin:
        t = t.pin_memory()
    return t.to(device) if device is not None else t


class MoELayer:
    """Forward of one quantized sparse-MoE SwitchGLU layer on one GPU.

    k_fixed > 0 routes every token to k experts; k_fixed = 0 applies the
    batch-entropy rule (k in {1, 2, 3}, kmax = 3).  ``fuse_gate_up`` (default:
    the environment variable MOE_GB300_FUSE_GATE_UP, on unless "0") packs
    gate and up once here; unfused layers run two RAW products plus the
    separate activation.  ``path`` forces a kernel family for the products.
    ``groups`` > 0 routes each token to the best expert of each of ``groups``
    groups of consecutive expert ids (k_fixed must equal it).  ``capacity``
    limits the assignments each expert takes per call (the lowest token
    slots stay; the others are dropped).  ``y_dtype`` is the storage type of
    the down product's rows between the down and combine kernels: None
    stores bf16 when a call's products run on the tensor cores (large
    batches, where y is hundreds of MB written and read again) and fp32
    otherwise.
    """

    def __init__(self, router_w: torch.Tensor, logit_bias: Optional[torch.Tensor], gate: QTensor,
                 up: QTensor, down: QTensor, k_fixed: int, kmax: Optional[int] = None,
                 inv_temperature: float = 1.0, renormalize: bool = True,
                 thresholds=(1.2, 2.5), fuse_gate_up: Optional[bool] = None,
                 path: int = PATH_AUTO, free_sources: bool = False, groups: int = 0,
                 capacity: Optional[int] = None, y_dtype: Optional[torch.dtype] = None):
        self.device = router_w.device
        self.router_w = router_w.contiguous()
        self.logit_bias = None if logit_bias is None else logit_bias.contiguous()
        self.E, self.H = router_w.shape
        self.I = gate.rows
        self.bits = gate.bits
        self.k_fixed = k_fixed
        self.kmax = kmax if kmax is not None else (k_fixed if k_fixed > 0 else 3)
        self.inv_temperature = float(inv_temperature)
        self.renormalize = renormalize
        self.thr = tuple(float(t) for t in thresholds)
        self.path = path
        self.groups = int(groups)
        self.capacity = None if capacity is None else int(capacity)
        if y_dtype not in (None, torch.float32, torch.bfloat16):
            raise ValueError("y_dtype must be None, torch.float32 or torch.bfloat16")
        self.y_dtype = y_dtype
        if self.groups > 0 and (self.E % self.groups or k_fixed != self.groups):
            raise ValueError("group-limited routing needs k_fixed == groups dividing E")
        self.down = down
        if fuse_gate_up is None:
            fuse_gate_up = os.environ.get(FUSE_ENV, "1") != "0"
        self.fused = False
        self.gate, self.up, self.gate_up = gate, up, None
        if fuse_gate_up:
            gd = B.qdesc(gate.rows, gate.cols, gate.bits)
            ud = B.qdesc(up.rows, up.cols, up.bits)
            try:
                q, s, b = B.moe_pack_gate_up(gd, ud, gate.q, gate.s, gate.b, up.q, up.s, up.b)
                self.gate_up = QTensor(q, s, b, gate.bits)
                self.fused = True
                if free_sources:
                    self.gate = self.up = None
            except MoEError as err:
                if err.status != 3:  # MOE_ERR_INCOMPATIBLE keeps the unfused path
                    raise
        self._bufs = {}

    @classmethod
    def from_workload(cls, layer_inputs, device, batch: int = 0, **kw) -> "MoELayer":
        cfg = layer_inputs.cfg
        rw = torch.from_numpy(layer_inputs.router_w).to(device)
        lb = None if layer_inputs.logit_bias is None else torch.from_numpy(layer_inputs.logit_bias).to(device)
        kw.setdefault("inv_temperature", cfg.inv_temperature(batch))
        return cls(rw, lb, qtensor_from_numpy(layer_inputs.gate, device),
                   qtensor_from_numpy(layer_inputs.up, device),
                   qtensor_from_numpy(layer_inputs.down, device), k_fixed=cfg.k,
                   kmax=cfg.slots, **kw)

    def resolved_path(self, T: int) -> int:
        """The kernel family of the products (with an adaptive k, the one for
        k = kmax; k_split says when smaller k take the other family)."""
        if self.path != PATH_AUTO:
            return self.path
        return self._family(T, self.kmax)

    def _family(self, T: int, k: int) -> int:
        if self.bits not in (4, 8):  # 5- and 6-bit codes: the GEMV family only
            return PATH_GEMV
        if (TC_BUILT and (T * k) // self.E >= TC_MIN_TOKENS_PER_EXPERT
                and min(self.H, self.I) * self.bits // 8 >= 128):
            return PATH_TC
        return PATH_GEMV

    def k_split(self, T: int) -> int:
        """With an adaptive k and the automatic path, the k (if any) from
        which the products take the tensor cores while smaller k take the
        streamed GEMV.  k is known only on the device, so both families are
        queued, each gated on its k values; 0 when one family serves every k."""
        if self.path != PATH_AUTO or self.k_fixed != 0 or not self.fused or self.E > 1024:
            return 0
        if self._family(T, 1) == self._family(T, self.kmax):
            return 0
        step = 256 if self.bits == 4 else 128  # the streamed GEMV's row granularity
        if self.H % step or self.I % step:
            return 0
        return next(k for k in range(2, self.kmax + 1) if self._family(T, k) == PATH_TC)

    def y_storage(self, T: int) -> torch.dtype:
        """Storage type of y for calls of T tokens."""
        if self.y_dtype is not None:
            return self.y_dtype
        tc = self.k_split(T) or self.resolved_path(T) == PATH_TC
        return torch.bfloat16 if tc else torch.float32

    def launches_per_call(self, T: int) -> int:
        """Kernels one forward of T tokens launches: the router (plus its
        batch finalize when the tokens span more than one token group of 32,
        16 when E > 256), the grouping (inside those launches when E <= 256
        and T * kmax <= 512, else its own kernel), the row permute on the
        tensor-core path, the gate_up product (or two RAW products and the
        activation when unfused), down and combine.  With a capacity the
        capped grouping is a kernel of its own.  When k_split is set both
        kernel families of each product are launched (one of them returns at
        once)."""
        group = 32 if self.E <= 256 else 16
        one_group = (T + group - 1) // group == 1
        n = 1 + (0 if one_group else 1)
        fused = self.E <= 256 and T * self.kmax <= 512
        if self.capacity is None:
            n += 0 if fused else 1
        else:
            # the capped grouping, after the group-limited route's own grouping
            n += 1 + ((0 if fused else 1) if self.groups > 0 else 0)
        if self.k_split(T):
            return n + 6  # row permute, two gated gate_up and two gated down launches, combine
        n += 1 if self.resolved_path(T) == PATH_TC else 0
        n += 1 if self.fused else 3
        return n + 2

    def buffers(self, T: int) -> dict:
        key = T
        if key not in self._bufs:
            dev, A = self.device, max(T * self.kmax, 1)
            # both kernel families consume h as bf16 (the GEMV's FMAs take bf16
            # operands, the tensor cores bf16 tiles)
            h_dtype = torch.bfloat16
            bufs = dict(
                topk_ids=torch.empty((T, self.kmax), dtype=torch.int32, device=dev),
                topk_w=torch.empty((T, self.kmax), dtype=torch.float32, device=dev),
                k_dev=torch.empty(1, dtype=torch.int32, device=dev),
                mean_entropy=torch.empty(1, dtype=torch.float32, device=dev),
                ws=torch.empty(B.moe_router_workspace_size(T), dtype=torch.uint8, device=dev),
                counts=torch.empty(self.E, dtype=torch.int32, device=dev),
                offsets=torch.empty(self.E + 1, dtype=torch.int32, device=dev),
                sorted=torch.empty(A, dtype=torch.int32, device=dev),
                inv_pos=torch.empty(A, dtype=torch.int32, device=dev),
                h=torch.empty((A, self.I), dtype=h_dtype, device=dev),
                x_sorted=torch.empty((A, self.H), dtype=torch.bfloat16, device=dev),
                y=torch.empty((A, self.H), dtype=self.y_storage(T), device=dev),
                out=torch.empty((T, self.H), dtype=torch.bfloat16, device=dev),
            )
            if not self.fused:
                bufs["g_raw"] = torch.empty((A, self.I), dtype=torch.float32, device=dev)
                bufs["u_raw"] = torch.empty((A, self.I), dtype=torch.float32, device=dev)
            self._bufs[key] = bufs
        return self._bufs[key]

    def forward(self, x: torch.Tensor, out: Optional[torch.Tensor] = None,
                inv_temperature: Optional[float] = None, events: Optional[dict] = None
                ) -> torch.Tensor:
        """x: bf16 [T, H] on the device.  Returns bf16 [T, H] (a reused buffer
        unless ``out`` is given).  ``events``, if given, receives per kernel
        ("router", "permute", "permute_rows", "gate_up", "down", "combine") a
        list of (start, end) CUDA events around its launches."""
        T = x.shape[0]
        b = self.buffers(T)
        path = self.resolved_path(T)
        it = self.inv_temperature if inv_temperature is None else float(inv_temperature)
        # router, top-k and the expert grouping (one launch for small batches)
        ev = _Timer(events, "route")
        if self.capacity is not None:
            # router (group-limited or top-k), then the grouping with each
            # expert's capacity (it replaces the uncapped grouping that the
            # group-limited route also writes)
            if self.groups > 0:
                B.moe_route_grouped(x, self.router_w, self.logit_bias, it, self.groups,
                                    self.kmax, self.renormalize, b["topk_ids"], b["topk_w"],
                                    b["k_dev"], b["mean_entropy"], b["ws"], b["counts"],
                                    b["offsets"], b["sorted"], b["inv_pos"])
            else:
                B.moe_router_topk(x, self.router_w, self.logit_bias, it, self.k_fixed, self.kmax,
                                  self.thr[0], self.thr[1], self.renormalize, b["topk_ids"],
                                  b["topk_w"], b["k_dev"], b["mean_entropy"], b["ws"])
            B.moe_permute_capped(b["topk_ids"], b["k_dev"], self.E, self.capacity, b["counts"],
                                 b["offsets"], b["sorted"], b["inv_pos"])
        elif self.groups > 0:
            B.moe_route_grouped(x, self.router_w, self.logit_bias, it, self.groups, self.kmax,
                                self.renormalize, b["topk_ids"], b["topk_w"], b["k_dev"],
                                b["mean_entropy"], b["ws"], b["counts"], b["offsets"],
                                b["sorted"], b["inv_pos"])
        else:
            B.moe_route(x, self.router_w, self.logit_bias, it, self.k_fixed, self.kmax,
                        self.thr[0], self.thr[1], self.renormalize, b["topk_ids"], b["topk_w"],
                        b["k_dev"], b["mean_entropy"], b["ws"], b["counts"], b["offsets"],
                        b["sorted"], b["inv_pos"])
        ev.stop()
        ks = self.k_split(T)
        if ks:
            return self._forward_k_split(x, b, ks, T, out, events)
        # tensor cores: token rows copied once into expert order, so every
        # tile loads contiguous rows; the GEMV reads x through sorted_assign
        if path == PATH_TC:
            ev = _Timer(events, "permute_rows")
            xs = B.moe_permute_rows(x, b["sorted"], b["k_dev"], self.kmax, b["x_sorted"])
            ev.stop()
            srt = None
        else:
            xs, srt = x, b["sorted"]
        ev = _Timer(events, "gate_up")
        if self.fused:
            g = self.gate_up
            B.moe_gate_up_qmm(xs, srt, b["offsets"], b["k_dev"], self.kmax, g.q, g.s, g.b,
                              self.bits, EPILOGUE_SWIGLU, b["h"].dtype, b["h"], path, T=T)
        else:
            for m, dst in ((self.gate, b["g_raw"]), (self.up, b["u_raw"])):
                B.moe_gate_up_qmm(xs, srt, b["offsets"], b["k_dev"], self.kmax, m.q, m.s,
                                  m.b, self.bits, EPILOGUE_RAW, torch.float32, dst, path, T=T)
            B.moe_swiglu(b["g_raw"], b["u_raw"], b["k_dev"], T, self.kmax, b["h"].dtype, b["h"])
        ev.stop()
        d = self.down
        ev = _Timer(events, "down")
        # the kernel just before this one (gate_up or the activation) writes
        # only h: the down weights may stream while it finishes
        B.moe_down_qmm(b["h"], b["offsets"], b["k_dev"], T, self.kmax, d.q, d.s, d.b, self.bits,
                       b["y"], path | PATH_FLAG_WEIGHTS_EARLY)
        ev.stop()
        res = out if out is not None else b["out"]
        ev = _Timer(events, "combine")
        B.moe_combine(b["y"], b["inv_pos"], b["topk_w"], b["k_dev"], T, self.kmax, res)
        ev.stop()
        return res

    def _forward_k_split(self, x, b, ks, T, out, events):
        """The products after routing when k < ks takes the streamed GEMV and
        k >= ks the tensor cores: each product's two launches are gated on k,
        so exactly one of them computes."""
        lo_gate, hi_gate = path_k_range(1, ks - 1), path_k_range(ks, self.kmax)
        ev = _Timer(events, "permute_rows")
        xs = B.moe_permute_rows(x, b["sorted"], b["k_dev"], self.kmax, b["x_sorted"])
        ev.stop()
        g = self.gate_up
        ev = _Timer(events, "gate_up")
        B.moe_gate_up_qmm(x, b["sorted"], b["offsets"], b["k_dev"], self.kmax, g.q, g.s, g.b,
                          self.bits, EPILOGUE_SWIGLU, b["h"].dtype, b["h"], PATH_GEMV | lo_gate,
                          T=T)
        B.moe_gate_up_qmm(xs, None, b["offsets"], b["k_dev"], self.kmax, g.q, g.s, g.b,
                          self.bits, EPILOGUE_SWIGLU, b["h"].dtype, b["h"], PATH_TC | hi_gate, T=T)
        ev.stop()
        d = self.down
        ev = _Timer(events, "down")
        # the GEMV's weights may stream early: the kernel ahead of it (the
        # gated tensor-core gate_up) writes only h
        B.moe_down_qmm(b["h"], b["offsets"], b["k_dev"], T, self.kmax, d.q, d.s, d.b, self.bits,
                       b["y"], PATH_GEMV | PATH_FLAG_WEIGHTS_EARLY | lo_gate)
        B.moe_down_qmm(b["h"], b["offsets"], b["k_dev"], T, self.kmax, d.q, d.s, d.b, self.bits,
                       b["y"], PATH_TC | hi_gate)
        ev.stop()
        res = out if out is not None else b["out"]
        ev = _Timer(events, "combine")
        B.moe_combine(b["y"], b["inv_pos"], b["topk_w"], b["k_dev"], T, self.kmax, res)
        ev.stop()
        return res

    __call__ = forward

    def forward_host(self, x_host: torch.Tensor, out_host: torch.Tensor,
                     inv_temperature: Optional[float] = None) -> torch.Tensor:
        """End-to-end call with host buffers: copies x (pinned host, bf16
        [T, H]) to the device, runs the layer and copies the result back into
        out_host, all enqueued on the current stream (no synchronization)."""
        T = x_host.shape[0]
        b = self.buffers(T)
        if "x_dev" not in b:
            b["x_dev"] = torch.empty((T, self.H), dtype=torch.bfloat16, device=self.device)
        b["x_dev"].copy_(x_host, non_blocking=True)
        res = self.forward(b["x_dev"], inv_temperature=inv_temperature)
        out_host.copy_(res, non_blocking=True)
        return out_host


class _Timer:
    def __init__(self, events: Optional[dict], name: str):
        self.events, self.name = events, name
        if events is not None:
            self.start = torch.cuda.Event(enable_timing=True)
            self.start.record()

    def stop(self):
        if self.events is not None:
            end = torch.cuda.Event(enable_timing=True)
            end.record()
            self.events.setdefault(self.name, []).append((self.start, end))
