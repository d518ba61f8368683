"""Seeded synthetic workloads for the quantized sparse-MoE layer forward.

This module serves the tests, the oracle checks and the benchmark alike.  It
defines the five workload shapes and draws their inputs; it contains none of
the layer's arithmetic.  Weights are drawn N(0, sigma) and quantized by a
min-max affine quantizer (group 64 along each matrix's contraction axis,
fp16 scale and bias), activations are N(0, 1) rounded to bf16.  All draws come
from the counter-based generator in ``synth.c`` (seed 0 by default).

Stream ids: 1 router weight, 2 gate, 3 up, 4 down, 5+b activations of batch b.
"""
from __future__ import annotations

import ctypes
import dataclasses
import os
from typing import Optional

import numpy as np

from . import _build

STREAM_ROUTER, STREAM_GATE, STREAM_UP, STREAM_DOWN, STREAM_X = 1, 2, 3, 4, 5


@dataclasses.dataclass(frozen=True)
class MoEConfig:
    name: str
    H: int            # hidden size (contraction axis of gate/up)
    I: int            # expert intermediate size (contraction axis of down)
    E: int            # number of experts
    k: int            # experts per token; 0 = batch-entropy adaptive top-1/2/3
    T: int            # tokens per layer call
    bits: int = 4     # code width of the affine-quantized expert weights
    kmax: int = 0     # routing slots per token (defaults to k, or 3 when adaptive)
    calls: int = 1    # independent layer calls per step (batch-1 decode uses 256)
    x_std: float = 1.0
    router_std: float = 0.02
    w_std: float = 0.02
    zipf_s: float = 0.0     # > 0: add -s*ln(rank) to expert e's logit (rank = e+1)
    batches: int = 1        # distinct activation batches (entropy workload uses 3)
    inv_temperatures: tuple = ()  # per batch; empty = 1.0

    @property
    def slots(self) -> int:
        if self.kmax:
            return self.kmax
        return self.k if self.k > 0 else 3

    def inv_temperature(self, batch: int = 0) -> float:
        return float(self.inv_temperatures[batch]) if self.inv_temperatures else 1.0

    def scaled(self, **kw) -> "MoEConfig":
        return dataclasses.replace(self, **kw)


# Inverse router temperatures of the three entropy-workload batches.  They are
# chosen so that the batch-mean routing entropy sits mid-band of the k=1, k=2
# and k=3 ranges (targets 0.6, 1.85, 3.0 nats).  The values were written by
# tests/golden/make_entropy_temperatures.py, which bisects with the oracle.
ENTROPY_INV_TEMPERATURES = (5.716348, 1.863968, 0.795742)

CONFIGS = {
    "tiny": MoEConfig("tiny", H=256, I=512, E=8, k=2, T=16, bits=4, router_std=0.05),
    "decode": MoEConfig("decode", H=4096, I=11008, E=64, k=4, T=1, calls=256, bits=4),
    "batched": MoEConfig("batched", H=4096, I=1536, E=64, k=4, T=64, bits=4, zipf_s=1.1),
    "prefill": MoEConfig("prefill", H=2048, I=768, E=128, k=8, T=4096, bits=4),
    "entropy": MoEConfig("entropy", H=4096, I=1536, E=32, k=0, T=512, bits=8, batches=3,
                         inv_temperatures=ENTROPY_INV_TEMPERATURES),
}

_lib = None


def _synth():
    global _lib
    if _lib is None:
        path = _build.build()
        lib = ctypes.CDLL(path)
        u64, i64 = ctypes.c_uint64, ctypes.c_int64
        vp = ctypes.c_void_p
        lib.synth_normal_f32.argtypes = [u64, u64, u64, i64, ctypes.c_double, vp]
        lib.synth_normal_bf16.argtypes = [u64, u64, u64, i64, ctypes.c_double, vp]
        lib.synth_quantized.argtypes = [u64, u64, i64, i64, ctypes.c_int, ctypes.c_int,
                                        ctypes.c_double, vp, vp, vp, vp, ctypes.c_int]
        lib.synth_quantized.restype = ctypes.c_int
        _lib = lib
    return _lib


def _ptr(a: Optional[np.ndarray]):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _threads() -> int:
    return max(1, min(32, os.cpu_count() or 1))


def normal_f32(seed: int, stream: int, shape, sigma: float, start: int = 0) -> np.ndarray:
    out = np.empty(shape, dtype=np.float32)
    _synth().synth_normal_f32(seed, stream, start, out.size, sigma, _ptr(out))
    return out


def normal_bf16(seed: int, stream: int, shape, sigma: float, start: int = 0) -> np.ndarray:
    """N(0, sigma) rounded to bf16; returned as the raw uint16 bit patterns."""
    out = np.empty(shape, dtype=np.uint16)
    _synth().synth_normal_bf16(seed, stream, start, out.size, sigma, _ptr(out))
    return out


@dataclasses.dataclass
class QuantMatrix:
    """Affine-quantized weights of E experts, each [rows, cols]."""
    q: np.ndarray   # uint32 [E, rows, cols*bits/32]
    s: np.ndarray   # float16 [E, rows, cols/64]
    b: np.ndarray   # float16 [E, rows, cols/64]
    bits: int
    cols: int
    group: int = 64

    @property
    def E(self) -> int:
        return self.q.shape[0]

    @property
    def rows(self) -> int:
        return self.q.shape[1]


def quantized(seed: int, stream: int, E: int, rows: int, cols: int, bits: int, sigma: float,
              experts=None, return_float: bool = False):
    """Draw and quantize expert weights.  ``experts`` selects a subset (the
    draws of expert e never depend on which others are generated)."""
    ex = list(range(E)) if experts is None else list(experts)
    n = len(ex)
    q = np.empty((n, rows, cols * bits // 32), dtype=np.uint32)
    s = np.empty((n, rows, cols // 64), dtype=np.float16)
    b = np.empty((n, rows, cols // 64), dtype=np.float16)
    w = np.empty((n, rows, cols), dtype=np.float32) if return_float else None
    lib = _synth()
    for i, e in enumerate(ex):
        rc = lib.synth_quantized(seed, stream, e * rows, rows, cols, bits, sigma,
                                 _ptr(q[i]), _ptr(s[i]), _ptr(b[i]),
                                 _ptr(w[i]) if w is not None else None, _threads())
        if rc != 0:
            raise ValueError("synth_quantized rejected its arguments")
    qm = QuantMatrix(q=q, s=s, b=b, bits=bits, cols=cols)
    return (qm, w) if return_float else qm


@dataclasses.dataclass
class LayerInputs:
    cfg: MoEConfig
    router_w: np.ndarray            # float32 [E, H]
    logit_bias: Optional[np.ndarray]  # float32 [E] or None
    gate: QuantMatrix               # [E, I, H]
    up: QuantMatrix                 # [E, I, H]
    down: QuantMatrix               # [E, H, I]


def zipf_log_prior(E: int, s: float) -> np.ndarray:
    return (-s * np.log(np.arange(1, E + 1, dtype=np.float64))).astype(np.float32)


def make_layer(cfg: MoEConfig, seed: int = 0) -> LayerInputs:
    router_w = normal_f32(seed, STREAM_ROUTER, (cfg.E, cfg.H), cfg.router_std)
    bias = zipf_log_prior(cfg.E, cfg.zipf_s) if cfg.zipf_s > 0 else None
    gate = quantized(seed, STREAM_GATE, cfg.E, cfg.I, cfg.H, cfg.bits, cfg.w_std)
    up = quantized(seed, STREAM_UP, cfg.E, cfg.I, cfg.H, cfg.bits, cfg.w_std)
    down = quantized(seed, STREAM_DOWN, cfg.E, cfg.H, cfg.I, cfg.bits, cfg.w_std)
    return LayerInputs(cfg, router_w, bias, gate, up, down)


def make_tokens(cfg: MoEConfig, seed: int = 0, batch: int = 0) -> np.ndarray:
    """bf16 activations (uint16 bits) for all calls of one batch: [calls*T, H]."""
    return normal_bf16(seed, STREAM_X + batch, (cfg.calls * cfg.T, cfg.H), cfg.x_std)


def bf16_bits_to_f32(x: np.ndarray) -> np.ndarray:
    """Widen raw bf16 bit patterns to float32 (exact)."""
    return (x.astype(np.uint32) << 16).view(np.float32)
