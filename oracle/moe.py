"""The oracle's stages (see the package docstring; test infrastructure only)."""
from __future__ import annotations

import ctypes
import dataclasses
from typing import Optional, Sequence

import numpy as np

from . import _build

__all__ = [
    "router_logits", "softmax_entropy", "batch_mean_entropy", "entropy_k", "topk_ids",
    "routing_weights", "group_top1_ids", "route", "Routing", "permute", "Permutation", "unpack_codes",
    "dequant", "DROPPED", "QDesc", "can_fuse", "pack_gate_up", "qmm_raw", "silu", "swiglu",
    "moe_forward", "Forward", "dense_masked_forward", "bf16_to_f64", "f64_to_bf16_bits",
    "ENTROPY_THRESHOLDS", "expert_health",
]

# Entropy bands of the adaptive top-k rule, page [B] section 2.2.
ENTROPY_THRESHOLDS = (1.2, 2.5)

_lib = None


def _router_lib():
    global _lib
    if _lib is None:
        lib = ctypes.CDLL(_build.build())
        vp = ctypes.c_void_p
        lib.oracle_router_logits.argtypes = [vp, vp, vp, ctypes.c_float, ctypes.c_int,
                                             ctypes.c_int, ctypes.c_int, vp]
        lib.oracle_router_logits.restype = ctypes.c_int
        _lib = lib
    return _lib


def bf16_to_f64(x_bits: np.ndarray) -> np.ndarray:
    """Raw bf16 bit patterns (uint16) -> float64, exactly."""
    return (np.asarray(x_bits, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def f64_to_bf16_bits(a: np.ndarray) -> np.ndarray:
    """float64 -> raw bf16 bit patterns, through fp32: round to nearest even
    to fp32, then to nearest even to bf16 (the layer rounds its fp32 output
    the same way; a chained layer's input is the previous layer's output).
    Finite values only."""
    b = np.asarray(a, dtype=np.float64).astype(np.float32).view(np.uint32).astype(np.uint64)
    b = (b + 0x7FFF + ((b >> 16) & 1)) >> 16
    return b.astype(np.uint16)


# --------------------------------------------------------------------------
# Routing: page [A] section 4.1 (linear -> softmax -> top-k), page [B]
# sections 2.1-2.2 (top-k routing; entropy-aware choice of k per batch).
# --------------------------------------------------------------------------

def router_logits(x_bits: np.ndarray, router_w: np.ndarray, logit_bias: Optional[np.ndarray],
                  inv_temperature: float = 1.0) -> np.ndarray:
    """fp32 logits [T, E] = (x . W[e] + bias[e]) * inv_temperature, in the
    fixed summation order documented in router_fp32.c."""
    x = np.ascontiguousarray(x_bits, dtype=np.uint16)
    w = np.ascontiguousarray(router_w, dtype=np.float32)
    T, H = x.shape
    E = w.shape[0]
    assert w.shape == (E, H)
    out = np.empty((T, E), dtype=np.float32)
    bias = None if logit_bias is None else np.ascontiguousarray(logit_bias, dtype=np.float32)
    rc = _router_lib().oracle_router_logits(
        x.ctypes.data_as(ctypes.c_void_p), w.ctypes.data_as(ctypes.c_void_p),
        None if bias is None else bias.ctypes.data_as(ctypes.c_void_p),
        ctypes.c_float(inv_temperature), T, H, E, out.ctypes.data_as(ctypes.c_void_p))
    if rc != 0:
        raise ValueError("router logits: H must be a multiple of 8")
    return out


def softmax_entropy(logits: np.ndarray) -> np.ndarray:
    """Per-token Shannon entropy (nats) of softmax(logits), float32 [T].

    The entropy decides an integer (the batch's k), so it is taken in the
    precision of the device path, fp32: H = -sum_e p_e ln p_e."""
    l = np.asarray(logits, dtype=np.float32)
    z = l - l.max(axis=1, keepdims=True)
    ez = np.exp(z)
    p = ez / ez.sum(axis=1, keepdims=True, dtype=np.float32)
    with np.errstate(divide="ignore", invalid="ignore"):
        terms = np.where(p > 0, p * np.log(p), np.float32(0.0)).astype(np.float32)
    return (-terms.sum(axis=1, dtype=np.float32)).astype(np.float32)


def batch_mean_entropy(h: np.ndarray) -> np.float32:
    h = np.asarray(h, dtype=np.float32)
    return np.float32(h.sum(dtype=np.float32) / np.float32(len(h)))


def entropy_k(mean_entropy, thresholds: Sequence[float] = ENTROPY_THRESHOLDS) -> int:
    """Page [B] section 2.2: H < 1.2 -> top-1; 1.2 <= H < 2.5 -> top-2;
    H >= 2.5 -> top-3.  Compared in fp32."""
    h = np.float32(mean_entropy)
    if h < np.float32(thresholds[0]):
        return 1
    if h < np.float32(thresholds[1]):
        return 2
    return 3


def topk_ids(logits: np.ndarray, k: int) -> np.ndarray:
    """Ids of the k largest logits per token, largest first; equal logits
    go to the lower expert id.  Softmax is strictly increasing, so these are
    also the k largest probabilities."""
    order = np.argsort(-np.asarray(logits, dtype=np.float32), axis=1, kind="stable")
    return order[:, :k].astype(np.int32)


def group_top1_ids(logits: np.ndarray, groups: int) -> np.ndarray:
    """Group-limited selection, page [A] section 1.1: the E experts form
    `groups` groups of E/groups consecutive ids and each token takes the best
    expert of every group (equal logits: the lower id).  The winners are
    listed largest logit first, equal logits by lower id, as topk_ids lists
    its choice."""
    l = np.asarray(logits, dtype=np.float32)
    T, E = l.shape
    assert groups > 0 and E % groups == 0
    gsz = E // groups
    out = np.empty((T, groups), dtype=np.int32)
    for t in range(T):
        winners = []
        for g in range(groups):
            lo = g * gsz
            seg = l[t, lo:lo + gsz]
            best = lo + int(np.argmax(seg))  # argmax returns the first maximum
            winners.append(best)
        winners.sort(key=lambda e: (-float(l[t, e]), e))
        out[t] = winners
    return out


def routing_weights(logits: np.ndarray, ids: np.ndarray, renormalize: bool = True) -> np.ndarray:
    """Softmax probabilities of the chosen experts in float64, either
    renormalised to sum to 1 over the chosen k, or as plain softmax values."""
    l = np.asarray(logits, dtype=np.float32).astype(np.float64)
    ez = np.exp(l - l.max(axis=1, keepdims=True))
    sel = np.take_along_axis(ez, ids.astype(np.int64), axis=1)
    denom = sel.sum(axis=1, keepdims=True) if renormalize else ez.sum(axis=1, keepdims=True)
    return sel / denom


@dataclasses.dataclass
class Routing:
    logits: np.ndarray        # float32 [T, E]
    ids: np.ndarray           # int32 [T, kmax], -1 past k
    weights: np.ndarray       # float64 [T, kmax], 0 past k
    k: int
    mean_entropy: np.float32
    token_entropy: np.ndarray  # float32 [T]


def route(x_bits, router_w, logit_bias=None, inv_temperature=1.0, k_fixed=2, kmax=None,
          renormalize=True, thresholds=ENTROPY_THRESHOLDS, groups=0) -> Routing:
    """Router logits, softmax, entropy, k (fixed, or adaptive when k_fixed=0)
    and the top-k ids and weights, padded to kmax slots.  groups > 0: the
    group-limited rule (one expert per group, k = groups)."""
    logits = router_logits(x_bits, router_w, logit_bias, inv_temperature)
    ent = softmax_entropy(logits)
    hbar = batch_mean_entropy(ent) if len(ent) else np.float32(0.0)
    k = int(k_fixed) if k_fixed > 0 else entropy_k(hbar, thresholds)
    if kmax is None:
        kmax = k if k_fixed > 0 else 3
    assert k <= kmax
    T = logits.shape[0]
    ids = np.full((T, kmax), -1, dtype=np.int32)
    w = np.zeros((T, kmax), dtype=np.float64)
    if T:
        if groups > 0:
            assert k == groups
            ids[:, :k] = group_top1_ids(logits, groups)
        else:
            ids[:, :k] = topk_ids(logits, k)
        w[:, :k] = routing_weights(logits, ids[:, :k], renormalize)
    return Routing(logits, ids, w, k, hbar, ent)


# --------------------------------------------------------------------------
# Grouping by expert: page [C] section 如何验证正确性 (the sorted path that
# groups token indices by expert), page [B] section 4.2 (per-expert counts).
# --------------------------------------------------------------------------

@dataclasses.dataclass
class Permutation:
    counts: np.ndarray         # int32 [E]
    offsets: np.ndarray        # int32 [E+1]
    sorted_assign: np.ndarray  # int32 [T*k] flat assignment a = t*kmax + j, grouped by expert
    inv_pos: np.ndarray        # int32 [T*kmax]: position of a in sorted_assign, -1 if j >= k,
                               # DROPPED if the expert's capacity turned it away


# inv_pos of an assignment dropped by an expert's capacity
DROPPED = -2


def permute(ids: np.ndarray, k: int, E: int, capacity: Optional[int] = None) -> Permutation:
    """Stable sort of the assignments (t, j), j < k, by expert id.

    capacity C (page [B] sections 4.3 and 5.2, expert_capacity): an expert
    takes at most C assignments per batch, those of the lowest a = t*kmax + j
    (the first C of its stable group); the rest are dropped, contribute
    nothing to the output, and the kept weights stay as they are."""
    T, kmax = ids.shape
    flat = (np.arange(T)[:, None] * kmax + np.arange(k)[None, :]).ravel()
    experts = ids[:, :k].ravel().astype(np.int64)
    order = np.argsort(experts, kind="stable")
    grouped = flat[order].astype(np.int32)
    full_counts = np.bincount(experts, minlength=E).astype(np.int32)
    inv_pos = np.full(T * kmax, -1, dtype=np.int32)
    if capacity is None:
        counts = full_counts
        sorted_assign = grouped
    else:
        assert capacity >= 0
        counts = np.minimum(full_counts, capacity).astype(np.int32)
        starts = np.concatenate([[0], np.cumsum(full_counts)])
        keep = []
        for e in range(E):
            seg = grouped[starts[e]:starts[e + 1]]
            keep.append(seg[:capacity])
            inv_pos[seg[capacity:]] = DROPPED
        sorted_assign = (np.concatenate(keep) if keep else grouped[:0]).astype(np.int32)
    offsets = np.concatenate([[0], np.cumsum(counts)]).astype(np.int32)
    inv_pos[sorted_assign] = np.arange(len(sorted_assign), dtype=np.int32)
    return Permutation(counts, offsets, sorted_assign, inv_pos)


# --------------------------------------------------------------------------
# Affine group quantization and the gate/up fusion, page [C] sections
# 融合原理 and 实现剖析 ② ③.
# --------------------------------------------------------------------------

def unpack_codes(q_words: np.ndarray, bits: int, cols: int) -> np.ndarray:
    """uint32 words -> codes [..., cols]: element i at bits [bits*i, bits*i +
    bits) of the row's little-endian bit stream (for 4 and 8 bits: word
    i/(32/bits), bit offset bits*(i mod 32/bits))."""
    # Little-endian words: byte j of a word holds elements 2j (low nibble) and
    # 2j+1 (high nibble) for 4-bit codes, element j for 8-bit codes.
    q = np.asarray(q_words)
    by = np.ascontiguousarray(q, dtype="<u4").view(np.uint8)
    if bits == 8:
        codes = by
    elif bits == 4:
        codes = np.empty(by.shape[:-1] + (2 * by.shape[-1],), dtype=np.uint8)
        codes[..., 0::2] = by & 0x0F
        codes[..., 1::2] = by >> 4
    elif bits in (5, 6):
        # bit j of the stream is bit j % 8 of byte j / 8
        stream = np.unpackbits(by, axis=-1, bitorder="little")[..., :cols * bits]
        digits = stream.reshape(stream.shape[:-1] + (cols, bits)).astype(np.uint16)
        codes = (digits << np.arange(bits, dtype=np.uint16)).sum(-1).astype(np.uint8)
    else:
        raise ValueError("bits must be 4, 5, 6 or 8")
    return codes.reshape(*q.shape[:-1], cols)


def dequant(q_words, scales, biases, bits: int, cols: int, group: int = 64) -> np.ndarray:
    """w = scale * code + bias, scale and bias shared by `group` consecutive
    elements along the row (the contraction axis).  float64, exact."""
    codes = unpack_codes(q_words, bits, cols).astype(np.float64)
    lead = codes.shape[:-1]
    w = codes.reshape(lead + (cols // group, group))
    w *= np.asarray(scales).astype(np.float64)[..., None]
    w += np.asarray(biases).astype(np.float64)[..., None]
    return w.reshape(lead + (cols,))


@dataclasses.dataclass(frozen=True)
class QDesc:
    """What the fusion eligibility check compares (page [C] 实现剖析 ②)."""
    quantized: bool
    bits: int
    group: int
    mode: str
    has_bias: bool
    rows: int
    cols: int
    scale_dtype: str


def can_fuse(gate: QDesc, up: QDesc) -> bool:
    """Gate and up are fused only when they are the same kind of projection
    with identical group size, bits and mode, the same presence of a bias,
    and the same shape and dtype."""
    return gate == up


def pack_gate_up(gate_q, gate_s, gate_b, up_q, up_s, up_b):
    """Concatenate [gate; up] along the output axis of every expert: codes,
    scales and biases each become [E, 2*rows, ...] (page [C] 实现剖析 ③)."""
    return (np.concatenate([gate_q, up_q], axis=1), np.concatenate([gate_s, up_s], axis=1),
            np.concatenate([gate_b, up_b], axis=1))


def qmm_raw(x_rows: np.ndarray, q, s, b, bits: int, cols: int) -> np.ndarray:
    """x_rows [m, cols] (float64) times one expert's dequantized matrix
    [rows, cols] transposed -> [m, rows]."""
    return np.asarray(x_rows, dtype=np.float64) @ dequant(q, s, b, bits, cols).T


def silu(z: np.ndarray) -> np.ndarray:
    with np.errstate(over="ignore"):
        return z / (1.0 + np.exp(-z))


def swiglu(gate_out: np.ndarray, up_out: np.ndarray) -> np.ndarray:
    """SwitchGLU activation: SiLU(gate) * up (page [C] 实现剖析 ④)."""
    return silu(gate_out) * up_out


# --------------------------------------------------------------------------
# The layer: page [A] section 4.2 (only the chosen experts run; output is the
# routing-weighted sum of their outputs) and page [C] 实现剖析 ④ (one gate_up
# product split into halves, activation, down projection).
# --------------------------------------------------------------------------

@dataclasses.dataclass
class Forward:
    routing: Routing
    perm: Permutation
    out: np.ndarray            # float64 [T, H] (rows of tokens not computed are NaN)
    h: Optional[np.ndarray]    # float64 [A, I] in sorted order (NaN rows skipped)
    y: Optional[np.ndarray]    # float64 [A, H] in sorted order
    computed_tokens: np.ndarray


def moe_forward(x_bits, layer, k_fixed=None, kmax=None, inv_temperature=None, renormalize=True,
                tokens=None, keep_intermediates=True, routing: Optional[Routing] = None,
                capacity: Optional[int] = None) -> Forward:
    """Whole-layer forward.  `layer` is a workloads.LayerInputs (gate and up
    are fused here with pack_gate_up).  `tokens` restricts the expert math to
    a subset of token indices (routing always covers the whole batch, since
    the adaptive k depends on all of it)."""
    cfg = layer.cfg
    if k_fixed is None:
        k_fixed = cfg.k
    if kmax is None:
        kmax = cfg.slots
    if inv_temperature is None:
        inv_temperature = cfg.inv_temperature(0)
    if routing is None:
        routing = route(x_bits, layer.router_w, layer.logit_bias, inv_temperature, k_fixed, kmax,
                        renormalize)
    T, H = x_bits.shape
    I, E, bits = cfg.I, cfg.E, cfg.bits
    k = routing.k
    perm = permute(routing.ids, k, E, capacity)
    want = np.ones(T, dtype=bool) if tokens is None else np.isin(np.arange(T), tokens)
    A = len(perm.sorted_assign)
    h_all = np.full((A, I), np.nan) if keep_intermediates else None
    y_all = np.full((A, H), np.nan)
    xf = bf16_to_f64(x_bits)
    for e in range(E):
        lo, hi = int(perm.offsets[e]), int(perm.offsets[e + 1])
        rows = np.arange(lo, hi)
        rows = rows[want[perm.sorted_assign[rows] // kmax]]
        if len(rows) == 0:
            continue
        toks = perm.sorted_assign[rows] // kmax
        gu_q, gu_s, gu_b = pack_gate_up(layer.gate.q[e:e + 1], layer.gate.s[e:e + 1],
                                        layer.gate.b[e:e + 1], layer.up.q[e:e + 1],
                                        layer.up.s[e:e + 1], layer.up.b[e:e + 1])
        gu = qmm_raw(xf[toks], gu_q[0], gu_s[0], gu_b[0], bits, H)      # [m, 2I]
        h = swiglu(gu[:, :I], gu[:, I:])                                 # [m, I]
        y = qmm_raw(h, layer.down.q[e], layer.down.s[e], layer.down.b[e], bits, I)  # [m, H]
        if h_all is not None:
            h_all[rows] = h
        y_all[rows] = y
    out = np.full((T, H), np.nan)
    for t in np.nonzero(want)[0]:
        acc = np.zeros(H)
        for j in range(k):
            r = perm.inv_pos[t * kmax + j]
            if r == DROPPED:
                continue
            acc = acc + routing.weights[t, j] * y_all[r]
        out[t] = acc
    return Forward(routing, perm, out, h_all, y_all if keep_intermediates else None,
                   np.nonzero(want)[0])


def dense_masked_forward(x_bits, layer, routing: Routing) -> np.ndarray:
    """Brute force: run every expert on every token, then sum over experts
    in id order with the routing weight of each (zero for experts that were
    not chosen).  Float64; for tiny inputs only."""
    cfg = layer.cfg
    T, H = x_bits.shape
    xf = bf16_to_f64(x_bits)
    mask = np.zeros((T, cfg.E))
    for t in range(T):
        for j in range(routing.k):
            mask[t, routing.ids[t, j]] = routing.weights[t, j]
    out = np.zeros((T, H))
    for e in range(cfg.E):
        wg = dequant(layer.gate.q[e], layer.gate.s[e], layer.gate.b[e], cfg.bits, H)
        wu = dequant(layer.up.q[e], layer.up.s[e], layer.up.b[e], cfg.bits, H)
        wd = dequant(layer.down.q[e], layer.down.s[e], layer.down.b[e], cfg.bits, cfg.I)
        ye = swiglu(xf @ wg.T, xf @ wu.T) @ wd.T
        out = out + mask[:, e:e + 1] * ye
    return out


# --------------------------------------------------------------------------
# Expert health: page [B] section 6 (per window, the least-activated expert
# and the standard deviation of all experts' activation counts) and section
# 4.2 (activation counts per expert).
# --------------------------------------------------------------------------
def expert_health(window_counts) -> tuple:
    """(least-activated expert id, mean, population standard deviation) of a
    window's per-expert activation counts; equal counts go to the lower id."""
    c = np.asarray(window_counts, dtype=np.int64)
    E = c.size
    least = int(np.argmin(c))
    mean = float(c.sum()) / E
    std = float(np.sqrt(((c.astype(np.float64) - mean) ** 2).sum() / E))
    return least, mean, std
