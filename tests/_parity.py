"""Helpers shared by the GPU parity tests (device plumbing and comparisons)."""
import numpy as np
import torch

import oracle
import workloads

# Layer-output tolerance fixed for this layer: bf16 out, fp32 accumulation,
# against the float64 oracle on the dequantized weights.
REL_L2 = 5e-3
MAX_REL = 1e-2


def rel_l2(a, ref):
    a = np.asarray(a, np.float64)
    ref = np.asarray(ref, np.float64)
    return float(np.linalg.norm(a - ref) / max(np.linalg.norm(ref), 1e-300))


def assert_layer_close(got, ref, what=""):
    got = np.asarray(got, np.float64)
    ref = np.asarray(ref, np.float64)
    e = rel_l2(got, ref)
    m = float(np.abs(got - ref).max()) if ref.size else 0.0
    assert e <= REL_L2, f"{what}: relative L2 {e:.3e} > {REL_L2}"
    assert m <= MAX_REL * float(np.abs(ref).max()), f"{what}: max err {m:.3e}"
    return e


def dev():
    return torch.device("cuda:0")


def to_np(t):
    if t.dtype == torch.bfloat16:
        return t.float().cpu().numpy().astype(np.float64)
    return t.cpu().numpy()


def route_gpu(moe, x_bits, layer_np, k_fixed, kmax, inv_t=1.0, renorm=True):
    d = dev()
    x = moe.bf16_from_bits(x_bits, d)
    w = torch.from_numpy(layer_np.router_w).to(d)
    lb = None if layer_np.logit_bias is None else torch.from_numpy(layer_np.logit_bias).to(d)
    ids, tw, kd, me = moe.moe_router_topk(x, w, lb, inv_t, k_fixed, kmax, renormalize=renorm)
    return x, ids, tw, kd, me
