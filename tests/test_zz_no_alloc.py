"""The allocation-free router entry point (moe_router_topk_noalloc).

It serves callers that cannot allocate device memory: a model runner that
keeps the whole device pool to itself and hands a plugged-in layer only its
input and output tensors, or a deployment that forbids allocation after
start-up because cudaMalloc can stall a latency-bound decode loop.  Its
scratch is a static device array inside the library, so it takes no
workspace.  This file is collected last on purpose: it runs after every
other GPU test, and also passes on its own in a fresh process.
"""
import ctypes

import numpy as np
import pytest
import torch

import oracle
import workloads

pytestmark = pytest.mark.gpu

MAX_TOKENS = 65536  # MOE_ROUTER_NOALLOC_MAX_TOKENS in include/moe_gb300.h


def _p(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _outputs(T, kmax, dev):
    return (torch.full((T, kmax), 7, dtype=torch.int32, device=dev),
            torch.full((T, kmax), 7.0, dtype=torch.float32, device=dev),
            torch.zeros(1, dtype=torch.int32, device=dev),
            torch.zeros(1, dtype=torch.float32, device=dev))


def _call_noalloc(lib, x, w, bias, it, k_fixed, kmax, renorm, outs):
    T, H = x.shape
    E = w.shape[0]
    ids, tw, kd, me = outs
    return lib.moe_router_topk_noalloc(
        _p(x), _p(w), _p(bias), ctypes.c_float(it), T, H, E, k_fixed, kmax, ctypes.c_float(1.2),
        ctypes.c_float(2.5), int(renorm), _p(ids), _p(tw), _p(kd), _p(me),
        ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))


def _call_with_workspace(lib, x, w, bias, it, k_fixed, kmax, renorm, outs):
    T, H = x.shape
    E = w.shape[0]
    ids, tw, kd, me = outs
    wsb = int(lib.moe_router_workspace_size(T))
    ws = torch.empty(wsb, dtype=torch.uint8, device=x.device)
    return lib.moe_router_topk(
        _p(x), _p(w), _p(bias), ctypes.c_float(it), T, H, E, k_fixed, kmax, ctypes.c_float(1.2),
        ctypes.c_float(2.5), int(renorm), _p(ids), _p(tw), _p(kd), _p(me), _p(ws), wsb,
        ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))


CASES = [
    # name, T, H, E, k_fixed, kmax, renorm, bias, inverse temperature
    ("decode_token", 1, 4096, 64, 4, 4, True, False, 1.0),
    ("prefill_like", 700, 2048, 128, 8, 8, True, False, 1.0),
    ("adaptive", 300, 1024, 32, 0, 3, True, True, 1.7),
    ("adaptive_raw", 97, 512, 16, 0, 4, False, False, 0.4),
]


@pytest.mark.parametrize("case", CASES, ids=[c[0] for c in CASES])
def test_noalloc_matches_workspace_router_on_two_calls(cuda_lib, case):
    name, T, H, E, k_fixed, kmax, renorm, use_bias, it = case
    lib = cuda_lib.lib()
    dev = torch.device("cuda:0")
    w = torch.from_numpy(workloads.normal_f32(3, 1, (E, H), 0.05)).to(dev)
    bias = torch.from_numpy(workloads.normal_f32(3, 2, (E,), 0.5)).to(dev) if use_bias else None
    for call in range(2):   # two calls in a row, different tokens, shared scratch
        x = torch.from_numpy(workloads.normal_bf16(3, 10 + call, (T, H), 1.0)).view(
            torch.bfloat16).to(dev)
        ref = _outputs(T, kmax, dev)
        got = _outputs(T, kmax, dev)
        assert _call_with_workspace(lib, x, w, bias, it, k_fixed, kmax, renorm, ref) == 0
        assert _call_noalloc(lib, x, w, bias, it, k_fixed, kmax, renorm, got) == 0
        torch.cuda.synchronize()
        assert torch.equal(got[0], ref[0]), f"{name} call {call}: ids differ"
        assert int(got[2].item()) == int(ref[2].item())
        assert np.allclose(got[1].cpu().numpy(), ref[1].cpu().numpy(), rtol=1e-6, atol=1e-7)
        assert abs(float(got[3].item()) - float(ref[3].item())) <= 1e-6


@pytest.mark.parametrize("case", [CASES[0], CASES[2]], ids=["decode_token", "adaptive"])
def test_noalloc_matches_oracle_on_two_calls(cuda_lib, case):
    """The allocation-free router against the oracle directly: ids and the
    batch's k exactly, weights and the mean entropy within the router's
    tolerances, on two calls in a row (the adaptive case also exercises the
    entropy and softmax sums that live in the shared scratch)."""
    name, T, H, E, k_fixed, kmax, renorm, use_bias, it = case
    lib = cuda_lib.lib()
    dev = torch.device("cuda:0")
    w_np = workloads.normal_f32(3, 1, (E, H), 0.05)
    b_np = workloads.normal_f32(3, 2, (E,), 0.5) if use_bias else None
    w = torch.from_numpy(w_np).to(dev)
    bias = torch.from_numpy(b_np).to(dev) if use_bias else None
    for call in range(2):
        x_bits = workloads.normal_bf16(3, 20 + call, (T, H), 1.0)
        x = torch.from_numpy(x_bits).view(torch.bfloat16).to(dev)
        got = _outputs(T, kmax, dev)
        assert _call_noalloc(lib, x, w, bias, it, k_fixed, kmax, renorm, got) == 0
        torch.cuda.synchronize()
        ref = oracle.route(x_bits, w_np, b_np, it, k_fixed, kmax, renorm)
        assert np.array_equal(got[0].cpu().numpy(), ref.ids), f"{name} call {call}: ids"
        assert int(got[2].item()) == ref.k
        assert np.allclose(got[1].cpu().numpy(), ref.weights, rtol=1e-6, atol=1e-7)
        assert abs(float(got[3].item()) - float(ref.mean_entropy)) <= 1e-4


def test_noalloc_rejects_batches_above_its_scratch(cuda_lib):
    lib = cuda_lib.lib()
    dev = torch.device("cuda:0")
    T, H, E = MAX_TOKENS + 1, 64, 8
    x = torch.zeros((T, H), dtype=torch.bfloat16, device=dev)
    w = torch.zeros((E, H), dtype=torch.float32, device=dev)
    outs = _outputs(T, 2, dev)
    assert _call_noalloc(lib, x, w, None, 1.0, 2, 2, True, outs) == 1   # MOE_ERR_INVALID_ARG
    torch.cuda.synchronize()
    assert int(outs[0][0, 0].item()) == 7   # nothing was launched
