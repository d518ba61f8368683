"""GPU path vs the CPU oracle, element by element, through the C ABI."""
import numpy as np
import pytest
import torch

import oracle
import workloads
from _parity import assert_layer_close, dev, rel_l2, route_gpu, to_np

pytestmark = pytest.mark.gpu

CFG = workloads.CONFIGS


def shrunk(name, **kw):
    return CFG[name].scaled(**kw)


# Sizes the oracle finishes in seconds that still span several GEMV items and
# 128-row tensor tiles with a ragged tail (I, H not multiples of 128).
SMALL = {
    "tiny": CFG["tiny"],
    "decode_s": shrunk("decode", H=1088, I=1344, E=16, T=3, calls=1),
    "batched_s": shrunk("batched", H=1024, I=576, E=24, T=48),
    "prefill_s": shrunk("prefill", H=576, I=320, E=16, k=4, T=600),
    "entropy_s": shrunk("entropy", H=1024, I=448, E=12, T=96,
                        inv_temperatures=(12.0, 3.0, 0.5)),
}


# ------------------------------------------------------------------ router

@pytest.mark.parametrize("name", ["tiny", "decode", "batched", "prefill", "entropy"])
def test_router_full_size_bit_exact(cuda_lib, name):
    cfg = CFG[name]
    layer = workloads.make_layer(cfg)
    for b in range(cfg.batches):
        x_bits = workloads.make_tokens(cfg, 0, b)
        if cfg.calls > 1:
            x_bits = x_bits[:64]   # decode: routing of 64 single-token calls, batched as T=64
        it = cfg.inv_temperature(b)
        ref = oracle.route(x_bits, layer.router_w, layer.logit_bias, it, cfg.k, cfg.slots)
        _, ids, tw, kd, me = route_gpu(cuda_lib, x_bits, layer, cfg.k, cfg.slots, it)
        assert int(kd.item()) == ref.k
        assert np.array_equal(to_np(ids), ref.ids)
        w = to_np(tw)
        assert np.allclose(w, ref.weights, rtol=1e-6, atol=1e-7)
        assert abs(float(me.item()) - float(ref.mean_entropy)) < 1e-4
        if cfg.k == 0:
            assert ref.k == b + 1   # the three entropy batches hit k = 1, 2, 3


def test_router_single_token_calls(cuda_lib):
    cfg = CFG["decode"]
    rw = workloads.normal_f32(0, workloads.STREAM_ROUTER, (cfg.E, cfg.H), cfg.router_std)
    L = type("L", (), {"router_w": rw, "logit_bias": None})
    x_all = workloads.make_tokens(cfg)
    for c in (0, 1, 255):
        x_bits = x_all[c:c + 1]
        ref = oracle.route(x_bits, rw, None, 1.0, cfg.k, cfg.k)
        _, ids, tw, kd, me = route_gpu(cuda_lib, x_bits, L, cfg.k, cfg.k)
        assert np.array_equal(to_np(ids), ref.ids)
        assert np.allclose(to_np(tw), ref.weights, rtol=1e-6)


@pytest.mark.parametrize("E,k,kmax,T,renorm,bias,it", [
    (5, 2, 4, 7, True, False, 1.0),
    (37, 3, 3, 33, False, True, 0.7),
    (64, 1, 1, 17, True, True, 2.0),
    (130, 8, 16, 40, True, False, 1.3),
    (1024, 4, 4, 9, True, True, 1.0),
    (8, 0, 5, 21, True, False, 3.0),    # adaptive with kmax > 3
    (8, 0, 3, 21, False, True, 0.2),
    (37, 3, 3, 700, True, True, 0.9),   # 22 token groups: the 4-CTA cluster router
    # 8+ tokens per SM: one CTA per token group with every expert
    (37, 3, 3, 1300, True, True, 0.9),     # ragged experts and a 20-token last group
    (300, 2, 4, 1219, False, False, 1.1),  # 16-token groups, a last group of 3 tokens
    (5, 2, 2, 1240, True, False, 1.0),     # fewer experts than a warp tile
    (8, 0, 3, 1500, True, True, 1.4),      # adaptive k
])
def test_router_edge_shapes(cuda_lib, E, k, kmax, T, renorm, bias, it):
    rng = np.random.default_rng(E * 100 + T)
    H = 192
    rw = rng.normal(0, 0.05, (E, H)).astype(np.float32)
    if E > 6:
        rw[6] = rw[2]      # exact ties between experts 2 and 6
    lb = rng.normal(0, 0.5, E).astype(np.float32) if bias else None
    L = type("L", (), {"router_w": rw, "logit_bias": lb})
    x_bits = workloads.normal_bf16(1, 9, (T, H), 1.0)
    ref = oracle.route(x_bits, rw, lb, it, k, kmax, renorm)
    _, ids, tw, kd, me = route_gpu(cuda_lib, x_bits, L, k, kmax, it, renorm)
    assert int(kd.item()) == ref.k
    assert np.array_equal(to_np(ids), ref.ids)
    assert np.allclose(to_np(tw), ref.weights, rtol=1e-6, atol=1e-7)


def test_router_empty_batch(cuda_lib):
    rw = np.zeros((8, 64), np.float32)
    L = type("L", (), {"router_w": rw, "logit_bias": None})
    _, ids, tw, kd, me = route_gpu(cuda_lib, np.zeros((0, 64), np.uint16), L, 0, 3)
    assert int(kd.item()) == 1 and float(me.item()) == 0.0


@pytest.mark.parametrize("E,k,kmax,T,H", [
    (64, 4, 4, 1, 4096),      # single-token decode: staged weights, sort in the router
    (8, 0, 3, 21, 192),       # adaptive k, sorted after the batch's k is chosen
    (16, 16, 16, 32, 256),    # 512 slots: the largest batch sorted in the router
    (64, 4, 4, 33, 256),      # two token groups: router, then the permute kernel
    (300, 2, 2, 5, 128),      # E > 256: router, then the permute kernel
])
def test_route_is_router_then_permute(cuda_lib, E, k, kmax, T, H):
    """moe_route (router with the expert grouping fused in when one cluster
    covers the batch) gives the oracle's routing and grouping bit for bit."""
    rng = np.random.default_rng(E + T + H)
    rw = rng.normal(0, 0.05, (E, H)).astype(np.float32)
    x_bits = workloads.normal_bf16(3, 5, (T, H), 1.0)
    ref = oracle.route(x_bits, rw, None, 1.0, k, kmax, True)
    pref = oracle.permute(ref.ids, ref.k, E)
    d = dev()
    x = cuda_lib.bf16_from_bits(x_bits, d)
    w = torch.from_numpy(rw).to(d)
    ids = torch.empty((T, kmax), dtype=torch.int32, device=d)
    tw = torch.empty((T, kmax), dtype=torch.float32, device=d)
    kd = torch.empty(1, dtype=torch.int32, device=d)
    me = torch.empty(1, dtype=torch.float32, device=d)
    ws = torch.empty(cuda_lib.moe_router_workspace_size(T), dtype=torch.uint8, device=d)
    cnt = torch.empty(E, dtype=torch.int32, device=d)
    off = torch.empty(E + 1, dtype=torch.int32, device=d)
    srt = torch.full((T * kmax,), -7, dtype=torch.int32, device=d)
    inv = torch.empty(T * kmax, dtype=torch.int32, device=d)
    cuda_lib.moe_route(x, w, None, 1.0, k, kmax, 1.2, 2.5, True, ids, tw, kd, me, ws, cnt, off,
                       srt, inv)
    torch.cuda.synchronize()
    assert int(kd.item()) == ref.k
    assert np.array_equal(to_np(ids), ref.ids)
    assert np.allclose(to_np(tw), ref.weights, rtol=1e-6, atol=1e-7)
    assert np.array_equal(to_np(cnt), pref.counts)
    assert np.array_equal(to_np(off), pref.offsets)
    A = T * ref.k
    assert np.array_equal(to_np(srt)[:A], pref.sorted_assign)
    assert np.array_equal(to_np(inv), pref.inv_pos)
    assert cuda_lib.moe_get_device_error() == 0


# ----------------------------------------------------------------- permute

@pytest.mark.parametrize("T,kmax,k,E,skew", [(1, 4, 4, 64, False), (64, 4, 4, 64, True),
                                             (4096, 8, 8, 128, False), (512, 3, 2, 32, False),
                                             (300, 16, 16, 1024, False), (100, 3, 3, 4, True),
                                             (0, 2, 2, 8, False),
                                             # 32768 slots over 1024 experts; ranges of
                                             # several chunks per CTA (past 64 chunks)
                                             (2048, 16, 16, 1024, True),
                                             (9000, 8, 8, 128, False), (6000, 12, 11, 512, True)])
def test_permute_bit_exact(cuda_lib, T, kmax, k, E, skew):
    rng = np.random.default_rng(T + E)
    ids = np.full((T, kmax), -1, np.int32)
    for t in range(T):
        if skew:
            p = np.exp(-np.arange(E) * 0.5)
            ids[t, :k] = rng.choice(E, size=k, replace=False, p=p / p.sum())
        else:
            ids[t, :k] = rng.choice(E, size=k, replace=False)
    ref = oracle.permute(ids, k, E)
    d = dev()
    kd = torch.tensor([k], dtype=torch.int32, device=d)
    cnt, off, srt, inv = cuda_lib.moe_permute(torch.from_numpy(ids).to(d), kd, E)
    assert np.array_equal(to_np(cnt), ref.counts)
    assert np.array_equal(to_np(off), ref.offsets)
    A = T * k
    assert np.array_equal(to_np(srt)[:A], ref.sorted_assign)
    if T:
        assert np.array_equal(to_np(inv)[:T * kmax], ref.inv_pos)


def test_permute_flags_bad_expert(cuda_lib):
    d = dev()
    cuda_lib.moe_get_device_error(clear=True)
    ids = torch.tensor([[0, 9], [1, 2]], dtype=torch.int32, device=d)
    kd = torch.tensor([2], dtype=torch.int32, device=d)
    cuda_lib.moe_permute(ids, kd, 4)
    assert cuda_lib.moe_get_device_error(clear=True) & cuda_lib.DEVERR_BAD_EXPERT
    assert cuda_lib.moe_get_device_error(clear=True) == 0


def test_bounded_wait_reports_timeout_and_context_stays_usable(cuda_lib):
    """A device wait that runs out (an mbarrier nothing arrives on) sets the
    timeout bit in the error word; the next layer call still matches the
    oracle."""
    cuda_lib.moe_get_device_error(clear=True)
    cuda_lib.moe_selftest_wait_timeout(2_000_000)   # about a millisecond
    assert cuda_lib.moe_get_device_error(clear=True) & cuda_lib.DEVERR_TIMEOUT
    assert cuda_lib.moe_get_device_error(clear=True) == 0
    cfg = workloads.CONFIGS["tiny"]
    layer_np = workloads.make_layer(cfg)
    x_bits = workloads.make_tokens(cfg)
    layer = cuda_lib.MoELayer.from_workload(layer_np, dev())
    out = to_np(layer(cuda_lib.bf16_from_bits(x_bits, dev())))
    ref = oracle.moe_forward(x_bits, layer_np)
    assert rel_l2(out, ref.out) <= 5e-3
    assert cuda_lib.moe_get_device_error() == 0


@pytest.mark.parametrize("E,G,T,renorm,bias", [
    (64, 4, 1, True, False),      # the pages' 4 groups of 16 experts, one decode token
    (64, 4, 37, True, True),      # two token groups
    (48, 8, 700, False, True),    # 22 token groups (4-CTA cluster router), raw softmax weights
    (16, 16, 9, True, False),     # one expert per group: every expert, in logit order
])
def test_group_limited_routing_matches_oracle(cuda_lib, E, G, T, renorm, bias):
    """Group-limited routing (page A section 1.1): ids and grouping bit for
    bit, weights to fp32 rounding, against the oracle's per-group argmax."""
    rng = np.random.default_rng(E * 7 + T)
    H = 256
    rw = rng.normal(0, 0.05, (E, H)).astype(np.float32)
    rw[5] = rw[2]                 # an exact tie inside the first group
    lb = rng.normal(0, 0.5, E).astype(np.float32) if bias else None
    x_bits = workloads.normal_bf16(3, 11, (T, H), 1.0)
    ref = oracle.route(x_bits, rw, lb, 0.8, G, G, renorm, groups=G)
    perm = oracle.permute(ref.ids, G, E)
    d = dev()
    x = cuda_lib.bf16_from_bits(x_bits, d)
    w = torch.from_numpy(rw).to(d)
    b = None if lb is None else torch.from_numpy(lb).to(d)
    ids = torch.empty((T, G), dtype=torch.int32, device=d)
    tw = torch.empty((T, G), dtype=torch.float32, device=d)
    kd = torch.empty(1, dtype=torch.int32, device=d)
    me = torch.empty(1, dtype=torch.float32, device=d)
    ws = torch.empty(cuda_lib.moe_router_workspace_size(T), dtype=torch.uint8, device=d)
    cnt = torch.empty(E, dtype=torch.int32, device=d)
    off = torch.empty(E + 1, dtype=torch.int32, device=d)
    srt = torch.empty(T * G, dtype=torch.int32, device=d)
    inv = torch.empty(T * G, dtype=torch.int32, device=d)
    cuda_lib.moe_route_grouped(x, w, b, 0.8, G, G, renorm, ids, tw, kd, me, ws, cnt, off, srt, inv)
    torch.cuda.synchronize()
    assert int(kd.item()) == G
    assert np.array_equal(to_np(ids), ref.ids)
    assert np.allclose(to_np(tw), ref.weights, rtol=1e-6, atol=1e-7)
    assert np.array_equal(to_np(cnt), perm.counts)
    assert np.array_equal(to_np(off), perm.offsets)
    assert np.array_equal(to_np(srt), perm.sorted_assign)
    assert np.array_equal(to_np(inv), perm.inv_pos)
    assert cuda_lib.moe_get_device_error() == 0


def test_group_limited_layer_matches_oracle(cuda_lib):
    """A whole layer with group-limited routing (4 groups of 16 experts, one
    expert each) against the oracle's forward with the same routing rule."""
    cfg = workloads.CONFIGS["tiny"].scaled(E=16, k=4)
    layer_np = workloads.make_layer(cfg)
    x_bits = workloads.make_tokens(cfg)
    layer = cuda_lib.MoELayer.from_workload(layer_np, dev(), groups=4)
    out = to_np(layer(cuda_lib.bf16_from_bits(x_bits, dev())))
    ref_r = oracle.route(x_bits, layer_np.router_w, None, 1.0, 4, 4, True, groups=4)
    ids = to_np(layer.buffers(cfg.T)["topk_ids"])
    assert np.array_equal(ids, ref_r.ids)
    ref = oracle.moe_forward(x_bits, layer_np, routing=ref_r)
    assert_layer_close(out, ref.out, "group-limited tiny layer")
    assert cuda_lib.moe_get_device_error() == 0


@pytest.mark.parametrize("T,k,kmax,E,C", [
    (64, 4, 4, 64, 3),     # batched-decode-like: popular experts overflow
    (700, 2, 3, 16, 40),   # several CTAs of the grouping kernel
    (25000, 2, 3, 16, 3500),  # several chunks per CTA
    (33, 3, 3, 8, 0),      # capacity 0: everything dropped
    (20, 2, 2, 8, 1000),   # capacity above every count: plain grouping
])
def test_permute_capacity_matches_oracle(cuda_lib, T, k, kmax, E, C):
    """Expert capacity: kept assignments, counts, offsets and the dropped
    marks bit for bit against the oracle; sorted rows past the kept total
    hold assignment 0."""
    rng = np.random.default_rng(T * 13 + C)
    ids_np = np.full((T, kmax), -1, np.int32)
    for t in range(T):
        # skewed: low ids are popular
        ids_np[t, :k] = rng.choice(E, size=k, replace=False, p=np.arange(E, 0, -1) / (E * (E + 1) / 2))
    ref = oracle.permute(ids_np, k, E, capacity=C)
    d = dev()
    ids = torch.from_numpy(ids_np).to(d)
    kd = torch.tensor([k], dtype=torch.int32, device=d)
    cnt = torch.empty(E, dtype=torch.int32, device=d)
    off = torch.empty(E + 1, dtype=torch.int32, device=d)
    srt = torch.full((T * kmax,), 12345, dtype=torch.int32, device=d)
    inv = torch.empty(T * kmax, dtype=torch.int32, device=d)
    cuda_lib.moe_permute_capped(ids, kd, E, C, cnt, off, srt, inv)
    torch.cuda.synchronize()
    kept = int(ref.offsets[-1])
    assert np.array_equal(to_np(cnt), ref.counts)
    assert np.array_equal(to_np(off), ref.offsets)
    assert np.array_equal(to_np(srt)[:kept], ref.sorted_assign)
    assert np.all(to_np(srt)[kept:T * k] == 0)
    assert np.array_equal(to_np(inv), ref.inv_pos)
    assert cuda_lib.moe_get_device_error() == 0


@pytest.mark.parametrize("path", ["gemv", "tc"])
def test_layer_with_capacity_matches_oracle(cuda_lib, path):
    """A whole layer whose popular experts hit their capacity: dropped slots
    contribute nothing, against the oracle's forward with the same rule."""
    cfg = SMALL["batched_s"]
    layer_np = workloads.make_layer(cfg)
    x_bits = workloads.make_tokens(cfg)
    C = 6
    pid = cuda_lib.PATH_GEMV if path == "gemv" else cuda_lib.PATH_TC
    layer = cuda_lib.MoELayer.from_workload(layer_np, dev(), path=pid, capacity=C)
    out = to_np(layer(cuda_lib.bf16_from_bits(x_bits, dev())))
    ref = oracle.moe_forward(x_bits, layer_np, capacity=C)
    assert (ref.perm.inv_pos == oracle.DROPPED).sum() > 0   # the case drops something
    assert np.array_equal(to_np(layer.buffers(cfg.T)["inv_pos"]), ref.perm.inv_pos)
    assert_layer_close(out, ref.out, f"capacity {C} ({path})")
    assert cuda_lib.moe_get_device_error() == 0


def test_group_limited_layer_with_capacity_matches_oracle(cuda_lib):
    """Group-limited routing and an expert capacity together: the ids follow
    the per-group rule and the grouping keeps each expert's C lowest
    assignments, against the oracle's grouped routing with its capacity."""
    cfg = SMALL["batched_s"].scaled(E=24, k=4)
    layer_np = workloads.make_layer(cfg)
    x_bits = workloads.make_tokens(cfg)
    C = 5
    layer = cuda_lib.MoELayer.from_workload(layer_np, dev(), groups=4, capacity=C)
    out = to_np(layer(cuda_lib.bf16_from_bits(x_bits, dev())))
    ref_r = oracle.route(x_bits, layer_np.router_w, layer_np.logit_bias,
                         cfg.inv_temperature(0), 4, 4, True, groups=4)
    ref = oracle.moe_forward(x_bits, layer_np, routing=ref_r, capacity=C)
    b = layer.buffers(cfg.T)
    assert np.array_equal(to_np(b["topk_ids"]), ref_r.ids)
    assert (ref.perm.inv_pos == oracle.DROPPED).sum() > 0   # the case drops something
    assert np.array_equal(to_np(b["counts"]), ref.perm.counts)
    assert np.array_equal(to_np(b["inv_pos"]), ref.perm.inv_pos)
    assert_layer_close(out, ref.out, f"groups 4, capacity {C}")
    assert cuda_lib.moe_get_device_error() == 0


@pytest.mark.parametrize("E", [1, 7, 64, 1000, 1024])
def test_expert_health_kernels_match_oracle(cuda_lib, E):
    """Window accumulation is exact (int64); the least-activated expert is
    exact (ties to the lower id); mean and population std within 1e-12."""
    rng = np.random.default_rng(E)
    window = torch.zeros(E, dtype=torch.int64, device=dev())
    total = np.zeros(E, np.int64)
    for call in range(3):
        c = rng.integers(0, 50, E).astype(np.int32)
        c[rng.integers(0, E, max(1, E // 8))] = 0          # ties at the minimum
        if call == 2:
            c[: min(E, 4)] = 2**30                          # large counts: int64 window
        total += c
        cuda_lib.moe_expert_counts_accumulate(torch.from_numpy(c).to(dev()), window)
    least, mean_std = cuda_lib.moe_expert_health(window)
    torch.cuda.synchronize()
    assert np.array_equal(to_np(window), total)
    l_ref, m_ref, s_ref = oracle.expert_health(total)
    assert int(least.item()) == l_ref
    ms = mean_std.cpu().numpy()
    assert abs(ms[0] - m_ref) <= 1e-12 * max(1.0, abs(m_ref))
    assert abs(ms[1] - s_ref) <= 1e-12 * max(1.0, s_ref)


def test_expert_health_monitor_on_layer_counts(cuda_lib):
    """The monitor on a layer's own expert_counts: a closed window equals the
    oracle's health of the summed counts of the calls it saw."""
    cfg = SMALL["batched_s"]
    layer = cuda_lib.MoELayer.from_workload(workloads.make_layer(cfg), dev())
    t = [0.0]
    mon = cuda_lib.ExpertHealthMonitor(cfg.E, dev(), window_s=60.0, clock=lambda: t[0])
    x_all = workloads.make_tokens(cfg)
    total = np.zeros(cfg.E, np.int64)
    for i in range(3):
        x = cuda_lib.bf16_from_bits(np.roll(x_all, i, axis=0), dev())
        layer(x)
        counts = layer.buffers(cfg.T)["counts"]
        total += to_np(counts).astype(np.int64)
        t[0] = 20.0 * i
        mon.record(counts)
    h = mon.close_window()
    l_ref, m_ref, s_ref = oracle.expert_health(total)
    assert h.least_expert == l_ref and abs(h.mean - m_ref) < 1e-9 and abs(h.std - s_ref) < 1e-9
    assert total.sum() == 3 * cfg.T * cfg.k


def test_expert_health_rejects_bad_arguments(cuda_lib):
    w = torch.zeros(1025, dtype=torch.int64, device=dev())
    with pytest.raises(cuda_lib.MoEError):
        cuda_lib.moe_expert_health(w)
    with pytest.raises(ValueError):
        cuda_lib.moe_expert_counts_accumulate(torch.zeros(4, dtype=torch.int32, device=dev()),
                                              torch.zeros(5, dtype=torch.int64, device=dev()))
