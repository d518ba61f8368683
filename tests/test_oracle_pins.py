"""Pins of the CPU oracle against facts that do not come from the oracle:
closed forms, the page's printed thresholds, brute force, the quantizer's
error bound, one-hot probes and a dense all-experts evaluation."""
import json
import math
import os

import numpy as np
import pytest

import oracle
import workloads

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def bf16(v):
    """float -> bf16 bit pattern (values used here are exact in bf16)."""
    a = np.asarray(v, dtype=np.float32)
    return (a.view(np.uint32) >> 16).astype(np.uint16)


# ---------------------------------------------------------------- router ---

def test_router_one_hot_picks_weight_column():
    rng = np.random.default_rng(1)
    E, H = 5, 512
    w = rng.normal(0, 1, (E, H)).astype(np.float32)
    for h in (0, 7, 8, 255, 256, 511):
        x = np.zeros((1, H), np.float32)
        x[0, h] = 1.0
        got = oracle.router_logits(bf16(x), w, None, 1.0)
        assert np.array_equal(got[0], w[:, h]), h


def test_router_bias_then_temperature():
    E, H = 3, 64
    w = np.zeros((E, H), np.float32)
    w[:, 0] = [1.0, 2.0, -3.0]
    x = np.zeros((1, H), np.float32)
    x[0, 0] = 1.0
    bias = np.array([0.5, -1.0, 0.25], np.float32)
    got = oracle.router_logits(bf16(x), w, bias, 2.0)
    assert np.array_equal(got[0], np.array([3.0, 2.0, -5.5], np.float32))


def test_router_summation_order_is_the_fixed_one():
    # x = 1 everywhere.  W puts 2^24 on element 0 (chunk 0, partial sum 0),
    # -2^24 on element 8 (chunk 1, partial sum 1) and 1 on element 256
    # (chunk 32, partial sum 0 again).  Partial sum 0 = fl(2^24 + 1) = 2^24,
    # partial sum 1 = -2^24, so the fixed order yields exactly 0, whereas a
    # left-to-right sum would give 1.
    H = 512
    w = np.zeros((1, H), np.float32)
    w[0, 0], w[0, 8], w[0, 256] = 2.0 ** 24, -(2.0 ** 24), 1.0
    x = np.ones((1, H), np.float32)
    assert oracle.router_logits(bf16(x), w, None, 1.0)[0, 0] == 0.0
    # The pairwise combination ends with (sum of even partials) + (sum of
    # odd partials).  A 1 in partial sum 2 (element 16) joins 2^24 on the
    # even side first and is lost: result 0.  A 1 in partial sum 3 (element
    # 24) joins -2^24 on the odd side (-2^24 + 1 is exact): result 1.
    w2 = w.copy()
    w2[0, 256], w2[0, 16] = 0.0, 1.0
    assert oracle.router_logits(bf16(x), w2, None, 1.0)[0, 0] == 0.0
    w3 = w.copy()
    w3[0, 256], w3[0, 24] = 0.0, 1.0
    assert oracle.router_logits(bf16(x), w3, None, 1.0)[0, 0] == 1.0


def test_router_close_to_exact_dot_product():
    rng = np.random.default_rng(2)
    T, E, H = 7, 9, 1024
    x = bf16(rng.normal(0, 1, (T, H)).astype(np.float32))
    w = rng.normal(0, 0.05, (E, H)).astype(np.float32)
    got = oracle.router_logits(x, w, None, 1.0).astype(np.float64)
    xf = oracle.bf16_to_f64(x)
    exact = xf @ w.astype(np.float64).T
    bound = 2 * H * 2.0 ** -24 * (np.abs(xf) @ np.abs(w.astype(np.float64)).T)
    assert np.all(np.abs(got - exact) <= bound)


# --------------------------------------------------------------- entropy ---

def test_entropy_closed_forms():
    E = 32
    uni = np.zeros((1, E), np.float32)
    assert abs(oracle.softmax_entropy(uni)[0] - math.log(E)) < 1e-5
    rule = json.load(open(os.path.join(GOLDEN, "entropy_rule.json")))
    for case in rule["dominant_logit_cases"]["cases"]:
        l = np.full((1, E), -40.0, np.float32)
        l[0, :case["n"]] = 0.0
        h = oracle.softmax_entropy(l)[0]
        assert abs(h - case["entropy"]) < 2e-5, case
        assert oracle.entropy_k(h) == case["k"], case


def test_entropy_rule_boundaries_from_page():
    rule = json.load(open(os.path.join(GOLDEN, "entropy_rule.json")))
    assert tuple(rule["thresholds"]) == oracle.ENTROPY_THRESHOLDS
    for case in rule["boundary_cases"]:
        assert oracle.entropy_k(case["mean_entropy"]) == case["k"], case


def test_entropy_matches_float64_definition():
    rng = np.random.default_rng(3)
    l = rng.normal(0, 2, (50, 64)).astype(np.float32)
    p = np.exp(l.astype(np.float64) - l.max(1, keepdims=True))
    p /= p.sum(1, keepdims=True)
    ref = -(p * np.log(p)).sum(1)
    assert np.allclose(oracle.softmax_entropy(l), ref, atol=2e-5)
    assert abs(oracle.batch_mean_entropy(oracle.softmax_entropy(l)) - ref.mean()) < 2e-5


def test_entropy_workload_batches_sit_mid_band():
    cfg = workloads.CONFIGS["entropy"].scaled(T=64)
    gold = json.load(open(os.path.join(GOLDEN, "entropy_temperatures.json")))
    assert tuple(gold["inv_temperatures"]) == workloads.ENTROPY_INV_TEMPERATURES
    for b, target in enumerate(gold["targets"]):
        assert oracle.entropy_k(target) == b + 1
        assert abs(gold["mean_entropy"][b] - target) < 1e-3
        assert min(abs(target - t) for t in oracle.ENTROPY_THRESHOLDS) >= 0.5


# ------------------------------------------------------------------ top-k ---

def brute_topk(l, k):
    T, E = l.shape
    out = np.zeros((T, k), np.int64)
    for t in range(T):
        for e in range(E):
            rank = sum(1 for f in range(E) if l[t, f] > l[t, e] or (l[t, f] == l[t, e] and f < e))
            if rank < k:
                out[t, rank] = e
    return out


@pytest.mark.parametrize("k", [1, 2, 4, 8])
def test_topk_brute_force(k):
    rng = np.random.default_rng(k)
    l = rng.normal(0, 1, (40, 16)).astype(np.float32)
    l[::3, 5] = l[::3, 2]          # exact ties
    l[1::4, 7] = l[1::4, 0]
    l[2, :] = 0.0                  # all equal
    assert np.array_equal(oracle.topk_ids(l, k), brute_topk(l, k))


@pytest.mark.parametrize("groups", [1, 2, 4, 16])
def test_group_top1_brute_force(groups):
    """Page [A] section 1.1: best expert of each group of consecutive ids.
    Checked against a per-group scan written from the definition; groups=1
    is plain top-1 and groups=E is the full descending order."""
    rng = np.random.default_rng(40 + groups)
    E = 16
    l = rng.normal(0, 1, (30, E)).astype(np.float32)
    l[::4, 3] = l[::4, 1]          # ties inside the first group
    l[5, :] = 1.0                  # all equal
    got = oracle.group_top1_ids(l, groups)
    gsz = E // groups
    for t in range(l.shape[0]):
        winners = []
        for g in range(groups):
            best = g * gsz
            for e in range(g * gsz, (g + 1) * gsz):
                if l[t, e] > l[t, best]:
                    best = e
            winners.append(best)
        # order: larger logit first, equal logits lower id first
        for i in range(len(winners)):
            for j in range(len(winners) - 1 - i):
                a, b = winners[j], winners[j + 1]
                if l[t, b] > l[t, a] or (l[t, b] == l[t, a] and b < a):
                    winners[j], winners[j + 1] = b, a
        assert list(got[t]) == winners
    if groups == 1:
        assert np.array_equal(got, brute_topk(l, 1))
    if groups == E:
        assert np.array_equal(got, brute_topk(l, E))


def test_group_routing_weights_and_k():
    rng = np.random.default_rng(41)
    H, E, G = 128, 16, 4
    w = rng.normal(0, 0.05, (E, H)).astype(np.float32)
    x = bf16(rng.normal(0, 1, (12, H)).astype(np.float32))
    r = oracle.route(x, w, None, 1.0, k_fixed=G, groups=G)
    assert r.k == G
    gsz = E // G
    for t in range(12):
        assert sorted(int(e) // gsz for e in r.ids[t]) == list(range(G))  # one per group
    np.testing.assert_allclose(r.weights.sum(axis=1), 1.0, rtol=0, atol=1e-12)


def test_topk_ties_from_duplicated_router_rows():
    rng = np.random.default_rng(5)
    H, E = 256, 8
    w = rng.normal(0, 0.05, (E, H)).astype(np.float32)
    w[6] = w[1]
    x = bf16(rng.normal(0, 1, (30, H)).astype(np.float32))
    r = oracle.route(x, w, None, 1.0, k_fixed=E)
    pos = {int(e): j for j, e in enumerate(r.ids[0])}
    assert np.array_equal(r.logits[:, 1], r.logits[:, 6])
    for t in range(30):
        row = list(r.ids[t])
        assert row.index(1) < row.index(6)
    assert pos  # ids are a permutation of all experts
    assert sorted(r.ids[0]) == list(range(E))


def test_routing_weights_properties():
    rng = np.random.default_rng(6)
    l = rng.normal(0, 1.5, (64, 32)).astype(np.float32)
    for k in (1, 2, 3, 8):
        ids = oracle.topk_ids(l, k)
        w = oracle.routing_weights(l, ids, renormalize=True)
        assert np.allclose(w.sum(1), 1.0, atol=1e-12)
        assert np.all(np.diff(w, axis=1) <= 0)
        if k == 1:
            assert np.all(w == 1.0)
        raw = oracle.routing_weights(l, ids, renormalize=False)
        ls = l.astype(np.float64)
        soft = np.exp(ls - ls.max(1, keepdims=True))
        soft /= soft.sum(1, keepdims=True)
        assert np.allclose(raw, np.take_along_axis(soft, ids.astype(np.int64), 1), rtol=1e-12)


# ---------------------------------------------------------------- permute ---

@pytest.mark.parametrize("T,k,kmax,E", [(16, 2, 2, 8), (37, 3, 3, 5), (50, 1, 3, 64), (1, 4, 4, 64), (0, 2, 2, 4)])
def test_permute_brute_force(T, k, kmax, E):
    rng = np.random.default_rng(T + E)
    ids = np.full((T, kmax), -1, np.int32)
    for t in range(T):
        ids[t, :k] = rng.choice(E, size=k, replace=False)
    p = oracle.permute(ids, k, E)
    expect = []
    for e in range(E):
        expect += [t * kmax + j for t in range(T) for j in range(k) if ids[t, j] == e]
    assert list(p.sorted_assign) == expect
    assert int(p.counts.sum()) == T * k and p.offsets[-1] == T * k
    for e in range(E):
        seg = p.sorted_assign[p.offsets[e]:p.offsets[e + 1]]
        assert all(ids[a // kmax, a % kmax] == e for a in seg)
        assert np.all(np.diff(seg) > 0)
    for t in range(T):
        for j in range(kmax):
            a = t * kmax + j
            if j < k:
                assert p.sorted_assign[p.inv_pos[a]] == a
            else:
                assert p.inv_pos[a] == -1


@pytest.mark.parametrize("C", [0, 1, 3, 1000])
def test_permute_capacity_brute_force(C):
    """Expert capacity: each expert keeps its C lowest assignments a =
    t*kmax + j; the rest are marked dropped.  C at least the largest count
    is the plain permutation; C = 0 drops everything."""
    rng = np.random.default_rng(70 + C)
    T, k, kmax, E = 40, 3, 4, 6
    ids = np.full((T, kmax), -1, np.int32)
    for t in range(T):
        ids[t, :k] = rng.choice(E, size=k, replace=False)
    p = oracle.permute(ids, k, E, capacity=C)
    expect, dropped = [], set()
    for e in range(E):
        mine = [t * kmax + j for t in range(T) for j in range(k) if ids[t, j] == e]
        expect += mine[:C]
        dropped |= set(mine[C:])
    assert list(p.sorted_assign) == expect
    assert list(p.counts) == [min(C, int((ids[:, :k] == e).sum())) for e in range(E)]
    for t in range(T):
        for j in range(kmax):
            a = t * kmax + j
            if j >= k:
                assert p.inv_pos[a] == -1
            elif a in dropped:
                assert p.inv_pos[a] == oracle.DROPPED
            else:
                assert p.sorted_assign[p.inv_pos[a]] == a
    if C >= T:
        plain = oracle.permute(ids, k, E)
        assert np.array_equal(p.sorted_assign, plain.sorted_assign)
        assert np.array_equal(p.inv_pos, plain.inv_pos)


def test_capacity_zero_gives_zero_output_and_large_capacity_changes_nothing():
    cfg = workloads.CONFIGS["tiny"]
    layer = workloads.make_layer(cfg)
    x = workloads.make_tokens(cfg)
    plain = oracle.moe_forward(x, layer)
    assert np.array_equal(oracle.moe_forward(x, layer, capacity=cfg.T).out, plain.out)
    assert np.array_equal(oracle.moe_forward(x, layer, capacity=0).out, np.zeros_like(plain.out))
    # a capped layer equals the dense masked sum over the kept (token, expert) pairs only
    fw = oracle.moe_forward(x, layer, capacity=2)
    kept = oracle.Routing(fw.routing.logits, fw.routing.ids.copy(), fw.routing.weights.copy(),
                          fw.routing.k, fw.routing.mean_entropy, fw.routing.token_entropy)
    for t in range(cfg.T):
        for j in range(fw.routing.k):
            if fw.perm.inv_pos[t * cfg.slots + j] == oracle.DROPPED:
                kept.weights[t, j] = 0.0
    dense = oracle.dense_masked_forward(x, layer, kept)
    np.testing.assert_allclose(fw.out, dense, rtol=1e-9, atol=1e-12)


# ---------------------------------------------------------------- dequant ---

def test_dequant_extreme_codes():
    for bits in (4, 5, 6, 8):
        cols = 128
        words = cols * bits // 32
        s = np.array([[0.25, 0.0625]], np.float16)
        b = np.array([[-1.5, 0.75]], np.float16)
        zero = oracle.dequant(np.zeros((1, words), np.uint32), s, b, bits, cols)
        assert np.all(zero[0, :64] == -1.5) and np.all(zero[0, 64:] == 0.75)
        full = oracle.dequant(np.full((1, words), 0xFFFFFFFF, np.uint32), s, b, bits, cols)
        top = (1 << bits) - 1
        assert np.all(full[0, :64] == -1.5 + top * 0.25) and np.all(full[0, 64:] == 0.75 + top * 0.0625)


def test_unpack_order_single_code():
    # code 5 at element 13 of a 4-bit row: word 1, bits 20..23
    q = np.zeros((1, 4), np.uint32)
    q[0, 1] = np.uint32(5 << 20)
    codes = oracle.unpack_codes(q, 4, 32)
    assert codes[0, 13] == 5 and codes.sum() == 5
    q8 = np.zeros((1, 4), np.uint32)
    q8[0, 2] = np.uint32(200 << 8)          # element 9 of an 8-bit row
    codes8 = oracle.unpack_codes(q8, 8, 16)
    assert codes8[0, 9] == 200 and codes8.sum() == 200


@pytest.mark.parametrize("bits,elem,code,words", [
    # 5-bit element 6 spans bits 30..34: word 0 bits 30-31, word 1 bits 0-2
    (5, 6, 0b10111, {0: 0b11 << 30, 1: 0b101}),
    # 6-bit element 5 spans bits 30..35: word 0 bits 30-31, word 1 bits 0-3
    (6, 5, 0b101101, {0: 0b01 << 30, 1: 0b1011}),
    # 5-bit element 7 at bits 35..39, inside word 1
    (5, 7, 31, {1: 31 << 3}),
    # 6-bit element 10 at bits 60..65: low 4 bits in word 1 bits 28-31, high 2 in word 2
    (6, 10, 0b110011, {1: 0b0011 << 28, 2: 0b11}),
])
def test_unpack_bit_stream_codes(bits, elem, code, words):
    q = np.zeros((1, 2 * bits), np.uint32)       # one group of 64 codes
    for w, v in words.items():
        q[0, w] = np.uint32(v)
    codes = oracle.unpack_codes(q, bits, 64)
    assert codes[0, elem] == code and int(codes.sum()) == code


@pytest.mark.parametrize("bits", [4, 5, 6, 8])
def test_dequant_within_quantizer_bound(bits):
    qm, wf = workloads.quantized(0, 77, 2, 24, 256, bits, 0.02, return_float=True)
    for e in range(2):
        deq = oracle.dequant(qm.q[e], qm.s[e], qm.b[e], bits, 256)
        s = np.repeat(qm.s[e].astype(np.float64), 64, -1)
        slack = 2.0 ** -9 * np.repeat(np.maximum(np.abs(qm.b[e].astype(np.float64)),
                                                 np.abs(qm.s[e].astype(np.float64)) * ((1 << bits) - 1)), 64, -1)
        assert np.all(np.abs(deq - wf[e]) <= s / 2 + slack + 1e-12)


def test_one_hot_probe_reads_weight_column():
    qm, wf = workloads.quantized(0, 78, 1, 40, 192, 4, 0.02, return_float=True)
    deq = oracle.dequant(qm.q[0], qm.s[0], qm.b[0], 4, 192)
    for j in (0, 63, 64, 191):
        x = np.zeros((1, 192))
        x[0, j] = 1.0
        y = oracle.qmm_raw(x, qm.q[0], qm.s[0], qm.b[0], 4, 192)
        assert np.array_equal(y[0], deq[:, j])
        s = qm.s[0][:, j // 64].astype(np.float64)
        assert np.all(np.abs(y[0] - wf[0][:, j]) <= s / 2 + 1e-4)


# ----------------------------------------------------------------- fusion ---

def test_can_fuse_checks_every_field():
    base = oracle.QDesc(True, 4, 64, "affine", False, 512, 256, "float16")
    assert oracle.can_fuse(base, base)
    import dataclasses
    for field, val in [("quantized", False), ("bits", 8), ("group", 32), ("mode", "mxfp4"),
                       ("has_bias", True), ("rows", 256), ("cols", 512), ("scale_dtype", "bfloat16")]:
        assert not oracle.can_fuse(base, dataclasses.replace(base, **{field: val})), field


@pytest.mark.parametrize("bits", [4, 8])
def test_fused_equals_two_matmuls_bitwise(bits):
    # x in {-2,-1,-0.5,0,0.5,1,2}: every product and every partial sum is exact
    # in float64, so the comparison is independent of summation order.
    rng = np.random.default_rng(bits)
    H, I, E = 256, 96, 3
    g = workloads.quantized(0, 90, E, I, H, bits, 0.02)
    u = workloads.quantized(0, 91, E, I, H, bits, 0.02)
    x = rng.choice([-2.0, -1.0, -0.5, 0.0, 0.5, 1.0, 2.0], size=(9, H))
    fq, fs, fb = oracle.pack_gate_up(g.q, g.s, g.b, u.q, u.s, u.b)
    assert fq.shape == (E, 2 * I, H * bits // 32)
    for e in range(E):
        fused = oracle.qmm_raw(x, fq[e], fs[e], fb[e], bits, H)
        assert np.array_equal(fused[:, :I], oracle.qmm_raw(x, g.q[e], g.s[e], g.b[e], bits, H))
        assert np.array_equal(fused[:, I:], oracle.qmm_raw(x, u.q[e], u.s[e], u.b[e], bits, H))


def test_silu_closed_forms():
    assert oracle.silu(np.array([0.0]))[0] == 0.0
    assert abs(oracle.silu(np.array([50.0]))[0] - 50.0) < 1e-15 * 50
    assert abs(oracle.silu(np.array([-50.0]))[0]) < 1e-19
    z = np.linspace(-8, 8, 33)
    assert np.allclose(oracle.silu(z), z * 0.5 * (1 + np.tanh(z / 2)), rtol=1e-11, atol=1e-300)


# ------------------------------------------------------------ whole layer ---

@pytest.mark.parametrize("name,over", [
    ("tiny", {}),
    ("tiny", {"H": 128, "I": 64, "E": 3, "k": 2, "T": 5}),
    ("entropy", {"H": 128, "I": 128, "E": 6, "T": 24, "inv_temperatures": (4.0, 1.5, 0.4)}),
    ("batched", {"H": 192, "I": 64, "E": 10, "k": 3, "T": 12}),
    ("tiny", {"H": 128, "I": 192, "E": 4, "k": 2, "T": 6, "bits": 5}),
    ("tiny", {"H": 192, "I": 128, "E": 4, "k": 2, "T": 6, "bits": 6}),
])
def test_sparse_matches_dense_masked(name, over):
    cfg = workloads.CONFIGS[name].scaled(**over)
    layer = workloads.make_layer(cfg)
    for b in range(cfg.batches):
        x = workloads.make_tokens(cfg, 0, b)
        f = oracle.moe_forward(x, layer, inv_temperature=cfg.inv_temperature(b))
        d = oracle.dense_masked_forward(x, layer, f.routing)
        assert np.allclose(f.out, d, rtol=1e-12, atol=1e-14 * np.abs(d).max())


def test_constant_weights_closed_form():
    # Every code of expert e equals c_e, scales are s, biases 0.  Then each
    # gate and up output of a token is g = s*c_e*sum(x), h = silu(g)*g for all
    # n, each down output is s*c_e*I*h, and the layer returns
    # sum_j w_j * s*c_j*I*silu(s*c_j*X)*(s*c_j*X) with X = sum(x).
    cfg = workloads.CONFIGS["tiny"].scaled(H=128, I=64, E=4, k=2, T=6)
    layer = workloads.make_layer(cfg)
    s = 2.0 ** -6
    for m in (layer.gate, layer.up, layer.down):
        for e in range(cfg.E):
            c = e + 1
            word = 0
            for i in range(8):
                word |= c << (4 * i)
            m.q[e] = np.uint32(word)
            m.s[e] = np.float16(s)
            m.b[e] = np.float16(0.0)
    x = workloads.make_tokens(cfg)
    f = oracle.moe_forward(x, layer)
    X = oracle.bf16_to_f64(x).sum(1)
    for t in range(cfg.T):
        expect = 0.0
        for j in range(cfg.k):
            c = f.routing.ids[t, j] + 1
            g = s * c * X[t]
            expect += f.routing.weights[t, j] * s * c * cfg.I * (g / (1 + math.exp(-g))) * g
        assert np.allclose(f.out[t], expect, rtol=1e-12)


def test_generator_is_deterministic_and_sliceable():
    a = workloads.quantized(3, 2, 4, 16, 128, 4, 0.02)
    b = workloads.quantized(3, 2, 4, 16, 128, 4, 0.02, experts=[2])
    assert np.array_equal(a.q[2], b.q[0]) and np.array_equal(a.s[2], b.s[0])
    x1 = workloads.normal_bf16(0, 5, (4, 64), 1.0)
    x2 = workloads.normal_bf16(0, 5, (2, 64), 1.0, start=128)
    assert np.array_equal(x1[2:], x2)


# --------------------------------------------------------------------------
# Expert health (page [B] section 6): closed forms of the least-activated
# expert, the mean and the population standard deviation.
# --------------------------------------------------------------------------
@pytest.mark.parametrize("E", [1, 2, 7, 64, 1024])
def test_expert_health_equal_counts(E):
    least, mean, std = oracle.expert_health(np.full(E, 37, np.int64))
    assert (least, mean, std) == (0, 37.0, 0.0)


@pytest.mark.parametrize("E,hot", [(8, 0), (8, 5), (64, 63), (1024, 300)])
def test_expert_health_single_busy_expert(E, hot):
    # one expert takes all n activations: std = n sqrt(E - 1) / E
    n = 1000
    c = np.zeros(E, np.int64)
    c[hot] = n
    least, mean, std = oracle.expert_health(c)
    assert least == (1 if hot == 0 else 0)
    assert mean == n / E
    assert math.isclose(std, n * math.sqrt(E - 1) / E, rel_tol=1e-14)


@pytest.mark.parametrize("E", [2, 5, 64, 1000])
def test_expert_health_permuted_ramp(E):
    # counts 0 .. E-1 in any order: variance (E^2 - 1) / 12, least = where the 0 is
    rng = np.random.default_rng(E)
    c = rng.permutation(np.arange(E, dtype=np.int64))
    least, mean, std = oracle.expert_health(c)
    assert least == int(np.where(c == 0)[0][0])
    assert mean == (E - 1) / 2
    assert math.isclose(std, math.sqrt((E * E - 1) / 12.0), rel_tol=1e-13)


def test_expert_health_two_levels_and_ties():
    # half the experts at a, half at b: std = |a - b| / 2; the lowest id of
    # the lower level is the least-activated expert
    c = np.array([9, 4, 9, 4, 9, 4, 9, 4], np.int64)
    least, mean, std = oracle.expert_health(c)
    assert (least, mean, std) == (1, 6.5, 2.5)
    # the page's alert level: 20 activations of spread
    c = np.array([0, 40] * 32, np.int64)
    assert oracle.expert_health(c)[2] == 20.0


def test_f64_to_bf16_bits_rounds_to_nearest_even():
    """bf16 keeps 8 significant bits.  Halfway cases go to the even
    neighbour: 1 + 2^-8 lies between 1 (even) and 1 + 2^-7 and goes to 1;
    1 + 3 2^-8 lies between 1 + 2^-7 and 1 + 2^-6 (even) and goes up; just
    above a halfway point rounds up; any other value lands within half a
    unit in the last place."""
    cases = [(1.0, 1.0), (1.0 + 2.0 ** -8, 1.0), (1.0 + 3 * 2.0 ** -8, 1.0 + 2.0 ** -6),
             (1.0 + 2.0 ** -8 + 2.0 ** -20, 1.0 + 2.0 ** -7), (-2.5, -2.5), (0.0, 0.0),
             (3.0e38, 2.0 ** 127 * (1 + 98 / 128))]
    for v, want in cases:
        got = oracle.bf16_to_f64(oracle.f64_to_bf16_bits(np.array([v])))[0]
        assert got == want, (v, got, want)
    rng = np.random.default_rng(5)
    v = rng.normal(0, 3, 1000) * 10.0 ** rng.integers(-8, 8, 1000)
    got = oracle.bf16_to_f64(oracle.f64_to_bf16_bits(v))
    ulp = 2.0 ** (np.floor(np.log2(np.abs(v))) - 7)
    assert np.all(np.abs(got - v) <= ulp / 2 * (1 + 1e-9))
