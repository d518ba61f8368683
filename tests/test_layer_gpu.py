"""Quantized products and the whole layer on the GPU vs the CPU oracle."""
import os

import numpy as np
import pytest
import torch

import oracle
import workloads
from _parity import assert_layer_close, dev, rel_l2, to_np
from test_parity_gpu import CFG, SMALL

pytestmark = pytest.mark.gpu

PATHS = ["gemv", "tc"]


def path_id(moe, name):
    return {"gemv": moe.PATH_GEMV, "tc": moe.PATH_TC}[name]


def run_layer(moe, layer_np, x_bits, path, batch=0, **kw):
    layer = moe.MoELayer.from_workload(layer_np, dev(), batch=batch, path=path, **kw)
    out = layer(moe.bf16_from_bits(x_bits, dev()))
    torch.cuda.synchronize()
    return layer, to_np(out)


@pytest.mark.parametrize("path", PATHS)
@pytest.mark.parametrize("name", list(SMALL))
def test_layer_small_configs(cuda_lib, name, path):
    cfg = SMALL[name]
    layer_np = workloads.make_layer(cfg)
    for b in range(cfg.batches):
        x_bits = workloads.make_tokens(cfg, 0, b)
        ref = oracle.moe_forward(x_bits, layer_np, inv_temperature=cfg.inv_temperature(b))
        layer, out = run_layer(cuda_lib, layer_np, x_bits, path_id(cuda_lib, path), batch=b)
        bufs = layer.buffers(x_bits.shape[0])
        assert np.array_equal(to_np(bufs["topk_ids"]), ref.routing.ids)
        A = len(ref.perm.sorted_assign)
        h = to_np(bufs["h"])[:A]
        y = to_np(bufs["y"])[:A]
        # h is stored as bf16: its rounding (2^-9 relative, ~1.6e-3 rel L2)
        # dominates on the GEMV and small-batch tensor-core paths (exact
        # weights); the prefill tensor-core path also rounds the dequantized
        # weights to bf16 (~1.7e-3 per product)
        h_tol, y_tol = (5e-3, 6e-3) if path == "tc" else (4e-3, 4e-3)
        assert rel_l2(h, ref.h) <= h_tol, f"h {rel_l2(h, ref.h):.2e}"
        assert rel_l2(y, ref.y) <= y_tol, f"y {rel_l2(y, ref.y):.2e}"
        assert_layer_close(out, ref.out, f"{name} batch {b}")
        assert cuda_lib.moe_get_device_error() == 0


@pytest.mark.parametrize("path", PATHS)
@pytest.mark.parametrize("bits", [4, 8])
@pytest.mark.parametrize("T,k,E", [(1, 4, 16), (40, 2, 8)])
def test_fused_gate_up_bit_identical_to_two_products(cuda_lib, path, bits, T, k, E):
    cfg = CFG["tiny"].scaled(H=512, I=384, E=E, k=k, T=T, bits=bits)
    layer_np = workloads.make_layer(cfg)
    x_bits = workloads.make_tokens(cfg)
    d = dev()
    moe = cuda_lib
    p = path_id(moe, path)
    layer = moe.MoELayer.from_workload(layer_np, d, path=p)
    assert layer.fused
    x = moe.bf16_from_bits(x_bits, d)
    layer(x)
    b = layer.buffers(T)
    gu = layer.gate_up
    raw_f = moe.moe_gate_up_qmm(x, b["sorted"], b["offsets"], b["k_dev"], cfg.slots, gu.q, gu.s,
                                gu.b, bits, moe.EPILOGUE_RAW, path=p)
    raw_g = moe.moe_gate_up_qmm(x, b["sorted"], b["offsets"], b["k_dev"], cfg.slots, layer.gate.q,
                                layer.gate.s, layer.gate.b, bits, moe.EPILOGUE_RAW, path=p)
    raw_u = moe.moe_gate_up_qmm(x, b["sorted"], b["offsets"], b["k_dev"], cfg.slots, layer.up.q,
                                layer.up.s, layer.up.b, bits, moe.EPILOGUE_RAW, path=p)
    A = T * k
    I = cfg.I
    assert torch.equal(raw_f[:A, :I].view(torch.int32), raw_g[:A].view(torch.int32))
    assert torch.equal(raw_f[:A, I:].view(torch.int32), raw_u[:A].view(torch.int32))
    for dt in (torch.float32, torch.bfloat16):
        fused = moe.moe_gate_up_qmm(x, b["sorted"], b["offsets"], b["k_dev"], cfg.slots, gu.q,
                                    gu.s, gu.b, bits, moe.EPILOGUE_SWIGLU, out_dtype=dt, path=p)
        sep = moe.moe_swiglu(raw_g, raw_u, b["k_dev"], T, cfg.slots, out_dtype=dt)
        isz = torch.int32 if dt == torch.float32 else torch.int16
        assert torch.equal(fused[:A].view(isz), sep[:A].view(isz)), dt
    # and the RAW product itself matches the oracle
    ref = oracle.moe_forward(x_bits, layer_np)
    gq, gs, gb = oracle.pack_gate_up(layer_np.gate.q, layer_np.gate.s, layer_np.gate.b,
                                     layer_np.up.q, layer_np.up.s, layer_np.up.b)
    srt = ref.perm.sorted_assign
    xf = oracle.bf16_to_f64(x_bits)
    got = to_np(raw_f)[:A]
    for e in range(E):
        lo, hi = ref.perm.offsets[e], ref.perm.offsets[e + 1]
        if hi > lo:
            want = oracle.qmm_raw(xf[srt[lo:hi] // cfg.slots], gq[e], gs[e], gb[e], bits, cfg.H)
            # GEMV and small-batch tensor cores: exact (128 + q) x products
            # accumulated in fp32 by the tensor cores, then the 128 X offset
            # removed and the per-group affine applied in fp32 (the offset
            # cancellation scales the accumulation rounding by about
            # 128 / mean|q - 7.5|); prefill tensor cores: weights rounded to bf16
            tol = {"gemv": 1e-4, "tc": 3e-3}[path]
            assert rel_l2(got[lo:hi], want) <= tol


@pytest.mark.parametrize("T,k,E,H", [(1, 4, 16, 512), (37, 3, 8, 1024), (300, 8, 64, 256)])
def test_permute_rows_is_the_sorted_gather(cuda_lib, T, k, E, H):
    cfg = CFG["tiny"].scaled(H=H, I=256, E=E, k=k, T=T)
    layer_np = workloads.make_layer(cfg)
    x_bits = workloads.make_tokens(cfg)
    d = dev()
    layer = cuda_lib.MoELayer.from_workload(layer_np, d)
    x = cuda_lib.bf16_from_bits(x_bits, d)
    layer(x)
    b = layer.buffers(T)
    xs = cuda_lib.moe_permute_rows(x, b["sorted"], b["k_dev"], cfg.slots)
    torch.cuda.synchronize()
    ref = oracle.moe_forward(x_bits, layer_np)
    srt = ref.perm.sorted_assign
    assert np.array_equal(to_np(xs.view(torch.int16))[:len(srt)].view(np.uint16),
                          x_bits[srt // cfg.slots])
    assert cuda_lib.moe_get_device_error() == 0


@pytest.mark.parametrize("path", PATHS)
@pytest.mark.parametrize("bits", [4, 8])
def test_gate_up_presorted_rows_match_gathered_bitwise(cuda_lib, path, bits):
    """x read through sorted_assign and x pre-permuted into sorted rows give
    the same products bit for bit (a 300-token, ragged-segment case)."""
    cfg = CFG["tiny"].scaled(H=512, I=384, E=16, k=4, T=300, bits=bits)
    layer_np = workloads.make_layer(cfg)
    x_bits = workloads.make_tokens(cfg)
    d = dev()
    p = path_id(cuda_lib, path)
    layer = cuda_lib.MoELayer.from_workload(layer_np, d, path=p)
    x = cuda_lib.bf16_from_bits(x_bits, d)
    layer(x)
    b = layer.buffers(cfg.T)
    gu = layer.gate_up
    xs = cuda_lib.moe_permute_rows(x, b["sorted"], b["k_dev"], cfg.slots)
    A = cfg.T * cfg.k
    for epi, dt in ((cuda_lib.EPILOGUE_SWIGLU, torch.bfloat16), (cuda_lib.EPILOGUE_RAW, torch.float32)):
        g = cuda_lib.moe_gate_up_qmm(x, b["sorted"], b["offsets"], b["k_dev"], cfg.slots, gu.q,
                                     gu.s, gu.b, bits, epi, out_dtype=dt, path=p)
        r = cuda_lib.moe_gate_up_qmm(xs, None, b["offsets"], b["k_dev"], cfg.slots, gu.q, gu.s,
                                     gu.b, bits, epi, out_dtype=dt, path=p, T=cfg.T)
        isz = torch.int32 if dt == torch.float32 else torch.int16
        assert torch.equal(g[:A].view(isz), r[:A].view(isz)), (epi, dt)
    assert cuda_lib.moe_get_device_error() == 0


@pytest.mark.parametrize("path", PATHS)
def test_unfused_switch_matches_fused_bitwise(cuda_lib, path):
    cfg = SMALL["batched_s"]
    layer_np = workloads.make_layer(cfg)
    x_bits = workloads.make_tokens(cfg)
    p = path_id(cuda_lib, path)
    _, fused = run_layer(cuda_lib, layer_np, x_bits, p)
    old = os.environ.get("MOE_GB300_FUSE_GATE_UP")
    os.environ["MOE_GB300_FUSE_GATE_UP"] = "0"
    try:
        layer, unfused = run_layer(cuda_lib, layer_np, x_bits, p)
        assert not layer.fused
    finally:
        if old is None:
            del os.environ["MOE_GB300_FUSE_GATE_UP"]
        else:
            os.environ["MOE_GB300_FUSE_GATE_UP"] = old
    assert np.array_equal(fused, unfused)


@pytest.mark.parametrize("path", PATHS)
def test_repeated_runs_are_bitwise_identical(cuda_lib, path):
    cfg = SMALL["prefill_s"]
    layer_np = workloads.make_layer(cfg)
    x_bits = workloads.make_tokens(cfg)
    layer = cuda_lib.MoELayer.from_workload(layer_np, dev(), path=path_id(cuda_lib, path))
    x = cuda_lib.bf16_from_bits(x_bits, dev())
    outs = [layer(x).clone() for _ in range(3)]
    for o in outs[1:]:
        assert torch.equal(o.view(torch.int16), outs[0].view(torch.int16))


# ------------------------------------------------- full sizes, sampled tokens

FULL_SAMPLES = {"decode": None, "batched": None, "prefill": 48, "entropy": 24}


@pytest.fixture(scope="module")
def full_layers():
    cache = {}

    def get(name):
        if name not in cache:
            cache.clear()
            cache[name] = workloads.make_layer(CFG[name])
        return cache[name]
    return get


def check_rows(layer, T, ref, what):
    """h and y of the sampled tokens' assignments (the rows the oracle
    computed) against the oracle, at full size."""
    b = layer.buffers(T)
    rows = np.nonzero(~np.isnan(ref.h[:, 0]))[0]
    assert len(rows) > 0
    y_bf16 = b["y"].dtype == torch.bfloat16
    # bf16 h (2^-9 relative) dominates; the tensor-core path also rounds the
    # dequantized weights to bf16, and bf16 y adds one more rounding
    h_tol, y_tol = (5e-3, 6e-3) if y_bf16 else (4e-3, 4e-3)
    h = to_np(b["h"])[rows]
    y = to_np(b["y"])[rows]
    assert rel_l2(h, ref.h[rows]) <= h_tol, f"{what}: h {rel_l2(h, ref.h[rows]):.2e}"
    assert rel_l2(y, ref.y[rows]) <= y_tol, f"{what}: y {rel_l2(y, ref.y[rows]):.2e}"


@pytest.mark.parametrize("name", ["decode", "batched", "prefill", "entropy"])
def test_full_size_sampled(cuda_lib, full_layers, name):
    cfg = CFG[name]
    layer_np = full_layers(name)
    d = dev()
    rng = np.random.default_rng(7)
    for b in range(cfg.batches):
        x_all = workloads.make_tokens(cfg, 0, b)
        layer = cuda_lib.MoELayer.from_workload(layer_np, d, batch=b)
        if cfg.calls > 1:
            # batch-1 decode: each call routes one token; check three calls
            for c in (0, 100, 255):
                x_bits = x_all[c:c + 1]
                out = to_np(layer(cuda_lib.bf16_from_bits(x_bits, d)))
                ref = oracle.moe_forward(x_bits, layer_np)
                assert_layer_close(out, ref.out, f"decode call {c}")
                check_rows(layer, 1, ref, f"decode call {c}")
            continue
        out = to_np(layer(cuda_lib.bf16_from_bits(x_all, d)))
        n = FULL_SAMPLES[name]
        toks = np.arange(cfg.T) if n is None else np.sort(rng.choice(cfg.T, n, replace=False))
        ref = oracle.moe_forward(x_all, layer_np, inv_temperature=cfg.inv_temperature(b),
                                 tokens=toks)
        assert np.array_equal(to_np(layer.buffers(cfg.T)["topk_ids"]), ref.routing.ids)
        assert_layer_close(out[toks], ref.out[toks], f"{name} batch {b}")
        check_rows(layer, cfg.T, ref, f"{name} batch {b}")
        del layer
        torch.cuda.empty_cache()


@pytest.mark.parametrize("bits", [5, 6])
def test_full_size_batched_five_and_six_bits_sampled(cuda_lib, bits):
    """The batched-decode workload at full size with 5- and 6-bit codes (the
    shared-memory ring GEMV over 8-token chunks, the busiest experts in
    several chunks): the routing, and output, h and y of 8 sampled tokens
    against the oracle."""
    cfg = CFG["batched"].scaled(bits=bits)
    layer_np = workloads.make_layer(cfg)
    d = dev()
    x_all = workloads.make_tokens(cfg)
    layer = cuda_lib.MoELayer.from_workload(layer_np, d)
    out = to_np(layer(cuda_lib.bf16_from_bits(x_all, d)))
    toks = np.sort(np.random.default_rng(bits).choice(cfg.T, 8, replace=False))
    ref = oracle.moe_forward(x_all, layer_np, inv_temperature=cfg.inv_temperature(0), tokens=toks)
    assert np.array_equal(to_np(layer.buffers(cfg.T)["topk_ids"]), ref.routing.ids)
    assert_layer_close(out[toks], ref.out[toks], f"batched {bits}-bit")
    check_rows(layer, cfg.T, ref, f"batched {bits}-bit")
    assert cuda_lib.moe_get_device_error() == 0


def test_adaptive_k_queues_both_families_and_runs_the_one_for_k(cuda_lib):
    """Adaptive k with the automatic path: below ks tokens per expert the
    streamed GEMV, from ks the tensor cores, decided on the device.  Each
    batch's output equals, bit for bit, the layer forced to the family its k
    selects, and stays within tolerance of the oracle."""
    cfg = CFG["entropy"].scaled(H=1024, I=512, E=12, T=144, batches=3,
                                inv_temperatures=(12.0, 3.0, 0.5))
    layer_np = workloads.make_layer(cfg)
    auto = cuda_lib.MoELayer.from_workload(layer_np, dev())
    assert auto.k_split(cfg.T) == 2  # k = 1: 12 tokens per expert, k = 2: 24
    forced = {p: cuda_lib.MoELayer.from_workload(layer_np, dev(), path=p)
              for p in (cuda_lib.PATH_GEMV, cuda_lib.PATH_TC)}
    seen = set()
    for bt in range(cfg.batches):
        x_bits = workloads.make_tokens(cfg, 0, bt)
        x = cuda_lib.bf16_from_bits(x_bits, dev())
        it = cfg.inv_temperature(bt)
        got = auto(x, inv_temperature=it).clone()
        k = int(auto.buffers(cfg.T)["k_dev"].item())
        seen.add(k)
        fam = cuda_lib.PATH_GEMV if k < 2 else cuda_lib.PATH_TC
        want = forced[fam](x, inv_temperature=it)
        torch.cuda.synchronize()
        assert torch.equal(got.view(torch.int16), want.view(torch.int16)), f"batch {bt} (k={k})"
        ref = oracle.moe_forward(x_bits, layer_np, inv_temperature=it)
        assert ref.routing.k == k
        assert_layer_close(to_np(got), ref.out, f"batch {bt}")
    assert seen == {1, 2}, seen
    assert cuda_lib.moe_get_device_error() == 0


@pytest.mark.parametrize("path", ["gemv", "tc"])
def test_k_gated_products_run_only_inside_their_range(cuda_lib, path):
    """A gated product whose range holds the device's k equals the ungated
    one bit for bit; one whose range misses it leaves its output untouched."""
    cfg = CFG["tiny"]  # k = kmax = 2
    layer_np = workloads.make_layer(cfg)
    layer = cuda_lib.MoELayer.from_workload(layer_np, dev(), path=path_id(cuda_lib, path))
    x = cuda_lib.bf16_from_bits(workloads.make_tokens(cfg), dev())
    layer(x)
    b = layer.buffers(cfg.T)
    T, kmax, fam = cfg.T, layer.kmax, path_id(cuda_lib, path)
    g, d = layer.gate_up, layer.down
    xs, srt = (x, b["sorted"]) if path == "gemv" else (b["x_sorted"], None)

    def gate_up(flags):
        h = torch.full_like(b["h"], float("nan"))
        cuda_lib.moe_gate_up_qmm(xs, srt, b["offsets"], b["k_dev"], kmax, g.q, g.s, g.b, cfg.bits,
                                 cuda_lib.EPILOGUE_SWIGLU, h.dtype, h, fam | flags, T=T)
        return h

    def down(flags):
        y = torch.full_like(b["y"], float("nan"))
        cuda_lib.moe_down_qmm(b["h"], b["offsets"], b["k_dev"], T, kmax, d.q, d.s, d.b, cfg.bits,
                              y, fam | flags)
        return y

    A = T * kmax
    for run in (gate_up, down):
        ref = run(0)
        for lo, hi in ((1, 2), (2, 2)):
            got = run(cuda_lib.path_k_range(lo, hi))
            assert torch.equal(got[:A].view(torch.int32 if got.dtype == torch.float32
                                            else torch.int16),
                               ref[:A].view(torch.int32 if ref.dtype == torch.float32
                                            else torch.int16)), (run.__name__, lo, hi)
        skipped = run(cuda_lib.path_k_range(1, 1))
        torch.cuda.synchronize()
        assert torch.isnan(skipped.float()).all(), run.__name__
    assert cuda_lib.moe_get_device_error() == 0


def test_k_gate_arguments_are_checked(cuda_lib):
    cfg = CFG["tiny"]
    layer = cuda_lib.MoELayer.from_workload(workloads.make_layer(cfg), dev())
    x = cuda_lib.bf16_from_bits(workloads.make_tokens(cfg), dev())
    layer(x)
    b, d = layer.buffers(cfg.T), layer.down
    bad = [cuda_lib.PATH_GEMV | cuda_lib.path_k_range(0, 1),       # lo < 1
           cuda_lib.PATH_GEMV | cuda_lib.path_k_range(2, 1),       # hi < lo
           cuda_lib.PATH_TC | cuda_lib.path_k_range(1, 3),         # hi > kmax
           cuda_lib.PATH_AUTO | cuda_lib.path_k_range(1, 2),       # gate needs a family
           3 | cuda_lib.path_k_range(1, 2),                         # no such family
           3,
           cuda_lib.PATH_GEMV | (1 << 16)]                         # range without the flag
    for flags in bad:
        with pytest.raises(cuda_lib.MoEError):
            cuda_lib.moe_down_qmm(b["h"], b["offsets"], b["k_dev"], cfg.T, layer.kmax, d.q, d.s,
                                  d.b, cfg.bits, b["y"], flags)


@pytest.mark.parametrize("name,T", [("decode", 1), ("batched", 24)])
def test_three_chained_layers_in_one_graph_match_the_oracle(cuda_lib, name, T):
    """Three layers captured in one CUDA graph, layer l's bf16 output feeding
    layer l+1 (the launches of consecutive layers overlap): every layer's
    output matches the oracle applied to that layer's input.  (The oracle's
    own three-layer chain is no reference for the end result: the per-layer
    rounding differences compound and can move a routing near a tie.)"""
    cfg = CFG[name].scaled(H=1024, I=1536, E=16, T=T, calls=1)
    layer_np = workloads.make_layer(cfg)
    x_bits = workloads.make_tokens(cfg)[:T]
    d = dev()
    layer = cuda_lib.MoELayer.from_workload(layer_np, d)
    x0 = cuda_lib.bf16_from_bits(x_bits, d)
    outs = [torch.empty_like(x0) for _ in range(3)]

    def chain():
        inp = x0
        for o in outs:
            layer.forward(inp, out=o)
            inp = o

    chain()
    torch.cuda.synchronize()
    for o in outs:
        o.zero_()
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph, stream=s):
            chain()
    torch.cuda.current_stream().wait_stream(s)
    graph.replay()
    torch.cuda.synchronize()

    def bits(t):
        return t.view(torch.int16).cpu().numpy().view(np.uint16)

    inp = x_bits
    for li, o in enumerate(outs):
        got = to_np(o)
        ref = oracle.moe_forward(inp, layer_np)
        ids = to_np(layer.buffers(T)["topk_ids"]) if li == len(outs) - 1 else None
        if ids is not None:   # the buffers hold the last layer's routing
            assert np.array_equal(ids, ref.routing.ids)
        assert_layer_close(got, ref.out, f"{name} chained layer {li}")
        inp = bits(o)
    assert cuda_lib.moe_get_device_error() == 0


@pytest.mark.parametrize("bits", [5, 6])
@pytest.mark.parametrize("T,k,E,H,I", [(1, 4, 16, 1024, 768), (40, 2, 8, 512, 384),
                                       (37, 3, 12, 192, 320)])
def test_five_and_six_bit_layers_match_the_oracle(cuda_lib, bits, T, k, E, H, I):
    """5- and 6-bit codes (a row's little-endian bit stream) on the GEMV
    family: h, y and the layer output against the oracle, and the fused
    gate_up product equal to the two separate products bit for bit (raw and
    with the activation)."""
    cfg = CFG["tiny"].scaled(H=H, I=I, E=E, k=k, T=T, bits=bits)
    layer_np = workloads.make_layer(cfg)
    x_bits = workloads.make_tokens(cfg)
    d = dev()
    moe = cuda_lib
    layer = moe.MoELayer.from_workload(layer_np, d)
    assert layer.fused and layer.resolved_path(T) == moe.PATH_GEMV
    x = moe.bf16_from_bits(x_bits, d)
    out = to_np(layer(x))
    ref = oracle.moe_forward(x_bits, layer_np)
    b = layer.buffers(T)
    A = len(ref.perm.sorted_assign)
    assert np.array_equal(to_np(b["topk_ids"]), ref.routing.ids)
    assert rel_l2(to_np(b["h"])[:A], ref.h) <= 4e-3
    assert rel_l2(to_np(b["y"])[:A], ref.y) <= 4e-3
    assert_layer_close(out, ref.out, f"{bits}-bit layer T={T}")
    gu = layer.gate_up
    raw_f = moe.moe_gate_up_qmm(x, b["sorted"], b["offsets"], b["k_dev"], cfg.slots, gu.q, gu.s,
                                gu.b, bits, moe.EPILOGUE_RAW)
    raw_g = moe.moe_gate_up_qmm(x, b["sorted"], b["offsets"], b["k_dev"], cfg.slots, layer.gate.q,
                                layer.gate.s, layer.gate.b, bits, moe.EPILOGUE_RAW)
    raw_u = moe.moe_gate_up_qmm(x, b["sorted"], b["offsets"], b["k_dev"], cfg.slots, layer.up.q,
                                layer.up.s, layer.up.b, bits, moe.EPILOGUE_RAW)
    assert torch.equal(raw_f[:A, :I].view(torch.int32), raw_g[:A].view(torch.int32))
    assert torch.equal(raw_f[:A, I:].view(torch.int32), raw_u[:A].view(torch.int32))
    fused = moe.moe_gate_up_qmm(x, b["sorted"], b["offsets"], b["k_dev"], cfg.slots, gu.q, gu.s,
                                gu.b, bits, moe.EPILOGUE_SWIGLU, out_dtype=torch.bfloat16)
    sep = moe.moe_swiglu(raw_g, raw_u, b["k_dev"], T, cfg.slots, out_dtype=torch.bfloat16)
    assert torch.equal(fused[:A].view(torch.int16), sep[:A].view(torch.int16))
    # the tensor-core family does not take these widths
    with pytest.raises(moe.MoEError):
        moe.moe_gate_up_qmm(x, b["sorted"], b["offsets"], b["k_dev"], cfg.slots, gu.q, gu.s, gu.b,
                            bits, moe.EPILOGUE_RAW, path=moe.PATH_TC)
    assert moe.moe_get_device_error() == 0


@pytest.mark.parametrize("path,bits,H,I", [("gemv", 4, 512, 384), ("gemv", 8, 512, 384),
                                           ("tc", 4, 512, 384), ("tc", 8, 512, 384),
                                           ("gemv", 5, 512, 384), ("gemv", 4, 320, 192)])
def test_bf16_y_is_the_rounded_fp32_y(cuda_lib, path, bits, H, I):
    """The down product stored as bf16 is, bit for bit, the nearest-even
    rounding of the fp32 product (every kernel family: the streamed GEMV,
    the 5/6-bit GEMV, the plain GEMV for rows that are not whole 128-byte
    blocks, the tensor cores); combine reading the bf16 rows equals combine
    reading their exact fp32 values; and a layer storing y as bf16 stays
    within the layer tolerance of the oracle."""
    cfg = CFG["tiny"].scaled(H=H, I=I, E=16, k=4, T=300, bits=bits)
    layer_np = workloads.make_layer(cfg)
    x_bits = workloads.make_tokens(cfg)
    d = dev()
    p = path_id(cuda_lib, path)
    layer = cuda_lib.MoELayer.from_workload(layer_np, d, path=p, y_dtype=torch.bfloat16)
    x = cuda_lib.bf16_from_bits(x_bits, d)
    out = to_np(layer(x))
    b = layer.buffers(cfg.T)
    assert b["y"].dtype == torch.bfloat16
    dn, T, kmax, A = layer.down, cfg.T, cfg.slots, cfg.T * cfg.k
    y32 = cuda_lib.moe_down_qmm(b["h"], b["offsets"], b["k_dev"], T, kmax, dn.q, dn.s, dn.b, bits,
                                path=p, y_dtype=torch.float32)
    y16 = cuda_lib.moe_down_qmm(b["h"], b["offsets"], b["k_dev"], T, kmax, dn.q, dn.s, dn.b, bits,
                                path=p, y_dtype=torch.bfloat16)
    assert torch.equal(y16[:A].view(torch.int16), y32[:A].to(torch.bfloat16).view(torch.int16))
    assert torch.equal(y16[:A].view(torch.int16), b["y"][:A].view(torch.int16))
    o16 = cuda_lib.moe_combine(y16, b["inv_pos"], b["topk_w"], b["k_dev"], T, kmax)
    o32 = cuda_lib.moe_combine(y16.float(), b["inv_pos"], b["topk_w"], b["k_dev"], T, kmax)
    assert torch.equal(o16.view(torch.int16), o32.view(torch.int16))
    ref = oracle.moe_forward(x_bits, layer_np)
    assert_layer_close(out, ref.out, f"bf16 y, {path} {bits}-bit")
    assert cuda_lib.moe_get_device_error() == 0
