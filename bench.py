"""Benchmark of the quantized sparse-MoE SwitchGLU layer forward on GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--config decode] [--impl reference]

Default workload (the headline): batch-1 decode, H 4096, I 11008, E 64,
top-4, 4-bit affine group 64, 256 single-token layer calls per step.  One
step = all 256 calls, each a full layer forward (router + top-k, permute,
fused gate_up + SiLU*up, down, combine), captured once in a CUDA graph and
replayed.  Metric: MoE-layer tokens/s over all ranks.  Inputs (4.9 GB of
expert weights, 304 MB active per call) are larger than L2.

Also reported: the dominant kernel's achieved HBM GB/s over its algorithmic
bytes (CUDA events around its launches), the end-to-end rate through the
public API with pinned host buffers, the SM clocks seen during the timed
region, and the CPU oracle on a bounded sample of the same workload.

N > 1 (torchrun): every rank runs its own 256 calls on its own tokens
against replicated weights -- independent replicas, weak scaling, no
collective on the data path.  --impl reference runs the CPU oracle as the
reference arm on rank 0 only.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402

import workloads  # noqa: E402

MEASURED_PEAKS = os.path.join(ROOT, "MEASURED_PEAKS.json")
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
TRAFFIC_FILE = os.path.join(ROOT, "profiles", "traffic.json")
CSRC = os.path.join(ROOT, "sparse_moe_expert_gb300", "csrc")
# the products' kernel and its source, by the path the layer resolved to
# (0 automatic, 1 streamed GEMV, 2 tcgen05 grouped GEMM)
KERNEL_NAME = {1: "gemv_stream_kernel", 2: "tc_qmm_kernel"}
KERNEL_SRC = {1: os.path.join(CSRC, "gemv_stream.cu"), 2: os.path.join(CSRC, "gemm_tc.cu")}


def parse_args(argv=None):
    p = argparse.ArgumentParser()
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=200)
    p.add_argument("--warmup", type=int, default=10)
    p.add_argument("--config", default="decode", choices=sorted(workloads.CONFIGS))
    p.add_argument("--impl", default="ours", choices=["ours", "reference"])
    p.add_argument("--no-cpu-baseline", action="store_true")
    p.add_argument("--cpu-sample", type=int, default=0, help="oracle sample size (calls/tokens)")
    p.add_argument("--path", default="auto", choices=["auto", "gemv", "tc"],
                   help="kernel family for the two quantized products")
    p.add_argument("--layers", type=int, default=1,
                   help="layers chained per call in the timed graph (each layer's output is "
                        "the next one's input; value counts layer-calls)")
    p.add_argument("--groups", type=int, default=0,
                   help="group-limited routing: best expert of each of G groups (k = G)")
    p.add_argument("--bits", type=int, default=0, choices=[0, 4, 5, 6, 8],
                   help="code width other than the workload's (5 or 6: the 5/6-bit GEMV)")
    p.add_argument("--experts", type=int, default=0,
                   help="smaller expert pool (same per-call work; for profiling captures)")
    p.add_argument("--y-dtype", default="auto", choices=["auto", "f32", "bf16"],
                   help="storage of the down product's rows before combine (auto: bf16 on the "
                        "tensor-core path)")
    p.add_argument("--no-configs", action="store_true",
                   help="skip the other workloads and the decode launch variants")
    return p.parse_args(argv)


def dist_env():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


def shard_calls(n_calls: int, rank: int, world: int):
    """Token stream offsets of this rank's calls: every rank runs n_calls
    independent calls on its own tokens (weak scaling)."""
    return [(rank * n_calls + c) for c in range(n_calls)]


def rank_tokens(cfg, rank: int, world: int) -> np.ndarray:
    """This rank's activations, bf16 bits [batches * calls * T, H]: batch b
    draws from stream STREAM_X + b at the offset of the rank's first call, so
    the ranks' tokens are disjoint pieces of one global stream."""
    starts = shard_calls(cfg.calls, rank, world)
    xb = [workloads.normal_bf16(0, workloads.STREAM_X + b, (cfg.calls * cfg.T, cfg.H), cfg.x_std,
                                start=starts[0] * cfg.T * cfg.H) for b in range(cfg.batches)]
    return np.concatenate(xb, axis=0)


def max_over_ranks(value: float, world: int, device=None) -> float:
    """The largest value over the ranks (the slowest rank's time)."""
    if world == 1:
        return value
    import torch
    import torch.distributed as dist
    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def load_peaks():
    try:
        with open(MEASURED_PEAKS) as f:
            return json.load(f), "measured"
    except (OSError, ValueError):
        return dict(FALLBACK_PEAKS), "fallback"


def file_sha(path):
    with open(path, "rb") as f:
        return hashlib.sha256(f.read()).hexdigest()[:16]


def active_bytes_per_expert(cfg, which):
    """Packed codes + fp16 scale + fp16 bias of one expert's matrix."""
    if which == "gate_up":
        rows, cols = 2 * cfg.I, cfg.H
    else:
        rows, cols = cfg.H, cfg.I
    return rows * (cols * cfg.bits // 8 + (cols // 64) * 4)


# ------------------------------------------------------------------ clocks

class ClockSampler:
    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_id: str):
        self.gpu_id = gpu_id
        self.proc = None
        self.tmp = None

    def __enter__(self):
        self.tmp = tempfile.NamedTemporaryFile("w+", suffix=".csv", delete=False)
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", self.gpu_id, f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=self.tmp, stderr=subprocess.DEVNULL)
        except OSError:
            self.proc = None
        time.sleep(0.3)
        return self

    def __exit__(self, *a):
        if self.proc is not None:
            time.sleep(0.25)
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
        self.tmp.close()

    def summary(self):
        rows = []
        try:
            with open(self.tmp.name) as f:
                for line in f:
                    parts = [x.strip() for x in line.split(",")]
                    if len(parts) >= 8 and parts[0].replace(".", "").isdigit():
                        rows.append(parts)
        finally:
            os.unlink(self.tmp.name)
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unavailable"], "samples": 0}
        sm = [float(r[0]) for r in rows]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if r[4 + i] == "Active"})
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": float(rows[0][1]),
                "reasons": reasons, "samples": len(rows),
                "power_w_max": max(float(r[2]) for r in rows if r[2].replace(".", "").isdigit())
                if any(r[2].replace(".", "").isdigit() for r in rows) else None}


# ------------------------------------------------------------- cpu oracle

def oracle_sample(cfg, layer_np, x_bits, n, batch=0):
    """Time the oracle (as it stands) on n tokens/calls of the workload."""
    import oracle
    t0, c0 = time.perf_counter(), time.process_time()
    if cfg.calls > 1:
        for c in range(n):
            oracle.moe_forward(x_bits[c:c + 1], layer_np, keep_intermediates=False)
        tokens = n
    else:
        toks = np.arange(n)
        oracle.moe_forward(x_bits, layer_np, inv_temperature=cfg.inv_temperature(batch),
                           tokens=toks, keep_intermediates=False)
        tokens = n
    wall = time.perf_counter() - t0
    cpu = time.process_time() - c0
    return tokens, wall, cpu


CPU_SAMPLE_SECONDS = 10.0


def default_sample(cfg):
    return {"decode": 2, "batched": 16, "prefill": 64, "entropy": 32, "tiny": 16}.get(cfg.name, 8)


def run_reference(args):
    rank, world, _ = dist_env()
    if rank != 0:
        return 0
    cfg = workloads.CONFIGS[args.config]
    layer_np = workloads.make_layer(cfg)
    x_bits = workloads.make_tokens(cfg)
    n = args.cpu_sample or (1 if cfg.calls > 1 else min(cfg.T, default_sample(cfg)))
    for _ in range(args.warmup):
        oracle_sample(cfg, layer_np, x_bits, n)
    tok = wall = cpu = 0.0
    for _ in range(args.steps):
        t, w, c = oracle_sample(cfg, layer_np, x_bits, n)
        tok += t
        wall += w
        cpu += c
    value = tok / wall
    cores = round(cpu / wall, 1) if wall > 0 else 1.0
    line = {
        "impl": "reference", "metric": metric_name(), "value": value, "unit": "tokens/s",
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": 1000.0 * wall / args.steps, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": workload_config(cfg),
        "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": cores, "kind": "oracle",
                         "sample": f"{n} {'calls' if cfg.calls > 1 else 'tokens'} per step"},
        "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


def metric_name():
    return "MoE-layer tokens/s; achieved HBM GB/s (decode) / tensor TFLOPS (prefill)"


def workload_config(cfg):
    kdesc = f"top-{cfg.k}" if cfg.k else "k from batch entropy"
    extra = {"batched": ", Zipf(1.1) log-prior",
             "decode": f", {cfg.calls} calls x 1 token"}.get(cfg.name, "")
    toks = "" if cfg.name == "decode" else f" T{cfg.T}"
    desc = (f"{cfg.name}: H{cfg.H} I{cfg.I} E{cfg.E} {kdesc}{toks}, {cfg.bits}-bit affine g64"
            f"{extra}")
    return {"workload": desc, "H": cfg.H, "I": cfg.I, "E": cfg.E, "k": cfg.k or "adaptive",
            "tokens_per_call": cfg.T, "calls_per_step": cfg.calls, "bits": cfg.bits,
            "l2": "inputs larger than L2 (expert weights stream from HBM every call)"}


# ----------------------------------------------------------------- ours

def workload_measure(moe, cfg, dev, rank, world, steps, warmup, layer_kw, nl=1, clocks_gpu=None,
                     per_kernel=True, layer_np=None):
    """One workload on this GPU: every layer call of a step (256 single-token
    calls for batch-1 decode, one call per activation batch otherwise)
    captured once in a CUDA graph and replayed `steps` times after `warmup`
    replays; then the same calls launched eagerly with CUDA events around
    each kernel (launch overlap off) for per-kernel durations, and the
    algorithmic bytes and FLOPs of the active experts.  Returns the layer,
    its inputs and a dict of results."""
    import torch
    if layer_np is None:
        layer_np = workloads.make_layer(cfg)
    layer = moe.MoELayer.from_workload(layer_np, dev, **layer_kw)
    T = cfg.T
    calls = cfg.calls * cfg.batches
    x_bits = rank_tokens(cfg, rank, world)
    x_dev = moe.bf16_from_bits(x_bits, dev)
    out_dev = torch.empty((calls * T, cfg.H), dtype=torch.bfloat16, device=dev)
    temps = [cfg.inv_temperature(c // cfg.calls) for c in range(calls)]
    chain = [torch.empty((T, cfg.H), dtype=torch.bfloat16, device=dev) for _ in range(2)]

    def step(events=None):
        for c in range(calls):
            if nl == 1 or events is not None:
                layer.forward(x_dev[c * T:(c + 1) * T], out=out_dev[c * T:(c + 1) * T],
                              inv_temperature=temps[c], events=events)
                continue
            # nl layers in a row: layer l reads layer l-1's output (the same
            # weights serve every layer; routing follows each layer's input)
            xin = x_dev[c * T:(c + 1) * T]
            for li in range(nl):
                dst = out_dev[c * T:(c + 1) * T] if li == nl - 1 else chain[li % 2]
                layer.forward(xin, out=dst, inv_temperature=temps[c])
                xin = dst

    # eager warm-up (sets kernel attributes), then capture one step in a graph
    step()
    torch.cuda.synchronize()
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        step()
    torch.cuda.current_stream().wait_stream(s)
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        step()
    torch.cuda.synchronize()
    for _ in range(max(3, warmup)):
        graph.replay()
    torch.cuda.synchronize()
    if world > 1:
        import torch.distributed as dist
        dist.barrier()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    clk = ClockSampler(clocks_gpu) if clocks_gpu else None
    if clk:
        clk.__enter__()
    e0.record()
    for _ in range(steps):
        graph.replay()
    e1.record()
    torch.cuda.synchronize()
    if clk:
        clk.__exit__()
    if world > 1:
        import torch.distributed as dist
        dist.barrier()
    ms = max_over_ranks(e0.elapsed_time(e1) / steps, world, dev)
    del graph
    res = {"ms": ms, "calls": calls, "T": T, "nl": nl,
           "clocks": clk.summary() if clk else None}
    # per-call active experts and k (one eager pass)
    per_call = []
    for c in range(calls):
        layer.forward(x_dev[c * T:(c + 1) * T], out=out_dev[c * T:(c + 1) * T],
                      inv_temperature=temps[c])
        bufs = layer.buffers(T)
        per_call.append((int((bufs["counts"] > 0).sum().item()), int(bufs["k_dev"].item())))
    res["per_call"] = per_call
    cnt = layer.buffers(T)["counts"].double().cpu()
    res["count_stats"] = {"experts": int(cnt.numel()), "active": int((cnt > 0).sum().item()),
                          "min": int(cnt.min().item()), "max": int(cnt.max().item()),
                          "std": round(float(cnt.std(unbiased=False).item()), 3)}
    # algorithmic bytes of the two products, summed over one step's calls:
    # the active experts' packed weights (codes + fp16 scale + fp16 bias)
    # plus the token rows read by gate_up; FLOPs 2 * rows * assignments * K
    res["gu_step_bytes"] = sum(active_bytes_per_expert(cfg, "gate_up") * na + T * cfg.H * 2
                               for na, _ in per_call)
    res["dn_step_bytes"] = sum(active_bytes_per_expert(cfg, "down") * na for na, _ in per_call)
    res["gu_step_flops"] = sum(2.0 * T * k * 2 * cfg.I * cfg.H for _, k in per_call)
    res["dn_step_flops"] = sum(2.0 * T * k * cfg.I * cfg.H for _, k in per_call)
    if per_kernel:
        ksteps = max(1, min(steps, 20))
        events = {}
        torch.cuda.synchronize()
        # each kernel on its own: no overlap with the kernel before it
        pdl_prev = moe.moe_set_launch_overlap(False)
        for _ in range(ksteps):
            step(events)
        torch.cuda.synchronize()
        moe.moe_set_launch_overlap(pdl_prev)
        res["ktot"] = {k: sum(a.elapsed_time(b) for a, b in v) / ksteps for k, v in events.items()}
        res["kavg"] = {k: sum(a.elapsed_time(b) for a, b in v) / len(v) for k, v in events.items()}
    return layer, layer_np, x_bits, temps, res


def recorded_traffic(name, kernel_src):
    """DRAM bytes (read + write) of one gate_up launch of workload `name`, from
    the ncu record in profiles/traffic.json taken with the kernel source as it
    is now (matched by its hash); None without such a record."""
    try:
        with open(TRAFFIC_FILE) as f:
            for rec in json.load(f).get("records", []):
                if rec.get("config") == name and rec.get("src") == os.path.basename(kernel_src) \
                        and rec.get("src_sha") == file_sha(kernel_src):
                    return rec.get("gate_up_dram_bytes_per_launch")
    except (OSError, ValueError):
        pass
    return None


def workload_summary(moe, cfg, layer, res, peaks, peak_src, name=None):
    """The measured numbers of one workload as the JSON fields of its line."""
    calls, T, nl, ms = res["calls"], res["T"], res["nl"], res["ms"]
    kt = res.get("ktot", {})
    gu_b, dn_b = res["gu_step_bytes"], res["dn_step_bytes"]
    gu_f, dn_f = res["gu_step_flops"], res["dn_step_flops"]
    path_used = layer.resolved_path(T)
    ks = layer.k_split(T)
    kname = "gemv_bits_kernel" if cfg.bits not in (4, 8) else KERNEL_NAME[path_used]
    kernel_label = kname + " (gate_up, SiLU*up epilogue)"
    if ks:
        kernel_label = (f"{KERNEL_NAME[moe.PATH_GEMV]} for k < {ks}, {KERNEL_NAME[moe.PATH_TC]} "
                        f"for k >= {ks} (gate_up, SiLU*up epilogue; both queued, gated on k)")
    gu_ms = kt.get("gate_up", 0.0)
    dn_ms = kt.get("down", 0.0)
    gu_gbs = gu_b / (gu_ms * 1e-3) / 1e9 if gu_ms else None
    dn_gbs = dn_b / (dn_ms * 1e-3) / 1e9 if dn_ms else None
    gu_tflops = gu_f / (gu_ms * 1e-3) / 1e12 if gu_ms else None
    dn_tflops = dn_f / (dn_ms * 1e-3) / 1e12 if dn_ms else None
    layer_gbs = (gu_b + dn_b) * nl / (ms * 1e-3) / 1e9
    layer_tflops = (gu_f + dn_f) * nl / (ms * 1e-3) / 1e12
    tensor_bound = path_used == moe.PATH_TC and cfg.name == "prefill"
    if tensor_bound:
        roof = {"bound": "tensor", "achieved": gu_tflops, "peak": peaks["bf16_tflops"],
                "unit": "TFLOP/s", "frac": gu_tflops / peaks["bf16_tflops"] if gu_tflops else None,
                "frac_of_sustained": (gu_tflops / peaks.get("bf16_tflops_sustained",
                                                            peaks["bf16_tflops"])
                                      if gu_tflops else None),
                "layer_frac": layer_tflops / peaks["bf16_tflops"],
                "kernel": kernel_label, "algorithmic_flops_per_launch": gu_f / calls,
                "peak_source": peak_src}
    else:
        roof = {"bound": "hbm", "achieved": gu_gbs, "peak": peaks["hbm_gbs"], "unit": "GB/s",
                "frac": gu_gbs / peaks["hbm_gbs"] if gu_gbs else None,
                "layer_frac": layer_gbs / peaks["hbm_gbs"],
                "kernel": kernel_label, "algorithmic_bytes_per_launch": gu_b / calls,
                "peak_source": peak_src}
    src = os.path.join(CSRC, "gemv_bits.cu") if cfg.bits not in (4, 8) else KERNEL_SRC[path_used]
    roof["traffic"] = recorded_traffic(name or cfg.name, src)
    kern = {"gate_up_us": gu_ms * 1e3 / calls if gu_ms else None,
            "down_us": dn_ms * 1e3 / calls if dn_ms else None,
            "gate_up_gbs": gu_gbs, "down_gbs": dn_gbs,
            "gate_up_tflops": gu_tflops, "down_tflops": dn_tflops,
            "layer_us_per_call": ms * 1e3 / (calls * nl), "layer_gbs": layer_gbs,
            "layer_tflops": layer_tflops,
            "active_experts_and_k_per_call": sorted(set(res["per_call"])),
            "expert_counts_last_call": res["count_stats"],
            "per_kernel_us": {k: v * 1e3 for k, v in res.get("kavg", {}).items()}}
    return roof, kern


def oracle_one_thread(cfg_name, n):
    """The oracle sample timed in a fresh process with one BLAS/OpenMP thread."""
    env = dict(os.environ, OMP_NUM_THREADS="1", OPENBLAS_NUM_THREADS="1", MKL_NUM_THREADS="1")
    out = subprocess.run([sys.executable, os.path.abspath(__file__), "--impl", "reference",
                          "--config", cfg_name, "--steps", "1", "--warmup", "0",
                          "--cpu-sample", str(n)], capture_output=True, text=True, env=env,
                         cwd=ROOT, timeout=600)
    for line in out.stdout.splitlines():
        if line.startswith("{"):
            d = json.loads(line)
            return {"value": d["value"], "cores": d["cpu_baseline"]["cores"],
                    "sample": d["cpu_baseline"]["sample"]}
    return None


def run_ours(args):
    import torch
    import torch.distributed as dist

    import sparse_moe_expert_gb300 as moe

    rank, world, local = dist_env()
    if world > 1:
        dist.init_process_group("nccl")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    cfg = workloads.CONFIGS[args.config]
    if args.experts:
        cfg = cfg.scaled(E=args.experts)
    if args.bits:
        cfg = cfg.scaled(bits=args.bits)
    path = {"auto": moe.PATH_AUTO, "gemv": moe.PATH_GEMV, "tc": moe.PATH_TC}[args.path]
    y_dtype = {"auto": None, "f32": torch.float32, "bf16": torch.bfloat16}[args.y_dtype]
    gpu_id = getattr(torch.cuda.get_device_properties(dev), "uuid", None)
    gpu_id = str(gpu_id) if gpu_id is not None else str(local)
    if gpu_id and not gpu_id.startswith("GPU-") and "-" in gpu_id:
        gpu_id = "GPU-" + gpu_id
    nl = max(1, args.layers)
    peaks, peak_src = load_peaks()

    layer, layer_np, x_bits, temps, res = workload_measure(
        moe, cfg, dev, rank, world, args.steps, args.warmup,
        dict(free_sources=True, path=path, groups=args.groups, y_dtype=y_dtype), nl=nl,
        clocks_gpu=gpu_id)
    T, calls, ms = res["T"], res["calls"], res["ms"]
    tokens_per_step = calls * T
    value = tokens_per_step * nl * world / (ms / 1000.0)  # layer-calls: tokens x layers
    clocks = res["clocks"]
    roof, kern = workload_summary(moe, cfg, layer, res, peaks, peak_src)

    # end to end through the public API with pinned host buffers
    x_host = torch.from_numpy(x_bits).view(torch.bfloat16).pin_memory()
    o_host = torch.empty((calls * T, cfg.H), dtype=torch.bfloat16).pin_memory()
    esteps = max(1, min(args.steps, 20))

    def e2e_step():
        for c in range(calls):
            layer.forward_host(x_host[c * T:(c + 1) * T], o_host[c * T:(c + 1) * T],
                               inv_temperature=temps[c])
    e2e_step()
    torch.cuda.synchronize()
    if world > 1:
        dist.barrier()
    t0 = time.perf_counter()
    for _ in range(esteps):
        e2e_step()
    torch.cuda.synchronize()
    e2e_s = (time.perf_counter() - t0) / esteps
    e2e_s = max_over_ranks(e2e_s, world, dev)
    e2e = {"value": tokens_per_step * world / e2e_s, "unit": "tokens/s",
           "h2d_bytes_per_step": tokens_per_step * cfg.H * 2,
           "d2h_bytes_per_step": tokens_per_step * cfg.H * 2,
           "how": "MoELayer.forward_host per call, eager launches, pinned host buffers"}

    line = {
        "metric": metric_name(), "value": value, "unit": "tokens/s", "n_gpus": world,
        "steps": args.steps, "warmup": max(3, args.warmup), "ms_per_step": ms,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": f"u{cfg.bits} affine weights x bf16 tokens, f32 accumulate",
        "data": "synthetic", "config": dict(workload_config(cfg), layers=nl, groups=args.groups,
                                            y_storage=str(layer.y_storage(T)).replace("torch.", "")),
        "roofline": roof, "kernels": kern,
        "clocks": {"sm_mhz": clocks["sm_mhz"], "sm_max_mhz": clocks["sm_max_mhz"],
                   "reasons": clocks["reasons"], "samples": clocks["samples"]},
        "e2e": e2e,
        "gpu_launches": layer.launches_per_call(T) * calls * nl * args.steps,
    }
    del layer
    torch.cuda.empty_cache()

    if world == 1 and not args.no_configs and args.config == "decode" and not args.experts \
            and not args.bits \
            and nl == 1 and args.groups == 0 and path == moe.PATH_AUTO and y_dtype is None:
        # the other workloads of the layer, measured the same way in this run
        cfgs = {}
        csteps = max(3, min(args.steps, 20))
        extra = {"batched_5bit": workloads.CONFIGS["batched"].scaled(bits=5),
                 "batched_6bit": workloads.CONFIGS["batched"].scaled(bits=6),
                 "prefill_y_f32": workloads.CONFIGS["prefill"]}
        for name in ("tiny", "batched", "prefill", "entropy", "batched_5bit", "batched_6bit",
                     "prefill_y_f32"):
            c = extra.get(name) or workloads.CONFIGS[name]
            # prefill_y_f32: the prefill layer with y kept in fp32 (the A/B of
            # the bf16 storage the tensor-core path uses by default)
            kw = dict(free_sources=True,
                      y_dtype=torch.float32 if name == "prefill_y_f32" else None)
            lay, _, _, _, r = workload_measure(moe, c, dev, rank, world, csteps, args.warmup, kw,
                                               clocks_gpu=gpu_id)
            rf, kn = workload_summary(moe, c, lay, r, peaks, peak_src, name=name)
            cfgs[name] = {"config": dict(workload_config(c),
                                         y_storage=str(lay.y_storage(r["T"])).replace("torch.", "")),
                          "value": r["calls"] * r["T"] / (r["ms"] / 1e3),
                          "unit": "tokens/s", "ms_per_step": r["ms"], "steps": csteps,
                          "roofline": rf, "kernels": kn,
                          "clocks": {k: r["clocks"][k] for k in ("sm_mhz", "sm_max_mhz", "reasons",
                                                                  "samples")},
                          "gpu_launches": lay.launches_per_call(r["T"]) * r["calls"] * csteps}
            del lay
            torch.cuda.empty_cache()
        line["configs"] = cfgs
        # the decode layer's launch-count variants (page "oMLX MoE gate/up 融合
        # 优化", 总结: one fewer launch per layer with gate and up fused): the
        # unfused product (gate, up, activation) and launches without overlap,
        # per layer call and for four chained layers
        ab = {}
        for label, kw, nlay, pdl in (("fused", {}, 1, True),
                                     ("unfused", {"fuse_gate_up": False}, 1, True),
                                     ("fused_no_overlap", {}, 1, False),
                                     ("fused_4_chained", {}, 4, True),
                                     ("unfused_4_chained", {"fuse_gate_up": False}, 4, True)):
            prev = moe.moe_set_launch_overlap(pdl)
            lay, _, _, _, r = workload_measure(moe, cfg, dev, rank, world, csteps, args.warmup,
                                               dict(free_sources=False, **kw), nl=nlay,
                                               clocks_gpu=None, per_kernel=False,
                                               layer_np=layer_np)
            moe.moe_set_launch_overlap(prev)
            ab[label] = {"layer_us_per_call": r["ms"] * 1e3 / (r["calls"] * nlay),
                         "kernels_per_layer": lay.launches_per_call(r["T"]), "layers": nlay}
            del lay
            torch.cuda.empty_cache()
        line["decode_launch_variants"] = ab

    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        # the oracle as it stands, repeated on the same bounded sample until
        # about ten seconds of host work have been timed; then the same sample
        # with one thread in a fresh process
        n = args.cpu_sample or default_sample(cfg)
        tok = wall = cpu = 0.0
        reps = 0
        while wall < CPU_SAMPLE_SECONDS and reps < 50:
            t_, w_, c_ = oracle_sample(cfg, layer_np, x_bits, n)
            tok, wall, cpu, reps = tok + t_, wall + w_, cpu + c_, reps + 1
        unit = "calls" if cfg.calls > 1 else "tokens"
        line["cpu_baseline"] = {"value": tok / wall, "unit": "tokens/s",
                                "cores": round(cpu / wall, 1), "kind": "oracle",
                                "sample": f"{n} {unit} of the same workload, {reps} times "
                                          f"({wall:.1f} s)"}
        one = oracle_one_thread(cfg.name, n)
        if one:
            line["cpu_baseline"]["one_thread"] = {"value": one["value"], "unit": "tokens/s",
                                                  "cores": one["cores"], "sample": one["sample"]}
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()
    return 0


def main(argv=None):
    args = parse_args(argv)
    if args.impl == "reference":
        return run_reference(args)
    return run_ours(args)


if __name__ == "__main__":
    sys.exit(main())
