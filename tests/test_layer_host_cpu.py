"""Host-side decisions of MoELayer that need no GPU: which kernel family the
products take, when an adaptive-k layer queues both (gated on k), and how
many kernels a call launches.  The layer object is built without weights."""
import pytest

import workloads
from sparse_moe_expert_gb300 import PATH_AUTO, PATH_GEMV, PATH_TC, path_k_range
from sparse_moe_expert_gb300.layer import MoELayer


def bare_layer(cfg, path=PATH_AUTO, fused=True, capacity=None):
    m = object.__new__(MoELayer)
    m.E, m.H, m.I, m.bits = cfg.E, cfg.H, cfg.I, cfg.bits
    m.k_fixed, m.kmax = cfg.k, cfg.slots
    m.path, m.fused, m.capacity, m.groups = path, fused, capacity, 0
    return m


CFG = workloads.CONFIGS


@pytest.mark.parametrize("name,family,split", [
    ("decode", PATH_GEMV, 0),     # 1 token
    ("batched", PATH_GEMV, 0),    # fixed k = 4: 4 tokens per expert
    ("prefill", PATH_TC, 0),      # fixed k = 8: 256 tokens per expert
    ("entropy", PATH_TC, 2),      # adaptive: k = 1 gives 16 tokens per expert, k = 2 gives 32
    ("tiny", PATH_GEMV, 0),
])
def test_family_and_k_split_of_the_workloads(name, family, split):
    cfg = CFG[name]
    m = bare_layer(cfg)
    assert m.resolved_path(cfg.T) == family
    assert m.k_split(cfg.T) == split


def test_k_split_needs_auto_adaptive_fused_and_streamable_rows():
    cfg = CFG["entropy"]
    assert bare_layer(cfg, path=PATH_TC).k_split(cfg.T) == 0
    assert bare_layer(cfg, fused=False).k_split(cfg.T) == 0
    assert bare_layer(cfg.scaled(k=3)).k_split(cfg.T) == 0            # fixed k
    assert bare_layer(cfg.scaled(I=1536 + 64)).k_split(cfg.T) == 0    # 8-bit rows of 1600 codes
    assert bare_layer(cfg.scaled(T=64)).k_split(64) == 0             # GEMV for every k
    assert bare_layer(cfg.scaled(T=2048)).k_split(2048) == 0         # tensor cores for every k
    # the split moves with the tokens per expert: T k / E >= 24 from k = 3
    assert bare_layer(cfg.scaled(T=256)).k_split(256) == 3


def test_launch_counts():
    e = CFG["entropy"]
    # router + finalize + permute (T 512 spans 16 token groups), row permute,
    # two gated launches per product, combine
    assert bare_layer(e).launches_per_call(e.T) == 3 + 6
    assert bare_layer(e, path=PATH_TC).launches_per_call(e.T) == 3 + 1 + 1 + 2
    d = CFG["decode"]
    assert bare_layer(d).launches_per_call(1) == 4   # router with the grouping, gate_up, down, combine
    b = CFG["batched"]
    # T 64 spans several token groups: router, then the finalize with the grouping
    assert bare_layer(b).launches_per_call(b.T) == 2 + 3


def test_k_range_flags_encode_the_header_layout():
    f = path_k_range(2, 3)
    assert f & 0x200 and (f >> 16) & 0xFF == 2 and (f >> 24) & 0x7F == 3
    assert (PATH_TC | f) & 0xFF == PATH_TC
