"""CPU oracle for the quantized sparse-MoE SwitchGLU layer forward.

TEST INFRASTRUCTURE ONLY.  Nothing in the product path imports, links or
executes this package: only ``tests/``, ``__graft_entry__.smoke()`` and the
``cpu_baseline`` / ``--impl reference`` legs of ``bench.py`` use it.  It shares
no code with the CUDA library (``sparse_moe_expert_gb300``); the two meet only
in the seeded inputs of ``workloads``.

What it computes, step by step, is the plain definition of each stage:

* router logits: a bias-free linear layer in fp32 with one fixed summation
  order (``router_fp32.c``); optional per-expert logit bias and inverse
  temperature;
* softmax, the k largest probabilities (ties to the lower expert id) and
  the routing weights, renormalised over the chosen k or not;
* the per-batch adaptive k from the mean per-token softmax entropy (nats):
  H < 1.2 -> 1, 1.2 <= H < 2.5 -> 2, otherwise 3;
* a stable grouping of the (token, slot) assignments by expert;
* the gate/up concatenation along the output axis, the affine dequantization
  w = scale * code + bias per group of 64, SiLU(gate) * up, the down
  projection and the routing-weighted sum back to token order, in float64.

Pages cited in this package:
  [A] "Qwen3.5 Block在llama.cpp中的映射与优化原理" (mokono.cn/news/2993189)
  [B] "Qwen3.5-MoE与Qwen3-MoE架构差异深度解析" (jsqmd.com/news/1062166)
  [C] "oMLX MoE gate/up 融合优化：qwen35_moe_gate_up 实现剖析" (xdnf.cn/news/169715)

Pins (tests/test_oracle_pins.py) tie every function to something other than
itself: closed-form entropies, brute-force top-k and sort, the quantizer's
error bound, one-hot probes, a dense all-experts evaluation and exactly
representable fusion cases.
"""
from .moe import *  # noqa: F401,F403
from .moe import __all__  # noqa: F401
