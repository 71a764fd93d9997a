"""CPU oracle of the routed-expert FFN step -- TEST INFRASTRUCTURE ONLY.

Plain, slow, fp64 numpy restatement of what the step computes, written from
the definitions so that a reader can check it by eye.  Only ``tests/``,
``__graft_entry__.smoke()`` and the CPU-baseline leg of ``bench.py`` may
import it.  The CUDA library never links, imports or calls it, and it shares
no code with the CUDA library; the only common module is ``moe_inputs``,
which draws seeded inputs and holds none of the step's arithmetic.

The pages this follows are three blog posts about an offloaded-MoE serving
engine:
  P1  "一张 RTX 4090 跑千亿模型，Strata 实测 155 tok/s" (cnblogs softlin/p/23460041)
  P2  "单卡5090跑125B 大模型：Strata 把服务器级 MoE 拉进普通 PC" (juejin 7694490288811999272)
  P3  "从一张到四张 RTX 4090:千亿模型从能单人用到能多人用" (cnblogs softlin/p/23486755)
They fix the structure (512 routed experts, top-10 plus one shared expert per
token per layer, a fixed-capacity VRAM cache keyed by (layer, expert) whose
misses are fetched from pinned host RAM, hits/lookups counted per token pick,
one expert fetch shared by all tokens of a verify batch).  They print no
formulas for routing or the expert FFN and no worked numeric example; those
come from the workload definition (softmax over all experts, top-k,
renormalise over the chosen k; SwiGLU; 3-bit groups of 32 with fp16 scales;
LRU by (layer, expert), ties to the lower slot id) and are restated here.

Pins (what each function is checked against, besides itself) are listed in
each module's docstring.  Parity unpinned: the Zipf-bias scale lambda of the
stack workloads is calibrated, not fixed by the pages.

Modules: ``packed`` (canonical 3-bit format -> fp64 weights), ``routing``,
``ffn``, ``cache`` (LRU slot cache), ``stack`` (multi-layer call driver).
"""

from .packed import unpack_expert, unpack_codes
from .routing import router_logits, softmax, topk_ascending, route
from .ffn import silu, expert_forward, layer_forward
from .cache import ExpertCache, LayerCallResult
from .stack import StackOracle

__all__ = ["unpack_expert", "unpack_codes", "router_logits", "softmax", "topk_ascending",
           "route", "silu", "expert_forward", "layer_forward", "ExpertCache",
           "LayerCallResult", "StackOracle"]
