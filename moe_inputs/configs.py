"""The five synthetic workloads of the routed-expert FFN step, by shape.

Every workload uses seed 0.  Shapes follow the pages' model: 48 MoE layers of
512 routed experts, top-10 plus one always-on shared expert, 24,576
(layer, expert) identities and an 8,445-slot VRAM expert cache
(page "一张 RTX 4090 跑千亿模型，Strata 实测 155 tok/s", §先看结果 and
§如何做到：三层存储; page "从一张到四张 RTX 4090", §先看结果: 48 layers).
Hidden size d=2048, expert width f=768, 3-bit weights in groups of 32 with an
fp16 scale are the workload definition's choices (the pages give no hidden
size or bit layout).

``bias_lambda`` scales the Zipf router bias b[e] = -lambda * s * ln(rank(e))
of the two stack workloads.  It is one global constant calibrated so that the
T=5 verify stack settles near a 95% token-level hit rate (the pages report
94-99% on one RTX 4090, page "一张 RTX 4090 跑千亿模型", §如何做到：三层存储, and
91.3-95.3% at 48% coverage, page "单卡5090跑125B 大模型", §7.2); the value is
written by ``oracle/calibrate_bias.py``.
"""

from dataclasses import dataclass, field
from typing import Optional, Tuple

GROUP = 32          # quantisation group along the input dimension
MARGIN_DELTA = 1e-3  # minimum fp64 gap between the k-th and (k+1)-th router logit

# Zipf bias scale, calibrated once for the T=5 verify stack (95% +- 1% token
# hit rate in the measured pass) and reused for the T=16 stack.
BIAS_LAMBDA = 0.6062


@dataclass(frozen=True)
class Workload:
    cfg_id: int
    name: str
    d: int
    f: int
    n_experts: int
    top_k: int
    n_layers: int
    tokens: int                 # T per call
    calls: int                  # calls per pass
    capacity: int               # expert-cache slots
    preload_all: bool           # every (layer, expert) resident from the start
    zipf_s: Optional[float] = None
    warm_passes: int = 0        # passes over the stream before the measured one
    sweep: Tuple[int, ...] = field(default_factory=tuple)
    seed: int = 0

    @property
    def keys(self) -> int:
        return self.n_layers * self.n_experts

    @property
    def expert_bytes(self) -> int:
        return expert_nbytes(self.d, self.f)


def expert_nbytes(d: int, f: int, group: int = GROUP) -> int:
    """Bytes of one packed expert: 3 matrices of d*f 3-bit weights plus one
    fp16 scale per group of 32 weights."""
    n = 3 * d * f
    return n * 3 // 8 + (n // group) * 2


WORKLOADS = {
    1: Workload(1, "tiny-layer", d=256, f=128, n_experts=16, top_k=2, n_layers=1,
                tokens=4, calls=1, capacity=16, preload_all=True),
    2: Workload(2, "decode-layer", d=2048, f=768, n_experts=512, top_k=10, n_layers=1,
                tokens=1, calls=10_000, capacity=512, preload_all=True),
    3: Workload(3, "verify-stack", d=2048, f=768, n_experts=512, top_k=10, n_layers=48,
                tokens=5, calls=2_000, capacity=8_445, preload_all=False,
                zipf_s=1.1, warm_passes=3),
    4: Workload(4, "concurrent-stack", d=2048, f=768, n_experts=512, top_k=10, n_layers=48,
                tokens=16, calls=2_000, capacity=8_445, preload_all=False,
                zipf_s=0.8, warm_passes=3),
    5: Workload(5, "prefill-chunk", d=2048, f=768, n_experts=512, top_k=10, n_layers=1,
                tokens=12_288, calls=1, capacity=512, preload_all=True,
                sweep=(4_096, 6_144, 8_192, 12_288, 16_384)),
}
