"""Seeded synthetic inputs of the routed-expert FFN step (no step arithmetic)."""

from .configs import GROUP, MARGIN_DELTA, BIAS_LAMBDA, Workload, WORKLOADS, expert_nbytes
from .gen import (Synth, synth, bf16_bits_from_f64, bf16_bits_to_f64, fp16_from_f64,
                  expert_sections)

__all__ = ["GROUP", "MARGIN_DELTA", "BIAS_LAMBDA", "Workload", "WORKLOADS", "expert_nbytes",
           "Synth", "synth", "bf16_bits_from_f64", "bf16_bits_to_f64", "fp16_from_f64",
           "expert_sections"]
