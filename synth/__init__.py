"""Seeded synthetic inputs for the fused LM-head GRPO/GSPO loss.

This package draws the raw inputs (hidden states, head weight, targets,
masks, sequence and document layouts, rewards and the noise added to the
old/reference log-probs).  It holds none of the method's arithmetic: no
logits, log-probs, advantages or losses are computed here.  Both the
oracle's tests and the GPU path's tests and benchmark draw their inputs
from it, so the two sides always see bit-identical data.

bf16 tensors are produced as raw uint16 bit patterns (round-to-nearest-even
from the float32 draw) so that no framework is needed to create them; use
``bf16_bits_to_f32`` for the exact float32 (and hence float64) value of each.
"""
from .workloads import (  # noqa: F401
    CONFIGS,
    WorkloadConfig,
    bf16_bits_to_f32,
    draw_gspo_layout,
    draw_grpo_layout,
    draw_noise,
    draw_rewards,
    f32_to_bf16_bits,
    make_workload,
)
