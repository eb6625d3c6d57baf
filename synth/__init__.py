"""Seeded synthetic inputs shared by the CPU oracle tests and the CUDA path.

This package holds no attention arithmetic: it only draws numbers, rounds
them to the dtype a kernel reads, and packs them into the ``[B, n, h, d]``
layout. Both sides of every parity test receive exactly the same values.
"""

from .inputs import (  # noqa: F401
    MASK_CAUSAL,
    MASK_KEY_PADDING,
    MASK_NONE,
    WORKLOADS,
    Workload,
    attn_inputs,
    bf16_bits_to_f64,
    draw_key_lens,
    draw_normal,
    mha_inputs,
    round_to_bf16_bits,
    round_to_f32,
    widen,
    workload,
)
