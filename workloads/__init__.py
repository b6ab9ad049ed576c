"""Seeded synthetic workloads for multi-LoRA SGMV.

This package is shared by the CUDA path's tests and benchmark and by the
oracle's tests. It draws random numbers, rounds them to bf16, builds
adapter-id patterns and names the workload shapes. It holds none of the SGMV
arithmetic (no shrink, expand, segmentation or reduction).
"""

from .gen import (  # noqa: F401
    LLAMA_DIMS,
    Proj,
    SlotInputs,
    Workload,
    WORKLOADS,
    bf16_bits_from_f32,
    distinct_ids,
    f32_from_bf16_bits,
    llama_projs,
    make_backbone_weights,
    make_inputs,
    make_slot_inputs,
    normal_bf16,
    prefill_ids,
    same_ids,
    seed_for,
    tiny_ids,
    workload,
    zipf_ids,
)
