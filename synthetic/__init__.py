"""Seeded synthetic inputs for the joint video-audio distillation objective.

This package draws random latents and network predictions with the shapes and
value distributions of the TurboT2VA workloads. It holds none of the objective's
arithmetic: no noising, no fields, no normalisation. The GPU path and the CPU
oracle both take their inputs from here and from nowhere else.
"""

from .workloads import (  # noqa: F401
    DMD,
    SCM,
    STAGE3,
    STAGE3_CFG,
    WORKLOADS,
    Inputs,
    Workload,
    bf16_bits_from_f32,
    f32_from_bf16_bits,
    make_inputs,
    make_workload_inputs,
    slice_samples,
    workload,
)
