"""CPU oracle (float64, numpy) for the joint video-audio sCM + DMD objective.

TEST INFRASTRUCTURE ONLY: imported by the test suite, the smoke check and the
benchmark's CPU-baseline leg. The CUDA library never uses it.
"""

from .t2va_oracle import (  # noqa: F401
    cfg_prediction,
    decode,
    dmd_objective,
    dmd_objective_cfg,
    dmd_residual_scale,
    encode,
    joint_jvp,
    l2_normalise,
    noise,
    noise_rf,
    round_to_bf16_bits,
    scm_direction,
    scm_objective,
    stage3_objective,
    stage3_objective_cfg,
    trigflow_field,
    trigflow_noise,
    trigflow_to_rf,
    valid_samples,
)
