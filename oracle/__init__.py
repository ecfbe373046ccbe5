"""CPU oracles (float64, numpy) for the joint video-audio sCM + DMD objective
(t2va_oracle), the post-scale W8A8 linear (w8a8_oracle) and the fused gated residual +
modulated RMS normalisation (fused_ops_oracle).

TEST INFRASTRUCTURE ONLY: imported by the test suite, the smoke check and the
benchmark's CPU legs. The CUDA library never uses them.
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
