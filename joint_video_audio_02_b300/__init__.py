"""B300-native (sm_103a) CUDA library for TurboT2VA's joint video-audio sCM + DMD
distillation objective, with a thin Python binding of its C ABI (include/t2va.h)."""

from .binding import (  # noqa: F401
    MAX_MODALITIES,
    STATUS_BAD_TIMESTEP,
    STATUS_BAD_WORKSPACE,
    STATUS_TIMEOUT,
    T2VAError,
    dmd_objective,
    error_string,
    load,
    new_workspace,
    noise,
    noise_rf,
    objective_plan,
    quantize_rows,
    residual_modnorm,
    scm_objective,
    selftest_wait_timeout,
    stage3_objective,
    stage3_objective_cfg,
    stage3_objective_noalloc,
    w8a8_linear,
    workspace_bytes,
    workspace_init,
)
