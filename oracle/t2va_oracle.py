"""CPU oracle for the TurboT2VA joint video-audio sCM + DMD distillation objective.

TEST INFRASTRUCTURE. This module exists to check the CUDA library. Only the test
suite, the smoke check and the benchmark's CPU-baseline leg (and its
``--impl reference`` arm) may import it. The library never calls it, and it shares
no code with the CUDA path: it reads the same seeded inputs (bfloat16 bit patterns
or float32 values) and nothing else.

Sources, cited below by the short names in brackets:

[zh] "TurboT2VA：分数正则化一致性蒸馏加速 19B 视频音频联合生成，四步采样 20.1×、
     H20 上全栈 54.67×" (robotworld.top/zh/papers/paper-2608.24674). The only page
     that prints the equations; sections 三 (joint cross-modal distillation),
     3.1 (joint sCM), 四 (joint DMD), 4.1 (modality-balanced joint optimisation).
[en] "TurboT2VA: Score-Regularized Consistency Distillation for Fast Large-Scale
     Text-to-Video-Audio Generation" (robotworld.top/en/papers/paper-2608.24674).
     Gives the paper's equation numbers: Eq. 6 is the per-modality L2
     normalisation of the sCM direction, Eq. 11-12 the DMD residual-scale
     normaliser.

Everything is computed in float64 from the exact values of the inputs (bfloat16
and float32 convert to float64 exactly). Each step is the definition on the page,
written out in the page's order: fields, then the JVP, then the direction, then the
norm, then the residual and the loss, then the gradient by the chain rule. Nothing
is fused, reordered or simplified algebraically.

Readings of points the pages leave open (each one is listed with its reason in the
design notes):
  R1 stop-gradient scope: the whole normalised sCM direction is a constant target,
     so only the first F_theta in r = F_theta - sg(F_theta) - g_bar carries a
     gradient; the DMD normaliser c and g_bar are inside sg as printed.
  R2 the supplied tangent is d/dt of the student x0 prediction along
     (dt, dz^v, dz^a) = (1, F_T^v, F_T^a); the TrigFlow parts of J are added here.
  R3 the forward value of r is -g_bar and of Delta is g_bar_DMD exactly.
  R4 the loss is per sample; gradients are those of the sum over samples.
  R5 c_DMD uses the teacher prediction at the re-noised sample, the same one as in
     g_DMD.
  R6 domain: 0 < t < pi/2 and 1 - gamma^2 sin^2 t > 0; a sample outside it gets NaN
     outputs. A modality with no elements contributes 0 and reports norm 0, c 0.

Pins (tests/test_oracle_pins.py): J against central finite differences and against
automatic differentiation of F_theta on small joint students; the gradients against
automatic differentiation of the loss as printed; closed forms for the direction,
the norm and the DMD term; exact special-angle values; library reductions; the
bfloat16 rounding against a library conversion. The beta/gamma coefficient of the
sCM direction is a definition: it is pinned only to the printed equation (exact
special-angle evaluation), not to an independent source.
"""

from __future__ import annotations

import math
from typing import Dict, List, Optional, Sequence

import numpy as np

HALF_PI = math.pi / 2


# ----------------------------------------------------------------------------
# storage formats
# ----------------------------------------------------------------------------

def decode(a: np.ndarray, dtype: str) -> np.ndarray:
    """Exact float64 value of stored inputs ("bf16" bit patterns, "f32" or "f64")."""
    if dtype == "bf16":
        bits = np.asarray(a, dtype=np.uint16).astype(np.uint32) << 16
        return bits.view(np.float32).astype(np.float64)
    if dtype in ("f32", "f64"):
        return np.asarray(a, dtype=np.float64)
    raise ValueError(dtype)


def round_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round float64 values ONCE to bfloat16, nearest-even; returns the bit patterns.

    bfloat16 keeps 8 significant bits and float32's exponent range, so the rounding
    quantum of a value x = m 2^e (0.5 <= |m| < 1) is 2^(e-8), and never below the
    subnormal quantum 2^-133.
    """
    x = np.asarray(x, dtype=np.float64)
    _, e = np.frexp(x)
    q = np.maximum(e - 8, -133)
    with np.errstate(over="ignore", invalid="ignore"):
        r = np.ldexp(np.rint(np.ldexp(x, -q)), q)
        f = r.astype(np.float32)            # exact: r has at most 8 significant bits
    bits = (f.view(np.uint32) >> 16).astype(np.uint16)
    nan = np.isnan(x)
    if nan.any():
        bits = np.where(nan, np.uint16(0x7FC0), bits)
    return bits


def encode(x: np.ndarray, dtype: str) -> np.ndarray:
    """Round float64 results once to the storage type."""
    if dtype == "bf16":
        return round_to_bf16_bits(x)
    if dtype == "f32":
        with np.errstate(over="ignore"):
            return np.asarray(x, dtype=np.float64).astype(np.float32)
    if dtype == "f64":
        return np.asarray(x, dtype=np.float64)
    raise ValueError(dtype)


def _f64_list(arrs: Sequence[np.ndarray], dtype: str) -> List[np.ndarray]:
    return [decode(a, dtype) for a in arrs]


def _trig(t: np.ndarray):
    """cos t and sin t per sample, shaped [B, 1] to broadcast over latent elements."""
    t64 = np.asarray(t, dtype=np.float64).reshape(-1, 1)
    return np.cos(t64), np.sin(t64)


def valid_samples(t: np.ndarray, gamma: float) -> np.ndarray:
    """R6: samples whose timestep lies in the open interval (0, pi/2) with 1 - gamma^2 sin^2 t > 0."""
    t64 = np.asarray(t, dtype=np.float64).reshape(-1)
    with np.errstate(invalid="ignore"):
        ok = np.isfinite(t64) & (t64 > 0.0) & (t64 < HALF_PI)
        ok &= (1.0 - (float(gamma) ** 2) * np.sin(t64) ** 2) > 0.0
    return ok


# ----------------------------------------------------------------------------
# TrigFlow noising  ([zh] section 三, the noising equation; [en] section 2)
# ----------------------------------------------------------------------------

def trigflow_noise(z0: Sequence[np.ndarray], eps: Sequence[np.ndarray], t: np.ndarray):
    """z_t^m = cos(t) z_0^m + sin(t) eps^m for every modality m, shared t per sample."""
    c, s = _trig(t)
    return [c * z + s * e for z, e in zip(z0, eps)]


def noise(z0, eps, t, dtype: str):
    """The noising step on stored inputs, rounded once to the storage type."""
    zt = trigflow_noise(_f64_list(z0, dtype), _f64_list(eps, dtype), t)
    return [encode(z, dtype) for z in zt]


# ----------------------------------------------------------------------------
# joint sCM  ([zh] section 3.1)
# ----------------------------------------------------------------------------

def trigflow_field(z_t: np.ndarray, x0: np.ndarray, t: np.ndarray) -> np.ndarray:
    """F_q^m = (cos(t) z_t^m - x0_q^m) / sin(t), q in {T, theta}  ([zh] 3.1, the field F_q)."""
    c, s = _trig(t)
    return (c * z_t - x0) / s


def joint_jvp(z_t: np.ndarray, F_theta: np.ndarray, F_teacher: np.ndarray,
              x0_tangent: np.ndarray, t: np.ndarray) -> np.ndarray:
    """J_theta^m = c_t (dF_theta^m/dt + dF_theta^m/dz^v F_T^v + dF_theta^m/dz^a F_T^a),
    c_t = cos t sin t  ([zh] 3.1, the joint JVP; [en] section 2).

    F_theta^m(z^v, z^a, t) = (cos t z^m - x0_theta^m(z^v, z^a, t)) / sin t. Its
    derivative along (1, F_T^v, F_T^a) has three parts:
      * the explicit t-derivative with z and x0_theta held fixed,
        d/dt[(cos t z - x)/sin t] = -z - (cos t / sin t) F_theta;
      * the explicit z-derivative: cos t z^m / sin t depends only on its own
        modality, so that block applied to F_T^m gives (cos t / sin t) F_T^m;
      * the network part -(1/sin t) times the tangent of x0_theta^m along
        (1, F_T^v, F_T^a), which is the supplied tangent (R2). This is where the
        cross-modal Jacobian blocks enter.
    """
    c, s = _trig(t)
    dF_dt_explicit = -z_t - (c / s) * F_theta
    dF_dz_explicit = (c / s) * F_teacher
    network_part = -x0_tangent / s
    c_t = c * s
    return c_t * (dF_dt_explicit + dF_dz_explicit + network_part)


def scm_direction(z_t, x0_teacher, x0_student, x0_tangent, t, beta: float, gamma: float):
    """g_sCM^m = -beta cos t / sqrt(1 - gamma^2 sin^2 t) (sg(F_theta^m) - F_T^m)
                 - gamma cos t sin t z_t^m - J_theta^m   ([zh] 3.1, the sCM direction).

    Inputs are float64 arrays [B, N] of one modality. sg() leaves values unchanged.
    Returns (g, F_theta, F_teacher).
    """
    c, s = _trig(t)
    F_T = trigflow_field(z_t, x0_teacher, t)
    F_theta = trigflow_field(z_t, x0_student, t)
    J = joint_jvp(z_t, F_theta, F_T, x0_tangent, t)
    with np.errstate(invalid="ignore", divide="ignore"):
        consistency = beta * c / np.sqrt(1.0 - gamma ** 2 * s ** 2)
    sg_F_theta = F_theta
    g = -consistency * (sg_F_theta - F_T) - gamma * c * s * z_t - J
    return g, F_theta, F_T


def l2_normalise(g: np.ndarray, eps: float):
    """g_bar = g / (||g||_2 + eps), the norm taken per sample over all latent elements of
    the modality  ([en] Eq. 6; [zh] 3.1). Returns (g_bar, ||g|| per sample)."""
    norm = np.sqrt(np.sum(g * g, axis=1))
    return g / (norm[:, None] + eps), norm


def scm_objective(z_t, x0_teacher, x0_student, x0_tangent, t, beta, gamma, eps_scm,
                  weight, lambda_scm=1.0, dtype="f64") -> Dict[str, object]:
    """Joint sCM loss  L = sum_m w_m ||r_sCM^m||^2 with r = F_theta - sg(F_theta) - g_bar,
    and its gradient with respect to the student x0 prediction ([zh] 3.1; [en] Eq. 6).

    Every argument holding latents is a list with one [B, N_m] array per modality.
    Returns loss [B] (already multiplied by lambda_scm), norm [B, M],
    grad_x0_student (list of [B, N_m]) and the direction g (list) for inspection.
    """
    z_t, x_T, x_S, x_dot = (_f64_list(a, dtype) for a in (z_t, x0_teacher, x0_student, x0_tangent))
    B, M = len(t), len(z_t)
    _, s = _trig(t)
    ok = valid_samples(t, gamma)
    loss = np.zeros(B)
    norms = np.zeros((B, M))
    grads, dirs = [], []
    with np.errstate(invalid="ignore", divide="ignore", over="ignore"):
        for m in range(M):
            g, F_theta, _ = scm_direction(z_t[m], x_T[m], x_S[m], x_dot[m], t, beta, gamma)
            g_bar, n = l2_normalise(g, eps_scm)
            # residual r = F_theta - sg(F_theta) - sg(g_bar); its value is -g_bar (R3)
            r = (F_theta - F_theta) - g_bar
            loss += weight[m] * np.sum(r * r, axis=1)
            norms[:, m] = n
            # chain rule: dL/dr = 2 w r; dr/dF_theta = 1 (first term only, R1);
            # dF_theta/dx0_theta = -1/sin t
            dL_dr = 2.0 * weight[m] * r
            dF_dx = -1.0 / s
            grad = lambda_scm * dL_dr * dF_dx
            grad[~ok] = np.nan
            grads.append(grad)
            dirs.append(g)
    loss = lambda_scm * loss
    loss[~ok] = np.nan
    norms[~ok] = np.nan
    return {"loss": loss, "norm": norms, "grad_x0_student": grads, "g": dirs, "valid": ok}


# ----------------------------------------------------------------------------
# joint DMD  ([zh] section 四; [en] Eq. 11-12)
# ----------------------------------------------------------------------------

def dmd_residual_scale(zhat0: np.ndarray, x0_teacher_hat: np.ndarray) -> np.ndarray:
    """c_DMD^m = (1/N_m) sum_i |zhat0_i^m - zhat0_{T,i}^m| per sample ([en] Eq. 11-12;
    [zh] 四). A modality with no elements gets c = 0 (R6)."""
    n = zhat0.shape[1]
    if n == 0:
        return np.zeros(zhat0.shape[0])
    return np.sum(np.abs(zhat0 - x0_teacher_hat), axis=1) / n


def _dmd_core(zh, yT, yF, eps_dmd, weight, lambda_dmd):
    """The DMD terms on float64 arrays (lists of [B, N_m]); see dmd_objective."""
    B, M = zh[0].shape[0], len(zh)
    loss = np.zeros(B)
    cdmd = np.zeros((B, M))
    grads = []
    for m in range(M):
        g = yF[m] - yT[m]
        c = dmd_residual_scale(zh[m], yT[m])
        g_bar = g / (c[:, None] + eps_dmd)
        # Delta = zhat0 - sg(zhat0 - g_bar); its value is g_bar (R3)
        delta = g_bar
        loss += weight[m] * np.sum(delta * delta, axis=1)
        cdmd[:, m] = c
        # chain rule: dL/dDelta = 2 w Delta; dDelta/dzhat0 = 1 (the sg term is constant)
        grads.append(lambda_dmd * 2.0 * weight[m] * delta)
    return {"loss": lambda_dmd * loss, "cdmd": cdmd, "grad_zhat0": grads}


def dmd_objective(zhat0, x0_teacher_hat, x0_fake, eps_dmd, weight, lambda_dmd=1.0,
                  dtype="f64") -> Dict[str, object]:
    """Joint DMD loss  L = sum_m w_m sum_i (Delta_i^m)^2,
    Delta = zhat0 - sg(zhat0 - g_bar_DMD), g_bar_DMD = g_DMD / (c_DMD + eps_DMD),
    g_DMD = x0_fake - x0_T at the re-noised sample  ([zh] 四; [en] Eq. 11-12).

    The reduction over latent elements is a sum, not a mean ([zh] 四).
    Returns loss [B] (times lambda_dmd), cdmd [B, M] and grad_zhat0 (list).
    """
    zh, yT, yF = (_f64_list(a, dtype) for a in (zhat0, x0_teacher_hat, x0_fake))
    return _dmd_core(zh, yT, yF, eps_dmd, weight, lambda_dmd)


# ----------------------------------------------------------------------------
# classifier-free guidance of the teacher  ([zh] 四, 七; [en] section 3)
# ----------------------------------------------------------------------------

def cfg_prediction(cond: np.ndarray, uncond: np.ndarray, scale: float) -> np.ndarray:
    """The guided teacher prediction uncond + s (cond - uncond).

    The pages state that the teacher's prediction is computed with classifier-free
    guidance, at scale 3.0 for video and 5.0 for audio, without printing the formula;
    this is the standard guidance extrapolation from the unconditional prediction
    through the conditional one (the reading is listed with the design notes).
    """
    return uncond + scale * (cond - uncond)


def dmd_objective_cfg(zhat0, x0_teacher_hat_cond, x0_teacher_hat_uncond, guidance, x0_fake,
                      eps_dmd, weight, lambda_dmd=1.0, dtype="f64") -> Dict[str, object]:
    """The DMD terms with the teacher prediction at the re-noised sample guided per
    modality: y_T^m = cfg_prediction(cond^m, uncond^m, guidance[m]), in float64 from the
    stored inputs; then exactly dmd_objective."""
    zh, yc, yu, yF = (_f64_list(a, dtype) for a in (zhat0, x0_teacher_hat_cond,
                                                    x0_teacher_hat_uncond, x0_fake))
    yT = [cfg_prediction(c, u, float(g)) for c, u, g in zip(yc, yu, guidance)]
    return _dmd_core(zh, yT, yF, eps_dmd, weight, lambda_dmd)


# ----------------------------------------------------------------------------
# stage-3 objective  ([zh] 4.1; [en] section 3)
# ----------------------------------------------------------------------------

def stage3_objective(z_t, x0_teacher, x0_student, x0_tangent, t,
                     zhat0, x0_teacher_hat, x0_fake,
                     beta, gamma, eps_scm, eps_dmd, weight,
                     lambda_scm, lambda_dmd, dtype="f64") -> Dict[str, object]:
    """L_stage3 = lambda_sCM L_sCM + lambda_DMD L_DMD over the same batch and the same
    paired latents ([zh] 4.1; [en] section 3). Both terms use the same w_m."""
    a = scm_objective(z_t, x0_teacher, x0_student, x0_tangent, t, beta, gamma, eps_scm,
                      weight, lambda_scm, dtype)
    b = dmd_objective(zhat0, x0_teacher_hat, x0_fake, eps_dmd, weight, lambda_dmd, dtype)
    ok = a["valid"]
    loss = a["loss"] + b["loss"]
    cdmd = b["cdmd"].copy()
    cdmd[~ok] = np.nan
    loss_dmd = b["loss"].copy()
    loss_dmd[~ok] = np.nan
    grad_dmd = []
    for g in b["grad_zhat0"]:
        g = g.copy()
        g[~ok] = np.nan
        grad_dmd.append(g)
    return {"loss": loss, "loss_scm": a["loss"], "loss_dmd": loss_dmd,
            "norm": a["norm"], "cdmd": cdmd,
            "grad_x0_student": a["grad_x0_student"], "grad_zhat0": grad_dmd,
            "g": a["g"], "valid": ok}



def stage3_objective_cfg(z_t, x0_teacher, x0_student, x0_tangent, t,
                         zhat0, x0_teacher_hat_cond, x0_teacher_hat_uncond, guidance, x0_fake,
                         beta, gamma, eps_scm, eps_dmd, weight,
                         lambda_scm, lambda_dmd, dtype="f64") -> Dict[str, object]:
    """stage3_objective with the DMD teacher prediction guided per modality
    (dmd_objective_cfg)."""
    a = scm_objective(z_t, x0_teacher, x0_student, x0_tangent, t, beta, gamma, eps_scm,
                      weight, lambda_scm, dtype)
    b = dmd_objective_cfg(zhat0, x0_teacher_hat_cond, x0_teacher_hat_uncond, guidance, x0_fake,
                          eps_dmd, weight, lambda_dmd, dtype)
    ok = a["valid"]
    cdmd = b["cdmd"].copy()
    cdmd[~ok] = np.nan
    loss_dmd = b["loss"].copy()
    loss_dmd[~ok] = np.nan
    grad_dmd = []
    for g in b["grad_zhat0"]:
        g = g.copy()
        g[~ok] = np.nan
        grad_dmd.append(g)
    return {"loss": a["loss"] + b["loss"], "loss_scm": a["loss"], "loss_dmd": loss_dmd,
            "norm": a["norm"], "cdmd": cdmd,
            "grad_x0_student": a["grad_x0_student"], "grad_zhat0": grad_dmd,
            "g": a["g"], "valid": ok}


# ----------------------------------------------------------------------------
# TrigFlow -> rectified-flow wrapper  ([zh] 4.2; [en] Eq. 16)
# ----------------------------------------------------------------------------

def trigflow_to_rf(z_trig: Sequence[np.ndarray], t: np.ndarray):
    """z_rf = z_trig / (cos t + sin t) per modality and t_rf = sin t / (cos t + sin t) per
    sample ([zh] 4.2; [en] Eq. 16). Returns (list of z_rf, t_rf [B])."""
    c, s = _trig(t)
    return [z / (c + s) for z in z_trig], (s / (c + s)).reshape(-1)


def noise_rf(z0, eps, t, dtype: str):
    """The noising step and the wrapper on stored inputs: z_t and z_rf, each computed in
    float64 from z0 and eps and rounded once to the storage type, and t_rf in float64."""
    zt = trigflow_noise(_f64_list(z0, dtype), _f64_list(eps, dtype), t)
    zrf, trf = trigflow_to_rf(zt, t)
    return [encode(z, dtype) for z in zt], [encode(z, dtype) for z in zrf], trf
