"""Workload definitions and seeded input draws.

The workloads follow the TurboT2VA latent shapes: the 512x768 and 1024x1792,
121-frame video latents with 128 channels (TurboT2VA, section 6.4 "default
inference configuration", and section 7 "experimental setup"), paired with an
audio latent of 126 or 504 frames x 128 channels. The value recipe is the same
for every workload:

* clean latents z0 and noises eps ~ N(0, 1);
* teacher prediction x0_T = z0 + 0.1 N(0, 1);
* student prediction x0_S = x0_T + 0.05 N(0, 1);
* student tangent ~ N(0, 0.5^2);
* on-policy student sample zhat0 = z0' + 0.1 N + 0.05 N for a fresh z0';
  fresh noise eps' ~ N(0, 1); teacher prediction at the re-noised sample
  y_T = zhat0 + 0.1 N; fake-score prediction y_fake = y_T + 0.1 N;
* per-sample timestep t = arctan(exp(tau)), tau ~ N(-0.8, 1.6^2), clamped to
  [1e-3, pi/2 - 1e-3] (fixed values for the tiny workload);
* with a guided teacher (mode "stage3_cfg"), the stored teacher prediction above is
  the conditional one and the unconditional one is u = y_T + 0.03 N, drawn after
  every other input of the modality; the guidance scales are 3.0 for video and 5.0
  for audio (TurboT2VA, section 七 training configuration).

Values are drawn in float32 and stored either as float32 or as bfloat16 bit
patterns (uint16, round-to-nearest-even). Nothing here computes any part of the
objective.
"""

from __future__ import annotations

import dataclasses
import math
from typing import Dict, List, Optional, Sequence

import numpy as np

SCM = "scm"
DMD = "dmd"
STAGE3 = "stage3"
STAGE3_CFG = "stage3_cfg"


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    batch: int
    shapes: tuple          # per modality, the per-sample latent shape
    dtype: str             # "f32" or "bf16"
    mode: str              # "scm", "dmd", "stage3" or "stage3_cfg"
    seed: tuple
    beta: float = 1.0
    gamma: float = 0.9
    eps_scm: float = 1e-6
    weight: tuple = (1.0, 1.0)
    lambda_scm: float = 1.0
    lambda_dmd: float = 0.25
    eps_dmd: float = 1e-6
    t_fixed: Optional[tuple] = None
    guidance: tuple = (3.0, 5.0)  # per modality, for "stage3_cfg"
    rf_wrapper: bool = False      # noising also writes the rectified-flow latents and times
    description: str = ""

    @property
    def numels(self) -> List[int]:
        return [int(np.prod(s)) for s in self.shapes]

    @property
    def num_modalities(self) -> int:
        return len(self.shapes)

    @property
    def total_elements(self) -> int:
        return self.batch * sum(self.numels)


def _w(name, **kw) -> Workload:
    return Workload(name=name, **kw)


VIDEO_512x768 = (128, 16, 16, 24)      # 786,432 elements per sample
VIDEO_1024x1792 = (128, 16, 32, 56)    # 3,670,016 elements per sample
AUDIO_126 = (126, 128)                 # 16,128 elements per sample
AUDIO_504 = (504, 128)                 # 64,512 elements per sample

WORKLOADS: Dict[str, Workload] = {}
for _wl in [
    _w("tiny_scm_f32", batch=2, shapes=((128, 2, 4, 6), (64, 16)), dtype="f32",
       mode=SCM, seed=(0,), beta=1.0, gamma=0.5, t_fixed=(0.3, 1.1),
       description="tiny sCM-only case in float32"),
    _w("scm_512x768_bf16", batch=4, shapes=(VIDEO_512x768, AUDIO_126), dtype="bf16",
       mode=SCM, seed=(1,), description="512x768 shape, sCM only, bf16 inputs"),
    _w("stage3_512x768_bf16", batch=4, shapes=(VIDEO_512x768, AUDIO_126), dtype="bf16",
       mode=STAGE3, seed=(2,), description="512x768 shape, sCM+DMD, bf16 inputs"),
    _w("stage3_1024x1792_bf16", batch=1, shapes=(VIDEO_1024x1792, AUDIO_126), dtype="bf16",
       mode=STAGE3, seed=(3,), description="1024x1792 shape, sCM+DMD, bf16 inputs"),
] + [
    _w(f"stage3_sweep_b{b}_bf16", batch=b, shapes=(VIDEO_512x768, AUDIO_504), dtype="bf16",
       mode=STAGE3, seed=(4, b), weight=(1.0, 4.0),
       description=f"batch/modality-imbalance sweep, B={b}, audio 504x128, w=(1,4)")
    for b in (1, 4, 16, 32)
] + [
    _w("stage3_cfg_512x768_bf16", batch=4, shapes=(VIDEO_512x768, AUDIO_126), dtype="bf16",
       mode=STAGE3_CFG, seed=(5,), description="512x768 shape, sCM+DMD with a guided teacher"),
    _w("stage3_cfg_1024x1792_bf16", batch=1, shapes=(VIDEO_1024x1792, AUDIO_126), dtype="bf16",
       mode=STAGE3_CFG, seed=(6,), description="1024x1792 shape, sCM+DMD with a guided teacher"),
    _w("stage3_cfg_rf_512x768_bf16", batch=4, shapes=(VIDEO_512x768, AUDIO_126), dtype="bf16",
       mode=STAGE3_CFG, seed=(7,), rf_wrapper=True,
       description="512x768 shape, noising with the rectified-flow wrapper, sCM+DMD with a "
                   "guided teacher"),
]:
    WORKLOADS[_wl.name] = _wl


def workload(name: str) -> Workload:
    return WORKLOADS[name]


def bf16_bits_from_f32(x: np.ndarray) -> np.ndarray:
    """float32 -> bfloat16 bit patterns, round to nearest even (NaN stays NaN)."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    u = x.view(np.uint32).astype(np.uint64)
    r = (u + 0x7FFF + ((u >> 16) & 1)) >> 16
    nan = np.isnan(x)
    if nan.any():
        r = np.where(nan, (u >> 16) | 0x40, r)
    return r.astype(np.uint16)


def f32_from_bf16_bits(b: np.ndarray) -> np.ndarray:
    return (np.asarray(b, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)


def _store(x: np.ndarray, dtype: str) -> np.ndarray:
    x = np.asarray(x, dtype=np.float32)
    if dtype == "f32":
        return x
    if dtype == "bf16":
        return bf16_bits_from_f32(x)
    raise ValueError(dtype)


@dataclasses.dataclass
class Inputs:
    """One batch of inputs; every list holds one [B, N_m] array per modality."""
    dtype: str
    mode: str
    t: np.ndarray                      # float32 [B]
    z0: List[np.ndarray]
    eps: List[np.ndarray]
    x0_teacher: List[np.ndarray] = None
    x0_student: List[np.ndarray] = None
    x0_tangent: List[np.ndarray] = None
    zhat0: List[np.ndarray] = None
    eps_hat: List[np.ndarray] = None
    x0_teacher_hat: List[np.ndarray] = None
    x0_fake: List[np.ndarray] = None
    x0_teacher_hat_uncond: List[np.ndarray] = None

    @property
    def batch(self) -> int:
        return int(self.t.shape[0])

    @property
    def numels(self) -> List[int]:
        return [int(a.shape[1]) for a in self.z0]


def draw_timesteps(rng: np.random.Generator, batch: int) -> np.ndarray:
    tau = rng.normal(-0.8, 1.6, size=batch)
    t = np.arctan(np.exp(tau))
    t = np.clip(t, 1e-3, math.pi / 2 - 1e-3)
    return t.astype(np.float32)


def make_inputs(batch: int, numels: Sequence[int], dtype: str, mode: str, seed,
                t: Optional[Sequence[float]] = None) -> Inputs:
    """Draw one batch. ``seed`` is an int or a tuple of ints (a numpy SeedSequence key)."""
    key = list(seed) if isinstance(seed, (tuple, list)) else [int(seed)]
    rng = np.random.Generator(np.random.PCG64(np.random.SeedSequence(key)))
    if t is None:
        tt = draw_timesteps(rng, batch)
    else:
        tt = np.asarray(t, dtype=np.float32).reshape(batch)

    def normal(n, scale=1.0):
        a = rng.standard_normal(size=(batch, n), dtype=np.float32)
        if scale != 1.0:
            a *= np.float32(scale)
        return a

    out = Inputs(dtype=dtype, mode=mode, t=tt, z0=[], eps=[])
    scm = mode in (SCM, STAGE3, STAGE3_CFG)
    dmd = mode in (DMD, STAGE3, STAGE3_CFG)
    if scm:
        out.x0_teacher, out.x0_student, out.x0_tangent = [], [], []
    if dmd:
        out.zhat0, out.eps_hat, out.x0_teacher_hat, out.x0_fake = [], [], [], []
    if mode == STAGE3_CFG:
        out.x0_teacher_hat_uncond = []
    for n in numels:
        z0 = normal(n)
        eps = normal(n)
        out.z0.append(_store(z0, dtype))
        out.eps.append(_store(eps, dtype))
        if scm:
            xt = z0 + normal(n, 0.1)
            xs = xt + normal(n, 0.05)
            out.x0_teacher.append(_store(xt, dtype))
            out.x0_student.append(_store(xs, dtype))
            out.x0_tangent.append(_store(normal(n, 0.5), dtype))
            del xt, xs
        if dmd:
            zh = normal(n) + normal(n, 0.1) + normal(n, 0.05)
            eh = normal(n)
            yt = zh + normal(n, 0.1)
            yf = yt + normal(n, 0.1)
            out.zhat0.append(_store(zh, dtype))
            out.eps_hat.append(_store(eh, dtype))
            out.x0_teacher_hat.append(_store(yt, dtype))
            out.x0_fake.append(_store(yf, dtype))
            if mode == STAGE3_CFG:
                out.x0_teacher_hat_uncond.append(_store(yt + normal(n, 0.03), dtype))
            del zh, eh, yt, yf
        del z0, eps
    return out


def make_workload_inputs(wl: Workload, seed_offset: Optional[int] = None) -> Inputs:
    seed = tuple(wl.seed) + ((seed_offset,) if seed_offset is not None else ())
    return make_inputs(wl.batch, wl.numels, wl.dtype, wl.mode, seed, t=wl.t_fixed)


def slice_samples(inp: Inputs, samples: Sequence[int]) -> Inputs:
    """The same inputs restricted to the listed samples (every sample is independent)."""
    idx = np.asarray(list(samples), dtype=np.int64)
    kw = {}
    for f in dataclasses.fields(Inputs):
        v = getattr(inp, f.name)
        if isinstance(v, list):
            kw[f.name] = [a[idx] for a in v]
        elif v is None:
            kw[f.name] = None
        elif f.name == "t":
            kw[f.name] = v[idx]
        else:
            kw[f.name] = v
    return Inputs(**kw)
