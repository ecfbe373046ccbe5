"""CPU oracle of the fused residual + modulated RMS normalisation (TurboT2VA, section 6.3 of
the robotworld.top/zh reading, "fused multimodal Transformer operations").

TEST INFRASTRUCTURE ONLY. Nothing in the library imports this module; only tests/,
__graft_entry__.smoke() and bench.py's CPU legs may call it.

The pages name the fused patterns of the joint Transformer (a normalisation combined
with a modality- and timestep-dependent modulation, followed by a gated residual
update; modulated RMS normalisation; adaptive scale-shift modulation; gated residual
update) but print no formulas. This oracle takes the standard forms of those
operations in diffusion Transformers, read as one step of the residual stream:

  h'  = h + gate * u                                   (gated residual update)
  y   = h' / sqrt(mean(h'^2) + eps) * (1 + scale) + shift
                                                       (modulated RMS normalisation)

per token row of width D, with gate, scale and shift vectors of width D per sample
(the timestep / modality modulation). h' is stored in the latent dtype, and the
normalisation reads the stored h' (as the unfused operators would, one after the
other). Everything else is float64.
"""

from __future__ import annotations

from typing import Optional

import numpy as np


def rms_norm(x: np.ndarray, eps: float) -> np.ndarray:
    """x / sqrt(mean(x^2) + eps) over the last axis, float64."""
    x = np.asarray(x, np.float64)
    ms = np.mean(x * x, axis=-1, keepdims=True)
    return x / np.sqrt(ms + eps)


def modulate(x: np.ndarray, scale: Optional[np.ndarray], shift: Optional[np.ndarray]) -> np.ndarray:
    """Adaptive scale-shift modulation x (1 + scale) + shift (either may be absent)."""
    y = np.asarray(x, np.float64)
    if scale is not None:
        y = y * (1.0 + np.asarray(scale, np.float64))
    if shift is not None:
        y = y + np.asarray(shift, np.float64)
    return y


def gated_residual(h: np.ndarray, u: np.ndarray, gate: Optional[np.ndarray]) -> np.ndarray:
    """h + gate * u, float64 (gate absent: 1)."""
    g = 1.0 if gate is None else np.asarray(gate, np.float64)
    return np.asarray(h, np.float64) + g * np.asarray(u, np.float64)


def per_row(vec: Optional[np.ndarray], rows: int, rows_per_sample: int) -> Optional[np.ndarray]:
    """Expand per-sample vectors [B, D] to per-row [rows, D] (row r belongs to sample
    r // rows_per_sample)."""
    if vec is None:
        return None
    v = np.asarray(vec, np.float64)
    return v[np.arange(rows) // rows_per_sample]


def residual_modnorm(h, u, gate, scale, shift, eps: float, rows_per_sample: int, round_to):
    """The fused step on float64 inputs [rows, D]: returns (h' rounded by `round_to`, y).
    `round_to` maps float64 values to the stored dtype's values (float64)."""
    rows = np.asarray(h).shape[0]
    if u is None:
        h2 = np.asarray(h, np.float64)
    else:
        h2 = round_to(gated_residual(h, u, per_row(gate, rows, rows_per_sample)))
    y = modulate(rms_norm(h2, eps), per_row(scale, rows, rows_per_sample),
                 per_row(shift, rows, rows_per_sample))
    return h2, y
