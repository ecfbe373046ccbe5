"""Helpers for the GPU parity tests: upload seeded inputs, run the library through
its C ABI, run the oracle on the same inputs, compare with the stated tolerances.

Tolerances (per-sample scalars relative, gradients against the largest gradient):
  loss / norm / c_DMD: rel <= 1e-5 for float32 inputs, <= 1e-4 for bfloat16 inputs;
  gradients: max |gpu - oracle| <= 1e-3 * max |oracle| per sample and modality.
Noise: one output ulp plus the float32 evaluation error of cos t z0 + sin t eps
(test_noise_parity).
"""

from __future__ import annotations

import dataclasses
from typing import List, Optional, Sequence

import numpy as np
import torch

import joint_video_audio_02_b300 as t2va
import oracle
import synthetic as S

RTOL = {"f32": 1e-5, "bf16": 1e-4}
GRAD_FRAC = 1e-3
STAGE3_MODES = (S.STAGE3, S.STAGE3_CFG)
SCM_MODES = (S.SCM,) + STAGE3_MODES
DMD_MODES = (S.DMD,) + STAGE3_MODES


def to_device(arrs: Sequence[np.ndarray], dtype: str, stride_pad: int = 0) -> List[torch.Tensor]:
    """Per-modality [B, N] arrays -> CUDA tensors; with stride_pad > 0 each sample is
    placed in a row of N + stride_pad elements (a strided view)."""
    out = []
    for a in arrs:
        if dtype == "bf16":
            t = torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16)
        else:
            t = torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32))
        if stride_pad:
            B, N = t.shape
            buf = torch.zeros((B, N + stride_pad), dtype=t.dtype)
            buf[:, :N] = t
            t = buf.cuda()[:, :N]
        else:
            t = t.cuda()
        out.append(t)
    return out


def to_host(ts: Sequence[torch.Tensor], dtype: str) -> List[np.ndarray]:
    if dtype == "bf16":
        return [t.contiguous().view(torch.int16).cpu().numpy().view(np.uint16) for t in ts]
    return [t.contiguous().cpu().numpy() for t in ts]


def alloc_like(ts: Sequence[torch.Tensor], dtype=None, fill: float = 0.0) -> List[torch.Tensor]:
    """New tensors with the same per-sample geometry (sample stride included)."""
    out = []
    for t in ts:
        B, N = t.shape
        dt = dtype or t.dtype
        rows = t.stride(0) if (B > 1 and t.stride(0) != N) else N
        buf = torch.full((B, rows), fill, dtype=dt, device=t.device)
        out.append(buf[:, :N])
    return out


def grads_like(ts: Sequence[torch.Tensor], fill: float = 0.0) -> List[torch.Tensor]:
    return alloc_like(ts, torch.float32, fill)


@dataclasses.dataclass
class Params:
    beta: float = 1.0
    gamma: float = 0.9
    eps_scm: float = 1e-6
    eps_dmd: float = 1e-6
    weight: tuple = (1.0, 1.0)
    lambda_scm: float = 1.0
    lambda_dmd: float = 0.25
    guidance: tuple = (3.0, 5.0)

    @staticmethod
    def of(wl: S.Workload) -> "Params":
        return Params(wl.beta, wl.gamma, wl.eps_scm, wl.eps_dmd, tuple(wl.weight), wl.lambda_scm,
                      wl.lambda_dmd, tuple(wl.guidance))


def gpu_run(inp: S.Inputs, p: Params, mode: str, stride_pad: int = 0, accumulate_into=None,
            alias: bool = False, workspace=None, t_override=None):
    """GPU noise -> objective through the C ABI. Returns numpy results and the status word."""
    dt = inp.dtype
    B = inp.batch
    t = torch.from_numpy(np.asarray(t_override if t_override is not None else inp.t, np.float32)).cuda()
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    M = len(inp.z0)
    ws = workspace if workspace is not None else t2va.new_workspace(B, M)
    out = {"status_tensor": status}
    loss = torch.full((B,), float("nan"), device="cuda")
    norm = torch.full((B * M,), float("nan"), device="cuda")
    cdmd = torch.full((B * M,), float("nan"), device="cuda")
    if mode in SCM_MODES:
        z0 = to_device(inp.z0, dt, stride_pad)
        eps = to_device(inp.eps, dt, stride_pad)
        zt = alloc_like(z0)
        t2va.noise(z0, eps, zt, t, status=status)
        xT = to_device(inp.x0_teacher, dt, stride_pad)
        xS = to_device(inp.x0_student, dt, stride_pad)
        tan = to_device(inp.x0_tangent, dt, stride_pad)
        gS = grads_like(zt)
        if accumulate_into is not None:
            for g, a in zip(gS, accumulate_into["grad_x0_student"]):
                g.copy_(torch.from_numpy(np.asarray(a, np.float32)))
        out["zt"] = to_host(zt, dt)
    if mode in DMD_MODES:
        zh = to_device(inp.zhat0, dt, stride_pad)
        yT = to_device(inp.x0_teacher_hat, dt, stride_pad)
        yF = to_device(inp.x0_fake, dt, stride_pad)
        gD = grads_like(zh)
        if accumulate_into is not None:
            for g, a in zip(gD, accumulate_into["grad_zhat0"]):
                g.copy_(torch.from_numpy(np.asarray(a, np.float32)))
    if mode == S.STAGE3_CFG:
        yU = to_device(inp.x0_teacher_hat_uncond, dt, stride_pad)
    acc = accumulate_into is not None
    if mode == S.SCM:
        t2va.scm_objective(zt, xT, xS, tan, t, beta=p.beta, gamma=p.gamma, eps_scm=p.eps_scm,
                           weight=p.weight, lambda_scm=p.lambda_scm, grad_x0_student=gS, loss=loss,
                           norm=norm, accumulate=acc, workspace=ws, status=status)
    elif mode == S.DMD:
        t2va.dmd_objective(zh, yT, yF, eps_dmd=p.eps_dmd, weight=p.weight, lambda_dmd=p.lambda_dmd,
                           grad_zhat0=gD, loss=loss, cdmd=cdmd, accumulate=acc, workspace=ws,
                           status=status)
    else:
        loss_s = torch.full((B,), float("nan"), device="cuda")
        loss_d = torch.full((B,), float("nan"), device="cuda")
        if alias:
            gD = gS
        common = dict(beta=p.beta, gamma=p.gamma, eps_scm=p.eps_scm, eps_dmd=p.eps_dmd,
                      weight=p.weight, lambda_scm=p.lambda_scm, lambda_dmd=p.lambda_dmd,
                      grad_x0_student=gS, grad_zhat0=gD, loss=loss, loss_scm=loss_s,
                      loss_dmd=loss_d, norm=norm, cdmd=cdmd, accumulate=acc, workspace=ws,
                      status=status)
        if mode == S.STAGE3_CFG:
            t2va.stage3_objective_cfg(zt, xT, xS, tan, t, zh, yT, yU, yF, guidance=p.guidance,
                                      **common)
        else:
            t2va.stage3_objective(zt, xT, xS, tan, t, zh, yT, yF, **common)
        out["loss_scm"] = loss_s.cpu().numpy()
        out["loss_dmd"] = loss_d.cpu().numpy()
    torch.cuda.synchronize()
    out["loss"] = loss.cpu().numpy()
    out["norm"] = norm.cpu().numpy().reshape(B, M)
    out["cdmd"] = cdmd.cpu().numpy().reshape(B, M)
    if mode in SCM_MODES:
        out["grad_x0_student"] = [g.contiguous().cpu().numpy() for g in gS]
    if mode in DMD_MODES:
        out["grad_zhat0"] = [g.contiguous().cpu().numpy() for g in gD]
    out["status"] = int(status.item())
    return out


def oracle_run(inp: S.Inputs, p: Params, mode: str, t_override=None):
    dt = inp.dtype
    t = np.asarray(t_override if t_override is not None else inp.t, np.float32)
    out = {}
    if mode in SCM_MODES:
        zt = oracle.noise(inp.z0, inp.eps, t, dt)
        out["zt"] = zt
    if mode == S.SCM:
        r = oracle.scm_objective(zt, inp.x0_teacher, inp.x0_student, inp.x0_tangent, t, p.beta, p.gamma,
                                 p.eps_scm, p.weight, p.lambda_scm, dt)
    elif mode == S.DMD:
        r = oracle.dmd_objective(inp.zhat0, inp.x0_teacher_hat, inp.x0_fake, p.eps_dmd, p.weight,
                                 p.lambda_dmd, dt)
    elif mode == S.STAGE3_CFG:
        r = oracle.stage3_objective_cfg(zt, inp.x0_teacher, inp.x0_student, inp.x0_tangent, t,
                                        inp.zhat0, inp.x0_teacher_hat, inp.x0_teacher_hat_uncond,
                                        p.guidance, inp.x0_fake, p.beta, p.gamma, p.eps_scm,
                                        p.eps_dmd, p.weight, p.lambda_scm, p.lambda_dmd, dt)
    else:
        r = oracle.stage3_objective(zt, inp.x0_teacher, inp.x0_student, inp.x0_tangent, t,
                                    inp.zhat0, inp.x0_teacher_hat, inp.x0_fake, p.beta, p.gamma,
                                    p.eps_scm, p.eps_dmd, p.weight, p.lambda_scm, p.lambda_dmd, dt)
    out.update(r)
    return out


def assert_rel(got, ref, rtol, what=""):
    got = np.asarray(got, np.float64)
    ref = np.asarray(ref, np.float64)
    assert got.shape == ref.shape, (what, got.shape, ref.shape)
    nan_ref = np.isnan(ref)
    assert np.array_equal(np.isnan(got), nan_ref), f"{what}: NaN pattern differs"
    g, r = got[~nan_ref], ref[~nan_ref]
    err = np.abs(g - r)
    lim = rtol * np.abs(r) + 1e-30
    assert np.all(err <= lim), f"{what}: worst rel err {np.max(err / (np.abs(r) + 1e-30)):.3e} > {rtol}"


def assert_grad(got, ref, what="", frac=GRAD_FRAC):
    """Per sample: max |got - ref| <= frac * max |ref| over that sample's elements."""
    got = np.asarray(got, np.float64)
    ref = np.asarray(ref, np.float64)
    assert got.shape == ref.shape, (what, got.shape, ref.shape)
    nan_ref = np.isnan(ref)
    assert np.array_equal(np.isnan(got), nan_ref), f"{what}: NaN pattern differs"
    for b in range(ref.shape[0]):
        ok = ~nan_ref[b]
        if not ok.any():
            continue
        scale = np.max(np.abs(ref[b, ok]))
        err = np.max(np.abs(got[b, ok] - ref[b, ok]))
        assert err <= frac * scale, f"{what} sample {b}: max abs err {err:.3e} > {frac} * {scale:.3e}"


def ulp_diff_bf16(a: np.ndarray, b: np.ndarray) -> np.ndarray:
    """Distance in bfloat16 units in the last place between two bit-pattern arrays."""
    def ordered(x):
        x = x.astype(np.int32)
        return np.where(x & 0x8000, 0x8000 - (x & 0x7FFF), x + 0x8000)
    return np.abs(ordered(a) - ordered(b))


def ulp_diff_f32(a: np.ndarray, b: np.ndarray) -> np.ndarray:
    def ordered(x):
        x = np.asarray(x, np.float32).view(np.int32).astype(np.int64)
        return np.where(x < 0, -(x & 0x7FFFFFFF), x)
    return np.abs(ordered(a) - ordered(b))


def select(gpu: dict, samples: Sequence[int]) -> dict:
    """GPU results restricted to the listed samples (to compare with an oracle run on them)."""
    idx = list(samples)
    out = dict(gpu)
    for k in ("loss", "loss_scm", "loss_dmd", "norm", "cdmd"):
        if k in gpu:
            out[k] = gpu[k][idx]
    for k in ("grad_x0_student", "grad_zhat0", "zt"):
        if k in gpu:
            out[k] = [a[idx] for a in gpu[k]]
    return out


def compare(gpu, ref, dtype: str, mode: str):
    """Assert parity of every output of one call."""
    rtol = RTOL[dtype]
    assert_rel(gpu["loss"], ref["loss"], rtol, "loss")
    M = gpu["norm"].shape[1]
    if mode in SCM_MODES:
        assert_rel(gpu["norm"], ref["norm"], rtol, "norm")
        for m in range(M):
            assert_grad(gpu["grad_x0_student"][m], ref["grad_x0_student"][m], f"grad_x0_student[{m}]")
    if mode in DMD_MODES:
        assert_rel(gpu["cdmd"], ref["cdmd"], rtol, "cdmd")
        for m in range(M):
            assert_grad(gpu["grad_zhat0"][m], ref["grad_zhat0"][m], f"grad_zhat0[{m}]")
    if mode in STAGE3_MODES:
        assert_rel(gpu["loss_scm"], ref["loss_scm"], rtol, "loss_scm")
        assert_rel(gpu["loss_dmd"], ref["loss_dmd"], rtol, "loss_dmd")
