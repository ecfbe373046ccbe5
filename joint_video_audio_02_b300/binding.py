"""Thin ctypes binding of the C ABI in include/t2va.h.

Argument marshalling only: every tensor is a CUDA tensor owned by the caller,
every step of the computation runs in libt2va.so's kernels on the caller's
current (or given) stream. There is no CPU path; loading fails loudly if the
library is not built.

A latent of modality m is a tensor whose first dimension is the sample and
whose remaining dimensions are contiguous; all tensors of one modality share
that geometry (the gradients too, in float32).
"""

from __future__ import annotations

import ctypes
import os
from typing import List, Optional, Sequence

import torch

from .build import LIB

c_int, c_float, c_void_p, c_size_t, c_int64, c_uint32 = (
    ctypes.c_int, ctypes.c_float, ctypes.c_void_p, ctypes.c_size_t, ctypes.c_int64, ctypes.c_uint32)

T2VA_FLOAT32 = 0
T2VA_BFLOAT16 = 1
T2VA_INT8 = 2
MAX_MODALITIES = 4

STATUS_BAD_TIMESTEP = 0x1
STATUS_TIMEOUT = 0x2
STATUS_BAD_WORKSPACE = 0x4

NOALLOC_SCRATCH_BYTES = 1 << 20   # T2VA_NOALLOC_SCRATCH_BYTES

EXPORTED = ("t2va_error_string", "t2va_abi_version", "t2va_workspace_bytes", "t2va_workspace_init",
            "t2va_noise", "t2va_scm_objective", "t2va_dmd_objective", "t2va_stage3_objective",
            "t2va_stage3_objective_noalloc", "t2va_noise_rf", "t2va_stage3_objective_cfg",
            "t2va_quantize_rows", "t2va_w8a8_linear", "t2va_selftest_wait_timeout",
            "t2va_residual_modnorm", "t2va_objective_plan_query")


class Segment(ctypes.Structure):
    _fields_ = [("numel", c_int64), ("sample_stride", c_int64)]


class ObjectivePlan(ctypes.Structure):
    _fields_ = [("grid", c_int), ("threads", c_int), ("vectors_per_chunk", c_int),
                ("chunks", c_int * MAX_MODALITIES), ("outputs_modality", c_int),
                ("outputs_chunk", c_int), ("one_wave", c_int)]


class T2VAError(RuntimeError):
    def __init__(self, code: int, where: str):
        self.code = code
        super().__init__(f"{where}: t2va error {code}: {error_string(code)}")


_LIB = None


def _declare(lib):
    P = c_void_p
    lib.t2va_error_string.argtypes = [c_int]
    lib.t2va_error_string.restype = ctypes.c_char_p
    lib.t2va_abi_version.argtypes = []
    lib.t2va_abi_version.restype = c_int
    lib.t2va_workspace_bytes.argtypes = [c_int, c_int]
    lib.t2va_workspace_bytes.restype = c_size_t
    lib.t2va_workspace_init.argtypes = [P, c_size_t, c_uint32, P]
    lib.t2va_workspace_init.restype = c_int
    seg = ctypes.POINTER(Segment)
    lib.t2va_noise.argtypes = [c_int, c_int, seg, c_int, P, P, P, P, P, P]
    lib.t2va_noise.restype = c_int
    lib.t2va_scm_objective.argtypes = [c_int, c_int, seg, c_int, P, P, P, P, P,
                                       c_float, c_float, c_float, P, c_float,
                                       P, c_int, P, P, P, c_size_t, P, P]
    lib.t2va_scm_objective.restype = c_int
    lib.t2va_dmd_objective.argtypes = [c_int, c_int, seg, c_int, P, P, P, c_float, P, c_float,
                                       P, c_int, P, P, P, c_size_t, P, P]
    lib.t2va_dmd_objective.restype = c_int
    lib.t2va_stage3_objective.argtypes = [c_int, c_int, seg, c_int, P, P, P, P, P, P, P, P,
                                          c_float, c_float, c_float, c_float, P, c_float, c_float,
                                          P, P, c_int, P, P, P, P, P, P, c_size_t, P, P]
    lib.t2va_stage3_objective.restype = c_int
    lib.t2va_stage3_objective_noalloc.argtypes = [c_int, c_int, seg, c_int, P, P, P, P, P, P, P, P,
                                                  c_float, c_float, c_float, c_float, P, c_float,
                                                  c_float, P, P, c_int, P, P, P, P, P, P, P]
    lib.t2va_stage3_objective_noalloc.restype = c_int
    lib.t2va_noise_rf.argtypes = [c_int, c_int, seg, c_int, P, P, P, P, P, P, P, P]
    lib.t2va_noise_rf.restype = c_int
    lib.t2va_stage3_objective_cfg.argtypes = [c_int, c_int, seg, c_int, P, P, P, P, P, P, P, P, P, P,
                                              c_float, c_float, c_float, c_float, P, c_float, c_float,
                                              P, P, c_int, P, P, P, P, P, P, c_size_t, P, P]
    lib.t2va_stage3_objective_cfg.restype = c_int
    lib.t2va_quantize_rows.argtypes = [c_int64, c_int64, c_int, P, c_int64, c_float, c_int, P, c_int64, P, P]
    lib.t2va_quantize_rows.restype = c_int
    lib.t2va_w8a8_linear.argtypes = [c_int64, c_int64, c_int64, c_int, P, P, P, P, P, c_int, P, P, P]
    lib.t2va_w8a8_linear.restype = c_int
    lib.t2va_selftest_wait_timeout.argtypes = [P, P]
    lib.t2va_selftest_wait_timeout.restype = c_int
    lib.t2va_residual_modnorm.argtypes = [c_int64, c_int64, c_int64, c_int, P, P, P, P, P, c_float, P, P, P]
    lib.t2va_residual_modnorm.restype = c_int
    lib.t2va_objective_plan_query.argtypes = [c_int, c_int, seg, c_int, c_int, ctypes.POINTER(ObjectivePlan)]
    lib.t2va_objective_plan_query.restype = c_int


def load(path: Optional[str] = None):
    """The loaded libt2va.so (raises if it has not been built)."""
    global _LIB
    if _LIB is None:
        p = path or LIB
        if not os.path.exists(p):
            raise RuntimeError(f"libt2va.so not found at {p}: build it with "
                               f"`python -m joint_video_audio_02_b300.build`")
        lib = ctypes.CDLL(p)
        _declare(lib)
        _LIB = lib
    return _LIB


def error_string(code: int) -> str:
    return load().t2va_error_string(int(code)).decode()


def _check(code: int, where: str):
    if code != 0:
        raise T2VAError(code, where)


def _stream(stream) -> int:
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, torch.cuda.Stream):
        return stream.cuda_stream
    return int(stream)


def _dtype_code(dt: torch.dtype) -> int:
    if dt == torch.bfloat16:
        return T2VA_BFLOAT16
    if dt == torch.float32:
        return T2VA_FLOAT32
    raise TypeError(f"unsupported latent dtype {dt}")


def _segments(groups: Sequence[Sequence[torch.Tensor]], batch: int):
    """Geometry per modality, checked to be shared by every tensor of that modality."""
    M = len(groups[0])
    segs = (Segment * M)()
    for m in range(M):
        ref = groups[0][m]
        for grp in groups:
            x = grp[m]
            if not x.is_cuda:
                raise ValueError("every latent must be a CUDA tensor")
            if x.shape[0] != batch:
                raise ValueError("first dimension must be the batch")
            if batch > 0 and x.dim() > 1 and not x[0].is_contiguous():
                raise ValueError("each sample's elements must be contiguous")
            empty = x.numel() == 0
            if x.shape[1:] != ref.shape[1:] or (batch > 1 and not empty and x.stride(0) != ref.stride(0)):
                raise ValueError("all tensors of one modality must share shape and sample stride")
        n = 1
        for d in ref.shape[1:]:
            n *= int(d)
        segs[m].numel = n
        segs[m].sample_stride = int(ref.stride(0)) if (batch > 1 and n > 0) else n
    return segs


def _ptrs(ts: Sequence[torch.Tensor]):
    return (c_void_p * len(ts))(*[t.data_ptr() for t in ts])


def _opt(t: Optional[torch.Tensor]):
    return None if t is None else t.data_ptr()


def _f32(t: torch.Tensor, name: str):
    if t.dtype != torch.float32 or not t.is_cuda:
        raise TypeError(f"{name} must be a float32 CUDA tensor")


def objective_plan(batch: int, numels: Sequence[int], dtype: str, sm_count: int,
                   sample_strides: Optional[Sequence[int]] = None) -> dict:
    """The launch plan of an objective call with these sizes (t2va_objective_plan_query):
    host arithmetic only, no device needed. `dtype` is "bf16" or "f32"; strides default
    to the numels (contiguous samples)."""
    M = len(numels)
    strides = list(numels) if sample_strides is None else list(sample_strides)
    segs = (Segment * M)()
    for m in range(M):
        segs[m].numel, segs[m].sample_stride = int(numels[m]), int(strides[m])
    code = {"bf16": T2VA_BFLOAT16, "f32": T2VA_FLOAT32}.get(dtype, -1)
    out = ObjectivePlan()
    _check(load().t2va_objective_plan_query(int(batch), M, segs, code, int(sm_count), ctypes.byref(out)),
           "t2va_objective_plan_query")
    return {"grid": out.grid, "threads": out.threads, "vectors_per_chunk": out.vectors_per_chunk,
            "chunks": [out.chunks[m] for m in range(M)], "outputs_modality": out.outputs_modality,
            "outputs_chunk": out.outputs_chunk, "one_wave": bool(out.one_wave)}


def workspace_bytes(batch: int, num_modalities: int) -> int:
    n = load().t2va_workspace_bytes(int(batch), int(num_modalities))
    if n == 0:
        raise T2VAError(1, "t2va_workspace_bytes")
    return int(n)


def workspace_init(workspace: torch.Tensor, timeout_ms: int = 1000, stream=None):
    _check(load().t2va_workspace_init(workspace.data_ptr(), workspace.numel() * workspace.element_size(),
                                      int(timeout_ms), _stream(stream)), "t2va_workspace_init")


def new_workspace(batch: int, num_modalities: int, device=None, timeout_ms: int = 1000, stream=None):
    """Allocate (through torch) and initialise a workspace for the objective calls."""
    ws = torch.empty(workspace_bytes(batch, num_modalities), dtype=torch.uint8,
                     device=device or torch.device("cuda"))
    workspace_init(ws, timeout_ms, stream)
    return ws


def noise(z0: Sequence[torch.Tensor], eps: Sequence[torch.Tensor], zt: Sequence[torch.Tensor],
          t: torch.Tensor, status: Optional[torch.Tensor] = None, stream=None):
    """z_t = cos(t) z0 + sin(t) eps per modality, into `zt` (t2va_noise)."""
    B, M = int(t.shape[0]), len(z0)
    segs = _segments([z0, eps, zt], B)
    dt = _dtype_code(z0[0].dtype)
    _f32(t, "t")
    _check(load().t2va_noise(B, M, segs, dt, _ptrs(z0), _ptrs(eps), _ptrs(zt), t.data_ptr(),
                             _opt(status), _stream(stream)), "t2va_noise")


def noise_rf(z0: Sequence[torch.Tensor], eps: Sequence[torch.Tensor],
             zt: Optional[Sequence[torch.Tensor]], z_rf: Sequence[torch.Tensor], t: torch.Tensor,
             t_rf: Optional[torch.Tensor] = None, status: Optional[torch.Tensor] = None,
             stream=None):
    """TrigFlow noising and its rectified-flow form in one pass (t2va_noise_rf): z_t
    into `zt` (may be None), z_t / (cos t + sin t) into `z_rf`, and
    sin t / (cos t + sin t) into `t_rf` (may be None)."""
    B, M = int(t.shape[0]), len(z0)
    groups = [z0, eps, z_rf] + ([zt] if zt is not None else [])
    segs = _segments(groups, B)
    dt = _dtype_code(z0[0].dtype)
    _f32(t, "t")
    if t_rf is not None:
        _f32(t_rf, "t_rf")
    _check(load().t2va_noise_rf(B, M, segs, dt, _ptrs(z0), _ptrs(eps),
                                _ptrs(zt) if zt is not None else None, _ptrs(z_rf), t.data_ptr(),
                                _opt(t_rf), _opt(status), _stream(stream)), "t2va_noise_rf")


def scm_objective(z_t, x0_teacher, x0_student, x0_student_tangent, t, *, beta, gamma, eps_scm,
                  weight, lambda_scm, grad_x0_student, loss, norm=None, accumulate=False,
                  workspace, status, stream=None):
    B, M = int(t.shape[0]), len(z_t)
    segs = _segments([z_t, x0_teacher, x0_student, x0_student_tangent, grad_x0_student], B)
    dt = _dtype_code(z_t[0].dtype)
    for g in grad_x0_student:
        _f32(g, "grad_x0_student")
    w = (c_float * M)(*[float(x) for x in weight])
    _check(load().t2va_scm_objective(
        B, M, segs, dt, _ptrs(z_t), _ptrs(x0_teacher), _ptrs(x0_student), _ptrs(x0_student_tangent),
        t.data_ptr(), float(beta), float(gamma), float(eps_scm), w, float(lambda_scm),
        _ptrs(grad_x0_student), int(bool(accumulate)), loss.data_ptr(), _opt(norm),
        workspace.data_ptr(), workspace.numel() * workspace.element_size(), status.data_ptr(),
        _stream(stream)), "t2va_scm_objective")


def dmd_objective(zhat0, x0_teacher_hat, x0_fake, *, eps_dmd, weight, lambda_dmd, grad_zhat0, loss,
                  cdmd=None, accumulate=False, workspace, status, stream=None):
    B, M = int(zhat0[0].shape[0]), len(zhat0)
    segs = _segments([zhat0, x0_teacher_hat, x0_fake, grad_zhat0], B)
    dt = _dtype_code(zhat0[0].dtype)
    for g in grad_zhat0:
        _f32(g, "grad_zhat0")
    w = (c_float * M)(*[float(x) for x in weight])
    _check(load().t2va_dmd_objective(
        B, M, segs, dt, _ptrs(zhat0), _ptrs(x0_teacher_hat), _ptrs(x0_fake), float(eps_dmd), w,
        float(lambda_dmd), _ptrs(grad_zhat0), int(bool(accumulate)), loss.data_ptr(), _opt(cdmd),
        workspace.data_ptr(), workspace.numel() * workspace.element_size(), status.data_ptr(),
        _stream(stream)), "t2va_dmd_objective")


def stage3_objective(z_t, x0_teacher, x0_student, x0_student_tangent, t, zhat0, x0_teacher_hat,
                     x0_fake, *, beta, gamma, eps_scm, eps_dmd, weight, lambda_scm, lambda_dmd,
                     grad_x0_student, grad_zhat0, loss, loss_scm=None, loss_dmd=None, norm=None,
                     cdmd=None, accumulate=False, workspace, status, stream=None):
    B, M = int(t.shape[0]), len(z_t)
    segs = _segments([z_t, x0_teacher, x0_student, x0_student_tangent, zhat0, x0_teacher_hat,
                      x0_fake, grad_x0_student, grad_zhat0], B)
    dt = _dtype_code(z_t[0].dtype)
    for g in list(grad_x0_student) + list(grad_zhat0):
        _f32(g, "gradient")
    w = (c_float * M)(*[float(x) for x in weight])
    _check(load().t2va_stage3_objective(
        B, M, segs, dt, _ptrs(z_t), _ptrs(x0_teacher), _ptrs(x0_student), _ptrs(x0_student_tangent),
        t.data_ptr(), _ptrs(zhat0), _ptrs(x0_teacher_hat), _ptrs(x0_fake),
        float(beta), float(gamma), float(eps_scm), float(eps_dmd), w, float(lambda_scm),
        float(lambda_dmd), _ptrs(grad_x0_student), _ptrs(grad_zhat0), int(bool(accumulate)),
        loss.data_ptr(), _opt(loss_scm), _opt(loss_dmd), _opt(norm), _opt(cdmd),
        workspace.data_ptr(), workspace.numel() * workspace.element_size(), status.data_ptr(),
        _stream(stream)), "t2va_stage3_objective")


def stage3_objective_cfg(z_t, x0_teacher, x0_student, x0_student_tangent, t, zhat0,
                         x0_teacher_hat_cond, x0_teacher_hat_uncond, x0_fake, *, guidance, beta,
                         gamma, eps_scm, eps_dmd, weight, lambda_scm, lambda_dmd, grad_x0_student,
                         grad_zhat0, loss, loss_scm=None, loss_dmd=None, norm=None, cdmd=None,
                         accumulate=False, workspace, status, stream=None):
    """stage3_objective with the DMD teacher prediction guided per modality:
    u + guidance[m] (k - u) from the conditional (k) and unconditional (u) predictions
    (t2va_stage3_objective_cfg)."""
    B, M = int(t.shape[0]), len(z_t)
    segs = _segments([z_t, x0_teacher, x0_student, x0_student_tangent, zhat0, x0_teacher_hat_cond,
                      x0_teacher_hat_uncond, x0_fake, grad_x0_student, grad_zhat0], B)
    dt = _dtype_code(z_t[0].dtype)
    for g in list(grad_x0_student) + list(grad_zhat0):
        _f32(g, "gradient")
    w = (c_float * M)(*[float(x) for x in weight])
    gs = (c_float * M)(*[float(x) for x in guidance])
    _check(load().t2va_stage3_objective_cfg(
        B, M, segs, dt, _ptrs(z_t), _ptrs(x0_teacher), _ptrs(x0_student), _ptrs(x0_student_tangent),
        t.data_ptr(), _ptrs(zhat0), _ptrs(x0_teacher_hat_cond), _ptrs(x0_teacher_hat_uncond), gs,
        _ptrs(x0_fake), float(beta), float(gamma), float(eps_scm), float(eps_dmd), w,
        float(lambda_scm), float(lambda_dmd), _ptrs(grad_x0_student), _ptrs(grad_zhat0),
        int(bool(accumulate)), loss.data_ptr(), _opt(loss_scm), _opt(loss_dmd), _opt(norm),
        _opt(cdmd), workspace.data_ptr(), workspace.numel() * workspace.element_size(),
        status.data_ptr(), _stream(stream)), "t2va_stage3_objective_cfg")


W8A8_EPS = 1e-4


def _code_dtype(dt: torch.dtype) -> int:
    if dt == torch.int8:
        return T2VA_INT8
    if dt == torch.bfloat16:
        return T2VA_BFLOAT16
    raise TypeError("codes are int8, or bfloat16 for the tensor-core contraction")


def quantize_rows(x: torch.Tensor, q: torch.Tensor, scale: torch.Tensor, eps: float = W8A8_EPS,
                  stream=None):
    """Per-row dynamic quantisation of a 2-D CUDA tensor (t2va_quantize_rows): codes into
    `q` (int8, or bfloat16 holding the same integers; same shape, rows 16-byte aligned)
    and scales into `scale` (float32)."""
    if x.dim() != 2 or q.dim() != 2 or q.shape != x.shape:
        raise ValueError("x and q must be 2-D of one shape")
    if x.stride(1) != 1 or q.stride(1) != 1:
        raise ValueError("rows must be contiguous")
    _f32(scale, "scale")
    _check(load().t2va_quantize_rows(int(x.shape[0]), int(x.shape[1]), _dtype_code(x.dtype), x.data_ptr(),
                                     int(x.stride(0)), float(eps), _code_dtype(q.dtype), q.data_ptr(),
                                     int(q.stride(0)), scale.data_ptr(), _stream(stream)), "t2va_quantize_rows")


def w8a8_linear(xq: torch.Tensor, sx: torch.Tensor, wq: torch.Tensor, sw: torch.Tensor,
                y: torch.Tensor, bias: Optional[torch.Tensor] = None, status: Optional[torch.Tensor] = None,
                stream=None):
    """y = sx sw (xq . wq^T) + bias with an exact integer sum (t2va_w8a8_linear). xq [M, K]
    and wq [N, K] are codes (int8: warp-level INT8 MMA; bfloat16 integers: tcgen05 tensor
    cores), contiguous; y [M, N] bfloat16 or float32, contiguous."""
    M, K = int(xq.shape[0]), int(xq.shape[1])
    N = int(wq.shape[0])
    if wq.shape[1] != K or tuple(y.shape) != (M, N):
        raise ValueError("shapes do not match")
    for t in (xq, wq, y):
        if not t.is_contiguous():
            raise ValueError("xq, wq and y must be contiguous")
    if xq.dtype != wq.dtype:
        raise TypeError("xq and wq must have one code dtype")
    _f32(sx, "sx")
    _f32(sw, "sw")
    if bias is not None:
        _f32(bias, "bias")
    _check(load().t2va_w8a8_linear(M, N, K, _code_dtype(xq.dtype), xq.data_ptr(), sx.data_ptr(), wq.data_ptr(),
                                   sw.data_ptr(), _opt(bias), _dtype_code(y.dtype), y.data_ptr(), _opt(status),
                                   _stream(stream)), "t2va_w8a8_linear")


def residual_modnorm(h: torch.Tensor, y: torch.Tensor, *, u: Optional[torch.Tensor] = None,
                     gate: Optional[torch.Tensor] = None, scale: Optional[torch.Tensor] = None,
                     shift: Optional[torch.Tensor] = None, eps: float = 1e-6,
                     h_out: Optional[torch.Tensor] = None, rows_per_sample: Optional[int] = None,
                     stream=None):
    """Fused gated residual + modulated RMS normalisation (t2va_residual_modnorm) over token
    rows: h [rows, D] (and u, h_out, y of that shape, contiguous, one dtype); gate, scale,
    shift float32 [samples, D]; row r belongs to sample r // rows_per_sample (default: all
    rows one sample)."""
    rows, D = int(h.shape[0]), int(h.shape[1])
    for t in [h, y] + [x for x in (u, h_out) if x is not None]:
        if tuple(t.shape) != (rows, D) or not t.is_contiguous() or t.dtype != h.dtype:
            raise ValueError("h, u, h_out and y must be contiguous [rows, D] of one dtype")
    for name, v in (("gate", gate), ("scale", scale), ("shift", shift)):
        if v is not None:
            _f32(v, name)
    rps = rows if rows_per_sample is None else int(rows_per_sample)
    _check(load().t2va_residual_modnorm(rows, D, max(1, rps), _dtype_code(h.dtype), h.data_ptr(), _opt(u),
                                        _opt(gate), _opt(scale), _opt(shift), float(eps), _opt(h_out),
                                        y.data_ptr(), _stream(stream)), "t2va_residual_modnorm")


def selftest_wait_timeout(status: torch.Tensor, stream=None):
    """Launch the tensor-core W8A8 kernel's bounded-wait self-test (t2va_selftest_wait_timeout):
    after about a second `status` holds STATUS_TIMEOUT."""
    _check(load().t2va_selftest_wait_timeout(status.data_ptr(), _stream(stream)), "t2va_selftest_wait_timeout")


def stage3_objective_noalloc(z_t, x0_teacher, x0_student, x0_student_tangent, t, zhat0,
                             x0_teacher_hat, x0_fake, *, beta, gamma, eps_scm, eps_dmd, weight,
                             lambda_scm, lambda_dmd, grad_x0_student, grad_zhat0, loss,
                             loss_scm=None, loss_dmd=None, norm=None, cdmd=None, accumulate=False,
                             status, stream=None):
    """stage3_objective for callers that cannot allocate device memory: no workspace
    argument; the library's own static scratch array is used instead (one per GPU,
    shared by every call, so calls that overlap on the GPU race). The first call on a
    device looks up the array's address and should come before any stream capture."""
    B, M = int(t.shape[0]), len(z_t)
    segs = _segments([z_t, x0_teacher, x0_student, x0_student_tangent, zhat0, x0_teacher_hat,
                      x0_fake, grad_x0_student, grad_zhat0], B)
    dt = _dtype_code(z_t[0].dtype)
    for g in list(grad_x0_student) + list(grad_zhat0):
        _f32(g, "gradient")
    w = (c_float * M)(*[float(x) for x in weight])
    _check(load().t2va_stage3_objective_noalloc(
        B, M, segs, dt, _ptrs(z_t), _ptrs(x0_teacher), _ptrs(x0_student), _ptrs(x0_student_tangent),
        t.data_ptr(), _ptrs(zhat0), _ptrs(x0_teacher_hat), _ptrs(x0_fake),
        float(beta), float(gamma), float(eps_scm), float(eps_dmd), w, float(lambda_scm),
        float(lambda_dmd), _ptrs(grad_x0_student), _ptrs(grad_zhat0), int(bool(accumulate)),
        loss.data_ptr(), _opt(loss_scm), _opt(loss_dmd), _opt(norm), _opt(cdmd),
        status.data_ptr(), _stream(stream)), "t2va_stage3_objective_noalloc")
