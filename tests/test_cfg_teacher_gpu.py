"""GPU parity of the stage-3 objective with a guided teacher
(t2va_stage3_objective_cfg) against the float64 oracle, with the tolerances of the
plain stage-3 objective: the guided prediction u + s (k - u) is one float32 fma per
element, within 1 ulp of |u| + s |k - u|, far inside them."""

import numpy as np
import pytest
import torch

import joint_video_audio_02_b300 as t2va
import synthetic as S
from joint_video_audio_02_b300.build import build
from t2va_gpu_util import Params, compare, gpu_run, oracle_run, to_device, grads_like

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    build()
    t2va.load()


@pytest.mark.parametrize("name", ["stage3_cfg_512x768_bf16", "stage3_cfg_1024x1792_bf16"])
def test_stage3_cfg_parity(name):
    wl = S.workload(name)
    inp = S.make_workload_inputs(wl)
    p = Params.of(wl)
    gpu = gpu_run(inp, p, S.STAGE3_CFG)
    assert gpu["status"] == 0
    compare(gpu, oracle_run(inp, p, S.STAGE3_CFG), wl.dtype, S.STAGE3_CFG)


RAGGED = [(3, [1, 7], 0), (2, [9, 8191], 3), (5, [100003, 5], 1), (2, [0, 77], 0),
          (2, [33, 64, 1, 250001], 7)]


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
@pytest.mark.parametrize("case", RAGGED, ids=[f"B{b}-{'-'.join(map(str, n))}-p{p}" for b, n, p in RAGGED])
def test_stage3_cfg_ragged(dtype, case):
    B, numels, pad = case
    inp = S.make_inputs(B, numels, dtype, S.STAGE3_CFG, seed=(600, B, len(numels), pad))
    M = len(numels)
    p = Params(weight=tuple(1.0 + 0.5 * m for m in range(M)), gamma=0.7, beta=1.2,
               guidance=tuple(3.0 + 2.0 * m - 0.25 * m * m for m in range(M)))
    gpu = gpu_run(inp, p, S.STAGE3_CFG, stride_pad=pad)
    assert gpu["status"] == 0
    compare(gpu, oracle_run(inp, p, S.STAGE3_CFG), dtype, S.STAGE3_CFG)


def test_cfg_equal_predictions_match_plain_stage3_bitwise():
    """With the conditional and unconditional predictions equal, u + s (k - u) = k
    exactly in float32 for every scale, so the guided call reproduces the plain
    stage-3 call bit for bit."""
    inp = S.make_inputs(3, [50_003, 701], "bf16", S.STAGE3_CFG, seed=(601,))
    inp.x0_teacher_hat_uncond = [a.copy() for a in inp.x0_teacher_hat]
    p = Params(guidance=(3.0, 5.0))
    a = gpu_run(inp, p, S.STAGE3_CFG)
    b = gpu_run(inp, p, S.STAGE3)
    for k in ("loss", "loss_scm", "loss_dmd", "norm", "cdmd"):
        assert np.array_equal(a[k], b[k]), k
    for k in ("grad_x0_student", "grad_zhat0"):
        for x, y in zip(a[k], b[k]):
            assert np.array_equal(x, y), k


def test_cfg_bad_timestep_and_guidance_errors():
    inp = S.make_inputs(3, [5000, 300], "bf16", S.STAGE3_CFG, seed=(602,))
    t = np.array([0.5, 0.0, 1.2], dtype=np.float32)
    p = Params()
    gpu = gpu_run(inp, p, S.STAGE3_CFG, t_override=t)
    assert gpu["status"] & t2va.STATUS_BAD_TIMESTEP
    assert np.array_equal(np.isnan(gpu["loss"]), [False, True, False])
    compare(gpu, oracle_run(inp, p, S.STAGE3_CFG, t_override=t), "bf16", S.STAGE3_CFG)
    z = to_device(inp.z0, "bf16")
    tt = torch.from_numpy(inp.t).cuda()
    g = grads_like(z)
    loss = torch.zeros(3, device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    ws = t2va.new_workspace(3, 2)
    with pytest.raises(t2va.T2VAError) as e:
        t2va.stage3_objective_cfg(z, z, z, z, tt, z, z, z, z, guidance=(3.0, float("nan")), beta=1,
                                  gamma=0.5, eps_scm=1e-6, eps_dmd=1e-6, weight=(1, 1),
                                  lambda_scm=1, lambda_dmd=1, grad_x0_student=g, grad_zhat0=g,
                                  loss=loss, workspace=ws, status=st)
    assert e.value.code == 1


def test_cfg_accumulate_and_alias():
    """The guided objective accumulates into existing gradients, and sums both gradients
    into one buffer when grad_zhat0 is grad_x0_student, as the plain stage-3 call does."""
    inp = S.make_inputs(2, [20000, 333], "bf16", S.STAGE3_CFG, seed=(603,))
    p = Params(guidance=(2.0, 4.5))
    rng = np.random.default_rng(1)
    prior = {"grad_x0_student": [rng.normal(size=a.shape).astype(np.float32) for a in inp.z0],
             "grad_zhat0": [rng.normal(size=a.shape).astype(np.float32) for a in inp.z0]}
    gpu = gpu_run(inp, p, S.STAGE3_CFG, accumulate_into=prior)
    ref = oracle_run(inp, p, S.STAGE3_CFG)
    for k in ("grad_x0_student", "grad_zhat0"):
        ref[k] = [r + q.astype(np.float64) for r, q in zip(ref[k], prior[k])]
    compare(gpu, ref, "bf16", S.STAGE3_CFG)
    gpu = gpu_run(inp, p, S.STAGE3_CFG, alias=True)
    ref = oracle_run(inp, p, S.STAGE3_CFG)
    summed = [a + b for a, b in zip(ref["grad_x0_student"], ref["grad_zhat0"])]
    ref["grad_x0_student"] = summed
    ref["grad_zhat0"] = summed
    compare(gpu, ref, "bf16", S.STAGE3_CFG)
