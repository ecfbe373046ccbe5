"""The allocation-free stage-3 entry point against the regular one.

t2va_stage3_objective_noalloc serves callers that cannot allocate device memory
(code running inside another runtime's memory pool or under an allocator that owns
all device memory, plugins handed only their inputs and outputs, hosts that forbid
allocation after set-up): it takes no workspace and uses the library's static
scratch array instead. It runs the same kernels on the same plan as
t2va_stage3_objective, so its results must be bit-identical to that entry point's
on the same inputs, on two calls in a row (the second call finds the scratch as the
first one left it); one case is also checked against the float64 oracle.

This file is collected last, so a run that stops at the first failure has run
every other test before it. It must also pass alone in a fresh process.
"""

import numpy as np
import pytest
import torch

import joint_video_audio_02_b300 as t2va
import oracle
import synthetic as S
from joint_video_audio_02_b300.build import build
from t2va_gpu_util import Params, compare, grads_like, to_device

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    build()
    t2va.load()


def _run(inp, p, noalloc):
    dt = inp.dtype
    B, M = inp.batch, len(inp.z0)
    t = torch.from_numpy(inp.t).cuda()
    zt = to_device(inp.z0, dt)               # the objective's z_t input (noising is not under test)
    xT, xS, tan = (to_device(getattr(inp, f), dt) for f in ("x0_teacher", "x0_student", "x0_tangent"))
    zh, yT, yF = (to_device(getattr(inp, f), dt) for f in ("zhat0", "x0_teacher_hat", "x0_fake"))
    gS, gD = grads_like(zt, float("nan")), grads_like(zh, float("nan"))
    loss = torch.full((B,), float("nan"), device="cuda")
    loss_s = torch.full((B,), float("nan"), device="cuda")
    loss_d = torch.full((B,), float("nan"), device="cuda")
    norm = torch.full((B * M,), float("nan"), device="cuda")
    cdmd = torch.full((B * M,), float("nan"), device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    kw = dict(beta=p.beta, gamma=p.gamma, eps_scm=p.eps_scm, eps_dmd=p.eps_dmd, weight=p.weight,
              lambda_scm=p.lambda_scm, lambda_dmd=p.lambda_dmd, grad_x0_student=gS, grad_zhat0=gD,
              loss=loss, loss_scm=loss_s, loss_dmd=loss_d, norm=norm, cdmd=cdmd, status=status)
    if noalloc:
        t2va.stage3_objective_noalloc(zt, xT, xS, tan, t, zh, yT, yF, **kw)
    else:
        ws = t2va.new_workspace(B, M)
        t2va.stage3_objective(zt, xT, xS, tan, t, zh, yT, yF, workspace=ws, **kw)
    torch.cuda.synchronize()
    return {"status": int(status.item()), "loss": loss.cpu().numpy(), "loss_scm": loss_s.cpu().numpy(),
            "loss_dmd": loss_d.cpu().numpy(), "norm": norm.cpu().numpy(), "cdmd": cdmd.cpu().numpy(),
            "gS": [g.cpu().numpy() for g in gS], "gD": [g.cpu().numpy() for g in gD]}


def _same(got, ref):
    """Bit-identical outputs: both entry points run the same deterministic kernels."""
    assert got["status"] == 0 and ref["status"] == 0
    for k in ("loss", "loss_scm", "loss_dmd", "norm", "cdmd"):
        assert np.array_equal(got[k], ref[k]), k
    for kind in ("gS", "gD"):
        for g, r in zip(got[kind], ref[kind]):
            assert np.array_equal(g, r), kind


def test_noalloc_matches_stage3_on_two_calls_in_a_row():
    p = Params(weight=(1.0, 4.0))
    first = S.make_inputs(3, [50_003, 701], "bf16", S.STAGE3, seed=(900,))
    second = S.make_inputs(5, [20_011, 1_999], "bf16", S.STAGE3, seed=(901,))
    for inp in (first, second):
        _same(_run(inp, p, noalloc=True), _run(inp, p, noalloc=False))


def test_noalloc_float32_and_at_its_batch_limit():
    """float32 inputs, then the largest batch the scratch holds for two modalities."""
    p = Params(weight=(1.0, 2.0))
    f32 = S.make_inputs(2, [4_099, 130], "f32", S.STAGE3, seed=(903,))
    _same(_run(f32, p, noalloc=True), _run(f32, p, noalloc=False))
    big = 1
    while t2va.workspace_bytes(big + 1, 2) - 256 <= t2va.binding.NOALLOC_SCRATCH_BYTES:
        big += 1
    at_limit = S.make_inputs(big, [3_000, 200], "bf16", S.STAGE3, seed=(904,))
    _same(_run(at_limit, p, noalloc=True), _run(at_limit, p, noalloc=False))


def test_noalloc_against_the_oracle():
    p = Params(weight=(1.0, 4.0))
    inp = S.make_inputs(2, [20_000, 333], "bf16", S.STAGE3, seed=(905,))
    got = _run(inp, p, noalloc=True)
    # the objective's z_t here is the upload of z0 (the noising is not under test)
    ref = oracle.stage3_objective(inp.z0, inp.x0_teacher, inp.x0_student, inp.x0_tangent, inp.t,
                                  inp.zhat0, inp.x0_teacher_hat, inp.x0_fake, p.beta, p.gamma,
                                  p.eps_scm, p.eps_dmd, p.weight, p.lambda_scm, p.lambda_dmd, "bf16")
    assert got["status"] == 0
    compare({"loss": got["loss"], "loss_scm": got["loss_scm"], "loss_dmd": got["loss_dmd"],
             "norm": got["norm"].reshape(inp.batch, 2), "cdmd": got["cdmd"].reshape(inp.batch, 2),
             "grad_x0_student": got["gS"], "grad_zhat0": got["gD"]}, ref, "bf16", S.STAGE3)


def test_noalloc_argument_errors_match_the_regular_entry_point():
    """Every argument check runs before the scratch is used, with the codes of
    t2va_stage3_objective."""
    inp = S.make_inputs(2, [64, 16], "bf16", S.STAGE3, seed=(906,))
    z = to_device(inp.z0, "bf16")
    g = grads_like(z)
    t = torch.from_numpy(inp.t).cuda()
    loss = torch.zeros(2, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    ws = t2va.new_workspace(2, 2)
    good = dict(beta=1, gamma=0.9, eps_scm=1e-6, eps_dmd=1e-6, weight=[1, 1], lambda_scm=1,
                lambda_dmd=0.25, grad_x0_student=g, grad_zhat0=g, loss=loss, status=status)
    flat = torch.zeros(2 * 64 + 8, dtype=torch.bfloat16, device="cuda")
    mis = [flat[1:129].view(2, 64), z[1]]
    bad = [("gamma", dict(good, gamma=1.5), z), ("eps_dmd", dict(good, eps_dmd=0.0), z),
           ("weight", dict(good, weight=[1, -1]), z), ("misaligned", good, mis)]
    for what, kw, zz in bad:
        codes = []
        for fn in (lambda: t2va.stage3_objective(zz, z, z, z, t, z, z, z, workspace=ws, **kw),
                   lambda: t2va.stage3_objective_noalloc(zz, z, z, z, t, z, z, z, **kw)):
            with pytest.raises(t2va.T2VAError) as e:
                fn()
            codes.append(e.value.code)
        assert codes[0] == codes[1] != 0, (what, codes)
    torch.cuda.synchronize()
    assert status.item() == 0


def test_noalloc_rejects_a_batch_beyond_its_scratch():
    inp = S.make_inputs(1, [64, 16], "bf16", S.STAGE3, seed=(902,))
    big = 1
    while t2va.workspace_bytes(big, 2) - 256 <= t2va.binding.NOALLOC_SCRATCH_BYTES:
        big *= 2
    z = [torch.zeros((big, 64), dtype=torch.bfloat16, device="cuda"),
         torch.zeros((big, 16), dtype=torch.bfloat16, device="cuda")]
    g = grads_like(z)
    t = torch.full((big,), 0.5, device="cuda")
    loss = torch.zeros(big, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    with pytest.raises(t2va.T2VAError) as e:
        t2va.stage3_objective_noalloc(z, z, z, z, t, z, z, z, beta=1, gamma=0.9, eps_scm=1e-6,
                                      eps_dmd=1e-6, weight=[1, 1], lambda_scm=1, lambda_dmd=0.25,
                                      grad_x0_student=g, grad_zhat0=g, loss=loss, status=status)
    assert e.value.code == 4
    torch.cuda.synchronize()
    assert status.item() == 0
    del inp
