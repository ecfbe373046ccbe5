"""The CUDA path, through the C ABI, against the hand-derived values of tests/golden/ (the
same fixtures that pin the oracle). Float32 storage throughout, so the only differences
are float32 rounding (and the float32 timestep): within 1e-6 relative, or exact where the
values are exact binary fractions (codes, scales, integer sums, the linear's outputs)."""

import numpy as np
import pytest
import torch

import joint_video_audio_02_b300 as t2va
from golden_util import ANGLES, load, num, scalar
from joint_video_audio_02_b300.build import build

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    build()
    t2va.load()


def _dev(a, dtype=torch.float32):
    return torch.from_numpy(np.ascontiguousarray(a)).to(dtype).cuda()


def test_golden_gpu_noise_rf():
    g = load("trigflow_noise_rf.txt")
    B = len(ANGLES)
    t = torch.tensor([np.pi / n for _, n in ANGLES], dtype=torch.float32, device="cuda")
    z0 = torch.full((B, 1), scalar(g["z0"]), device="cuda")
    ep = torch.full((B, 1), scalar(g["eps"]), device="cuda")
    zt, zrf, trf = torch.empty_like(z0), torch.empty_like(z0), torch.empty(B, device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    t2va.noise_rf([z0], [ep], [zt], [zrf], t, t_rf=trf, status=st)
    torch.cuda.synchronize()
    assert st.item() == 0
    for i, (key, _) in enumerate(ANGLES):
        # the float32 timestep is within 6e-8 of the angle; every output moves by at most
        # 2.3 times that, plus float32 rounding
        for got, name in ((zt[i, 0], "z_t"), (zrf[i, 0], "z_rf"), (trf[i], "t_rf")):
            ref = scalar(g[f"{key}.{name}"])
            assert abs(float(got) - ref) <= 3e-7 + 2e-7 * abs(ref), (key, name)


def test_golden_gpu_stage3_guided():
    """The matched-student sCM case and the guided DMD case in one guided stage-3 call
    (one sample, one modality of two elements, guidance 3.0, lambdas 1)."""
    s = load("scm_direction_closed_form.txt")
    c = load("cfg_guided_teacher.txt")
    row = lambda v: _dev(num(v)[None])
    t = torch.tensor([num(s["t"])], dtype=torch.float32, device="cuda")
    gS, gD = torch.empty((1, 2), device="cuda"), torch.empty((1, 2), device="cuda")
    loss, ls, ld = (torch.empty(1, device="cuda") for _ in range(3))
    norm, cdmd = torch.empty(1, device="cuda"), torch.empty(1, device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    x0 = row(s["x0"])
    t2va.stage3_objective_cfg([row(s["z_t"])], [x0], [x0.clone()], [row(s["tangent"])], t, [row(c["dmd.zhat0"])],
                              [row(c["dmd.cond"])], [row(c["dmd.uncond"])], [row(c["dmd.x0_fake"])],
                              guidance=[scalar(c["scale_video"])], beta=scalar(s["beta"]), gamma=scalar(s["gamma"]),
                              eps_scm=scalar(s["eps_scm"]), eps_dmd=scalar(c["dmd.eps_dmd"]), weight=[1.0],
                              lambda_scm=1.0, lambda_dmd=1.0, grad_x0_student=[gS], grad_zhat0=[gD], loss=loss,
                              loss_scm=ls, loss_dmd=ld, norm=norm, cdmd=cdmd, workspace=t2va.new_workspace(1, 1),
                              status=st)
    torch.cuda.synchronize()
    assert st.item() == 0
    close = lambda got, ref: np.testing.assert_allclose(np.asarray(got, np.float64), ref, rtol=1e-6, atol=1e-7)
    close(ls.item(), scalar(s["loss"]))
    close(norm.item(), scalar(s["norm"]))
    close(gS.cpu().numpy()[0], num(s["grad_x0_student"]))
    close(ld.item(), scalar(c["dmd.loss"]))
    close(cdmd.item(), scalar(c["dmd.cdmd"]))
    close(gD.cpu().numpy()[0], num(c["dmd.grad_zhat0"]))
    close(loss.item(), scalar(s["loss"]) + scalar(c["dmd.loss"]))


def test_golden_gpu_dmd_residual_scale():
    g = load("dmd_residual_scale.txt")
    row = lambda v: _dev(num(v)[None])
    gD, loss, cdmd = torch.empty((1, 4), device="cuda"), torch.empty(1, device="cuda"), torch.empty(1, device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    t2va.dmd_objective([row(g["zhat0"])], [row(g["x0_teacher_hat"])], [row(g["x0_fake"])], eps_dmd=scalar(g["eps_dmd"]),
                       weight=[1.0], lambda_dmd=1.0, grad_zhat0=[gD], loss=loss, cdmd=cdmd,
                       workspace=t2va.new_workspace(1, 1), status=st)
    torch.cuda.synchronize()
    assert st.item() == 0
    assert cdmd.item() == scalar(g["cdmd"])
    np.testing.assert_allclose(loss.item(), scalar(g["loss"]), rtol=1e-6)
    np.testing.assert_allclose(gD.cpu().numpy()[0], num(g["grad_zhat0"]), rtol=1e-6, atol=1e-7)


@pytest.mark.parametrize("code", [torch.int8, torch.bfloat16], ids=["int8", "bf16codes"])
def test_golden_gpu_quantise_rows(code):
    g = load("w8a8_quantise_and_linear.txt")
    for k in ("row1", "row2", "row3", "row4"):
        x = num(g[k])
        n = -(-len(x) // 4) * 4                     # float32 rows of whole 16-byte vectors
        xp = np.zeros((1, n), np.float32)
        xp[0, :len(x)] = x
        q = torch.empty((1, n), dtype=code, device="cuda")
        s = torch.empty(1, device="cuda")
        t2va.quantize_rows(_dev(xp), q, s)
        torch.cuda.synchronize()
        codes = q.float().cpu().numpy()[0, :len(x)].astype(np.int64)
        assert np.array_equal(codes, num(g[k + ".codes"]).astype(np.int64)), k
        assert s.item() == float(np.float32(scalar(g[k + ".scale"]))), k


@pytest.mark.parametrize("code", [torch.int8, torch.bfloat16], ids=["int8", "bf16codes"])
@pytest.mark.parametrize("N", [128, 256])
def test_golden_gpu_w8a8_linear(code, N):
    """The fixture's 2 x 3 x 4 linear in the corner of a 128 x N x 128 launch (zero codes
    elsewhere, unit scales): float32 outputs equal the fixture exactly, every other output
    its bias."""
    g = load("w8a8_quantise_and_linear.txt")
    M = K = 128
    xq, wq = np.zeros((M, K), np.int8), np.zeros((N, K), np.int8)
    xq[:2, :4], wq[:3, :4] = num(g["xq"]), num(g["wq"])
    sx, sw, b = np.ones(M, np.float32), np.ones(N, np.float32), np.zeros(N, np.float32)
    sx[:2], sw[:3], b[:3] = num(g["sx"]), num(g["sw"]), num(g["bias"])
    y = torch.empty((M, N), device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    t2va.w8a8_linear(torch.from_numpy(xq).cuda().to(code), _dev(sx), torch.from_numpy(wq).cuda().to(code), _dev(sw),
                     y, _dev(b), status=st)
    torch.cuda.synchronize()
    assert st.item() == 0
    want = np.broadcast_to(b, (M, N)).astype(np.float64).copy()
    want[:2, :3] = num(g["y"])
    assert np.array_equal(y.cpu().numpy().astype(np.float64), want)


def test_golden_gpu_residual_modnorm():
    g = load("residual_modnorm.txt")
    row = lambda k: _dev(num(g[k])[None])
    h = row("h")
    y, h_out = torch.empty_like(h), torch.empty_like(h)
    t2va.residual_modnorm(h, y, u=row("u"), gate=row("gate"), scale=row("scale"), shift=row("shift"),
                          eps=scalar(g["eps"]), h_out=h_out)
    torch.cuda.synchronize()
    assert np.array_equal(h_out.cpu().numpy()[0], num(g["h_new"]))
    np.testing.assert_allclose(y.cpu().numpy()[0], num(g["y"]), rtol=1e-6, atol=0)
