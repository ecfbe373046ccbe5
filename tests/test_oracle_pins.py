"""Pins for the float64 CPU oracle, each against something other than the oracle.

* J against central finite differences and against torch.func.jvp of F_theta on
  small joint students whose video and audio outputs depend on both modalities;
* the whole sCM direction against an exact symbolic derivation (sympy) at special
  angles, with J obtained by symbolic differentiation;
* closed forms: zero student error and zero tangent give g = (1-gamma) cos t sin t z_t;
  gamma = beta = 1 gives g = sin t (x0_S - x0_T) + cos t tangent; constant directions
  give known norms; the DMD term with constant offsets has a closed form;
* the gradients against autograd of the losses as printed (sg = detach);
* reductions against numpy library routines;
* bfloat16 rounding against torch's float32 -> bfloat16 conversion and hand ties.

Every pin is a function of the oracle module, so test_pins_catch_planted_mistakes
can run them on copies of the oracle with one mistake planted in each.
"""

import importlib.util
import math
import os

import numpy as np
import pytest
import sympy as sp
import torch

import oracle as ORACLE

ORACLE_FILE = os.path.join(os.path.dirname(ORACLE.__file__), "t2va_oracle.py")


def _rng(seed):
    return np.random.default_rng(seed)


def _close(a, b, rtol, atol=0.0):
    a = np.asarray(a, dtype=np.float64)
    b = np.asarray(b, dtype=np.float64)
    assert a.shape == b.shape, (a.shape, b.shape)
    err = np.abs(a - b)
    lim = atol + rtol * np.abs(b)
    assert np.all(err <= lim), f"max err {err.max():.3e}, worst rel {np.max(err / (np.abs(b) + 1e-300)):.3e}"


# ---------------------------------------------------------------------------
# a small joint student: x0^m = tanh-free linear map of both modalities + t terms
# ---------------------------------------------------------------------------

NV, NA = 5, 3


def _linear_student(seed):
    r = _rng(seed)
    A = r.normal(0, 0.4, size=(NV + NA, NV + NA))     # couples video and audio
    b0 = r.normal(0, 0.3, size=NV + NA)
    b1 = r.normal(0, 0.3, size=NV + NA)

    def x0(z, t):          # z: [N], t: scalar
        return A @ z + b0 + b1 * t

    def tangent(F_T):      # d x0 along (dt, dz) = (1, F_T)
        return A @ F_T + b1

    return x0, tangent


def _field(z, x0, t):
    return (math.cos(t) * z - x0) / math.sin(t)


def pin_jvp_finite_difference(orc):
    """J = c_t d/dh F_theta(z + h F_T, t + h) at h = 0, by central differences."""
    x0_fn, tan_fn = _linear_student(1)
    r = _rng(2)
    for t in (0.3, 0.9, 1.4):
        z = r.normal(size=NV + NA)
        x_T = z * 0.8 + r.normal(0, 0.1, size=NV + NA)
        F_T = _field(z, x_T, t)
        h = 1e-5
        Fp = _field(z + h * F_T, x0_fn(z + h * F_T, t + h), t + h)
        Fm = _field(z - h * F_T, x0_fn(z - h * F_T, t - h), t - h)
        J_fd = math.cos(t) * math.sin(t) * (Fp - Fm) / (2 * h)
        tt = np.array([t])
        tangent = tan_fn(F_T)
        for sl in (slice(0, NV), slice(NV, NV + NA)):     # video block, audio block
            zt = z[None, sl]
            F_theta = orc.trigflow_field(zt, x0_fn(z, t)[None, sl], tt)
            F_teach = orc.trigflow_field(zt, x_T[None, sl], tt)
            J = orc.joint_jvp(zt, F_theta, F_teach, tangent[None, sl], tt)
            _close(J[0], J_fd[sl], rtol=1e-7, atol=1e-9)


def pin_jvp_autodiff(orc):
    """J against torch.func.jvp of F_theta for a nonlinear cross-modal student."""
    g = torch.Generator().manual_seed(3)
    n = NV + NA
    A = torch.randn(n, n, generator=g, dtype=torch.float64) * 0.5
    bt = torch.randn(n, generator=g, dtype=torch.float64)

    def x0(z, t):
        return torch.tanh(A @ z + bt * t) + 0.1 * z

    def F(z, t):
        return (torch.cos(t) * z - x0(z, t)) / torch.sin(t)

    for tv in (0.05, 0.7, 1.5):
        t = torch.tensor(tv, dtype=torch.float64)
        z = torch.randn(n, generator=g, dtype=torch.float64)
        x_T = 0.9 * z + 0.1 * torch.randn(n, generator=g, dtype=torch.float64)
        F_T = (torch.cos(t) * z - x_T) / torch.sin(t)
        one = torch.ones((), dtype=torch.float64)
        _, tangent = torch.func.jvp(x0, (z, t), (F_T, one))
        _, dF = torch.func.jvp(F, (z, t), (F_T, one))
        J_ref = (torch.cos(t) * torch.sin(t) * dF).numpy()
        tt = np.array([tv], dtype=np.float64)
        zn, xs, xtn, tg = z.numpy(), x0(z, t).numpy(), x_T.numpy(), tangent.numpy()
        for sl in (slice(0, NV), slice(NV, n)):
            F_theta = orc.trigflow_field(zn[None, sl], xs[None, sl], tt)
            F_teach = orc.trigflow_field(zn[None, sl], xtn[None, sl], tt)
            J = orc.joint_jvp(zn[None, sl], F_theta, F_teach, tg[None, sl], tt)
            _close(J[0], J_ref[sl], rtol=1e-10, atol=1e-12)


def pin_direction_symbolic(orc):
    """g at t in {pi/6, pi/3}: exact sympy derivation of the printed direction, with J by
    symbolic differentiation of a linear cross-modal student."""
    tt, zv, za = sp.symbols("t z_v z_a")
    a = [[sp.Rational(1, 3), sp.Rational(-1, 4)], [sp.Rational(1, 5), sp.Rational(1, 2)]]
    b = [sp.Rational(2, 7), sp.Rational(-3, 5)]
    d = [sp.Rational(1, 9), sp.Rational(1, 11)]
    zs = [zv, za]
    x0 = [a[m][0] * zv + a[m][1] * za + b[m] * tt + d[m] for m in range(2)]
    xT = [sp.Rational(3, 4), sp.Rational(-1, 2)]
    F_T = [(sp.cos(tt) * zs[m] - xT[m]) / sp.sin(tt) for m in range(2)]
    F_S = [(sp.cos(tt) * zs[m] - x0[m]) / sp.sin(tt) for m in range(2)]
    for beta, gamma, tval in ((sp.Rational(7, 10), sp.Rational(3, 5), sp.pi / 3),
                              (sp.Integer(1), sp.Rational(9, 10), sp.pi / 6),
                              (sp.Rational(13, 10), sp.Integer(0), sp.pi / 3)):
        point = {tt: tval, zv: sp.Rational(6, 5), za: sp.Rational(-2, 3)}
        FTv = [F_T[m].subs(point) for m in range(2)]
        for m in range(2):
            ct = sp.cos(tt) * sp.sin(tt)
            J = ct * (sp.diff(F_S[m], tt) + sp.diff(F_S[m], zv) * F_T[0] + sp.diff(F_S[m], za) * F_T[1])
            g = (-beta * sp.cos(tt) / sp.sqrt(1 - gamma ** 2 * sp.sin(tt) ** 2) * (F_S[m] - F_T[m])
                 - gamma * sp.cos(tt) * sp.sin(tt) * zs[m] - J)
            exact = float(sp.N(g.subs(point), 30))
            tangent = float(sp.N(a[m][0] * FTv[0] + a[m][1] * FTv[1] + b[m], 30))
            tf = np.array([float(sp.N(tval, 30))])
            zt = np.array([[float(point[zs[m]])]])
            x_S = np.array([[float(sp.N(x0[m].subs(point), 30))]])
            x_Tn = np.array([[float(xT[m])]])
            got, _, _ = orc.scm_direction(zt, x_Tn, x_S, np.array([[tangent]]), tf,
                                          float(beta), float(gamma))
            _close(got[0, 0], exact, rtol=1e-12, atol=1e-14)


def pin_direction_closed_forms(orc):
    """x0_S = x0_T with zero tangent: g = (1 - gamma) cos t sin t z_t (the analytic
    dF/dt along the teacher flow is -z_t). gamma = beta = 1: g = sin t (x0_S - x0_T) +
    cos t tangent."""
    r = _rng(5)
    B, N = 3, 64
    t = np.array([0.01, 0.8, 1.55])
    z = r.normal(size=(B, N))
    xT = r.normal(size=(B, N))
    xS = xT + r.normal(0, 0.05, size=(B, N))
    tan = r.normal(0, 0.5, size=(B, N))
    c, s = np.cos(t)[:, None], np.sin(t)[:, None]
    for gamma in (0.0, 0.5, 0.9, 1.0):
        g, _, _ = orc.scm_direction(z, xT, xT.copy(), np.zeros((B, N)), t, 0.8, gamma)
        _close(g, (1 - gamma) * c * s * z, rtol=1e-11, atol=1e-13)
    g, _, _ = orc.scm_direction(z, xT, xS, tan, t, 1.0, 1.0)
    _close(g, s * (xS - xT) + c * tan, rtol=1e-9, atol=1e-11)


def _scm_inputs(seed, B=3, numels=(40, 12)):
    r = _rng(seed)
    t = np.array([0.2, 0.9, 1.3][:B])
    z = [r.normal(size=(B, n)) for n in numels]
    xT = [zz * 0.9 + r.normal(0, 0.1, size=zz.shape) for zz in z]
    xS = [x + r.normal(0, 0.05, size=x.shape) for x in xT]
    tan = [r.normal(0, 0.5, size=zz.shape) for zz in z]
    return z, xT, xS, tan, t


def pin_norm_and_loss(orc):
    """||g|| against numpy.linalg.norm; ||g_bar|| < 1; L_sCM = sum_m w_m n^2/(n+eps)^2;
    a constant direction (1-gamma) c s a over N elements has norm |(1-gamma) c s a| sqrt(N)."""
    z, xT, xS, tan, t = _scm_inputs(7)
    w, eps, lam = (1.0, 3.0), 1e-3, 0.7
    out = orc.scm_objective(z, xT, xS, tan, t, 1.0, 0.9, eps, w, lam)
    expect = np.zeros(len(t))
    for m in range(2):
        n_ref = np.linalg.norm(out["g"][m], axis=1)
        _close(out["norm"][:, m], n_ref, rtol=1e-13)
        expect += w[m] * n_ref ** 2 / (n_ref + eps) ** 2
        assert np.all(n_ref / (n_ref + eps) < 1.0)
    _close(out["loss"], lam * expect, rtol=1e-12)
    # constant direction
    B, N, a, gamma = 2, 1000, 0.37, 0.6
    tt = np.array([0.4, 1.2])
    zc = [np.full((B, N), a)]
    x = [np.ones((B, N))]
    o2 = orc.scm_objective(zc, x, [x[0].copy()], [np.zeros((B, N))], tt, 1.0, gamma, 1e-6, (1.0,), 1.0)
    _close(o2["norm"][:, 0], np.abs((1 - gamma) * np.cos(tt) * np.sin(tt) * a) * math.sqrt(N), rtol=1e-12)


def pin_zero_direction(orc):
    """gamma = 1, x0_S = x0_T, zero tangent: g = 0, so norm, loss and gradient are 0."""
    r = _rng(11)
    B, N = 2, 50
    z = [r.normal(size=(B, N))]
    x = [r.normal(size=(B, N))]
    out = orc.scm_objective(z, x, [x[0].copy()], [np.zeros((B, N))], np.array([0.5, 1.0]),
                            1.0, 1.0, 1e-6, (2.0,), 1.0)
    # the literal float64 evaluation leaves rounding residue of order 1e-16 in g
    assert np.all(out["norm"] < 1e-13)
    assert np.all(out["loss"] < 1e-12)
    assert np.all(np.abs(out["grad_x0_student"][0]) < 1e-6)


def pin_scm_gradient_autograd(orc):
    """dL/dx0_S from torch autograd of L = lam sum_m w_m ||F_theta - sg(F_theta) - sg(g_bar)||^2."""
    z, xT, xS, tan, t = _scm_inputs(13)
    w, eps, lam = (1.0, 2.5), 1e-6, 0.6
    out = orc.scm_objective(z, xT, xS, tan, t, 1.0, 0.5, eps, w, lam)
    tt = torch.tensor(t)[:, None]
    total = torch.zeros(len(t), dtype=torch.float64)
    leaves = []
    for m in range(2):
        xs = torch.tensor(xS[m], requires_grad=True)
        leaves.append(xs)
        F_theta = (torch.cos(tt) * torch.tensor(z[m]) - xs) / torch.sin(tt)
        g = torch.tensor(out["g"][m])
        g_bar = g / (torch.linalg.vector_norm(g, dim=1, keepdim=True) + eps)
        rres = F_theta - F_theta.detach() - g_bar.detach()
        total = total + w[m] * (rres * rres).sum(dim=1)
    L = lam * total
    L.sum().backward()
    _close(out["loss"], L.detach().numpy(), rtol=1e-12)
    for m in range(2):
        _close(out["grad_x0_student"][m], leaves[m].grad.numpy(), rtol=1e-10, atol=1e-14)


def _dmd_inputs(seed, B=3, numels=(40, 12)):
    r = _rng(seed)
    zh = [r.normal(size=(B, n)) for n in numels]
    yT = [x + r.normal(0, 0.1, size=x.shape) for x in zh]
    yF = [y + r.normal(0, 0.1, size=y.shape) for y in yT]
    return zh, yT, yF


def pin_dmd_closed_form(orc):
    """y_fake = y_T + k, y_T = zhat0 + delta: c = |delta|,
    L = lam w N k^2 / (|delta| + eps)^2, grad = 2 lam w k / (|delta| + eps)."""
    r = _rng(17)
    B, N, k, delta, w, eps, lam = 2, 300, 0.3, -0.2, 1.7, 1e-3, 0.25
    zh = [r.normal(size=(B, N))]
    yT = [zh[0] + delta]
    yF = [yT[0] + k]
    out = orc.dmd_objective(zh, yT, yF, eps, (w,), lam)
    _close(out["cdmd"][:, 0], np.full(B, abs(delta)), rtol=1e-12)
    _close(out["loss"], np.full(B, lam * w * N * k * k / (abs(delta) + eps) ** 2), rtol=1e-10)
    _close(out["grad_zhat0"][0], np.full((B, N), 2 * lam * w * k / (abs(delta) + eps)), rtol=1e-10)


def pin_dmd_autograd(orc):
    """c against numpy mean(abs); loss and grad against autograd of
    L = lam sum_m w_m sum_i (zhat0 - sg(zhat0 - g_bar))^2."""
    zh, yT, yF = _dmd_inputs(19)
    w, eps, lam = (1.0, 4.0), 1e-6, 0.25
    out = orc.dmd_objective(zh, yT, yF, eps, w, lam)
    total = torch.zeros(zh[0].shape[0], dtype=torch.float64)
    leaves = []
    for m in range(2):
        c = np.mean(np.abs(zh[m] - yT[m]), axis=1)
        _close(out["cdmd"][:, m], c, rtol=1e-13)
        x = torch.tensor(zh[m], requires_grad=True)
        leaves.append(x)
        g_bar = torch.tensor((yF[m] - yT[m]) / (c[:, None] + eps))
        delta = x - (x - g_bar).detach()
        total = total + w[m] * (delta * delta).sum(dim=1)
    L = lam * total
    L.sum().backward()
    _close(out["loss"], L.detach().numpy(), rtol=1e-12)
    for m in range(2):
        _close(out["grad_zhat0"][m], leaves[m].grad.numpy(), rtol=1e-10)


def pin_stage3_composition(orc):
    """L_stage3 = lam_s L_sCM + lam_d L_DMD on the same batch, gradients unchanged."""
    z, xT, xS, tan, t = _scm_inputs(23)
    zh, yT, yF = _dmd_inputs(29)
    w = (1.0, 4.0)
    s3 = orc.stage3_objective(z, xT, xS, tan, t, zh, yT, yF, 1.0, 0.9, 1e-6, 1e-6, w, 1.0, 0.25)
    a = orc.scm_objective(z, xT, xS, tan, t, 1.0, 0.9, 1e-6, w, 1.0)
    b = orc.dmd_objective(zh, yT, yF, 1e-6, w, 0.25)
    _close(s3["loss"], a["loss"] + b["loss"], rtol=1e-14)
    for m in range(2):
        _close(s3["grad_x0_student"][m], a["grad_x0_student"][m], rtol=0)
        _close(s3["grad_zhat0"][m], b["grad_zhat0"][m], rtol=0)


def pin_bf16_rounding(orc):
    """Single round-to-nearest-even to bfloat16: agrees with torch's float32 -> bfloat16
    conversion on float32 values, and on hand-made ties and near-ties."""
    r = _rng(31)
    x32 = np.concatenate([r.normal(size=20000), r.normal(size=2000) * 1e-30,
                          r.normal(size=2000) * 1e30, [0.0, -0.0, 1.0, -2.5]]).astype(np.float32)
    ref = torch.from_numpy(x32).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    got = orc.round_to_bf16_bits(x32.astype(np.float64))
    assert np.array_equal(got, ref)
    u = 2.0 ** -8
    cases = {1 + u: 0x3F80,                 # tie, round to even (down)
             1 + 3 * u: 0x3F82,             # tie, round to even (up)
             1 + u + 2.0 ** -40: 0x3F81,    # just above the tie: up (double rounding via float32 would go down)
             -(1 + u + 2.0 ** -40): 0xBF81}
    for v, bits in cases.items():
        assert int(orc.round_to_bf16_bits(np.array([v]))[0]) == bits, hex(bits)


def pin_noise(orc):
    """z_t = z0 at t -> 0 and z_t = eps at t = pi/2; the rotation preserves
    ||z_t||^2 + ||cos t eps - sin t z0||^2 = ||z0||^2 + ||eps||^2."""
    r = _rng(37)
    z0 = [r.normal(size=(2, 33))]
    eps = [r.normal(size=(2, 33))]
    out = orc.trigflow_noise(z0, eps, np.array([0.0, math.pi / 2]))[0]
    _close(out[0], z0[0][0], rtol=0, atol=0)
    _close(out[1], eps[0][1], rtol=0, atol=1e-15)
    t = np.array([0.3, 1.2])
    zt = orc.trigflow_noise(z0, eps, t)[0]
    other = np.cos(t)[:, None] * eps[0] - np.sin(t)[:, None] * z0[0]
    _close((zt ** 2).sum(1) + (other ** 2).sum(1), (z0[0] ** 2).sum(1) + (eps[0] ** 2).sum(1), rtol=1e-13)
    # stored path: bf16 in, one rounding out, against exact products of representable values
    zb = orc.round_to_bf16_bits(np.array([[1.0, 0.5, -3.0]]))
    eb = orc.round_to_bf16_bits(np.array([[0.0, 0.0, 0.0]]))
    got = orc.noise([zb], [eb], np.array([math.pi / 3]), "bf16")[0]
    assert np.array_equal(got, orc.round_to_bf16_bits(np.array([[0.5, 0.25, -1.5]]) * (2 * math.cos(math.pi / 3))))


def pin_domain(orc):
    """t outside (0, pi/2) gives NaN outputs for that sample only."""
    z, xT, xS, tan, _ = _scm_inputs(41)
    t = np.array([0.0, 0.7, math.pi / 2])
    out = orc.scm_objective(z, xT, xS, tan, t, 1.0, 0.9, 1e-6, (1.0, 1.0), 1.0)
    assert np.isnan(out["loss"][0]) and np.isnan(out["loss"][2]) and np.isfinite(out["loss"][1])
    assert np.all(np.isnan(out["grad_x0_student"][0][0])) and np.all(np.isfinite(out["grad_x0_student"][0][1]))


def pin_rf_wrapper(orc):
    """The rectified-flow reading of a TrigFlow sample: with t_rf = s/(c+s),
    z_rf = (1 - t_rf) z0 + t_rf eps (a straight line from data to noise);
    t_rf / (1 - t_rf) = tan t; t = pi/4 halves the sum z0 + eps; t = 0 and pi/2 give
    z0 and eps; t_rf rises strictly with t."""
    r = _rng(43)
    z0 = [r.normal(size=(4, 29)), r.normal(size=(4, 7))]
    eps = [r.normal(size=(4, 29)), r.normal(size=(4, 7))]
    t = np.array([0.05, 0.6, 1.1, 1.5])
    zt = orc.trigflow_noise(z0, eps, t)
    zrf, trf = orc.trigflow_to_rf(zt, t)
    for m in range(2):
        _close(zrf[m], (1 - trf)[:, None] * z0[m] + trf[:, None] * eps[m], rtol=1e-13, atol=1e-15)
    _close(trf / (1 - trf), np.tan(t), rtol=1e-13)
    assert np.all(np.diff(trf) > 0)
    zq, tq = orc.trigflow_to_rf(orc.trigflow_noise(z0, eps, np.full(4, math.pi / 4)), np.full(4, math.pi / 4))
    _close(tq, np.full(4, 0.5), rtol=1e-15)
    _close(zq[0], 0.5 * (z0[0] + eps[0]), rtol=1e-13, atol=1e-15)
    te = np.array([0.0, math.pi / 2, 0.0, math.pi / 2])
    ze, tre = orc.trigflow_to_rf(orc.trigflow_noise(z0, eps, te), te)
    _close(tre, np.array([0.0, 1.0, 0.0, 1.0]), rtol=0, atol=1e-15)
    _close(ze[1][0], z0[1][0], rtol=0, atol=0)
    _close(ze[1][1], eps[1][1], rtol=0, atol=1e-15)
    # stored path: both outputs rounded once; at t = pi/4 with eps = 0 the RF sample is
    # exactly z0 / 2, and the TrigFlow one is z0 / sqrt 2 rounded once
    zb = orc.round_to_bf16_bits(np.array([[1.0, 0.5, -3.0, 0.375]]))
    eb = orc.round_to_bf16_bits(np.zeros((1, 4)))
    zt_b, zrf_b, trf_b = orc.noise_rf([zb], [eb], np.array([math.pi / 4]), "bf16")
    assert np.array_equal(zrf_b[0], orc.round_to_bf16_bits(np.array([[0.5, 0.25, -1.5, 0.1875]])))
    assert np.array_equal(zt_b[0], orc.round_to_bf16_bits(np.array([[1.0, 0.5, -3.0, 0.375]]) / math.sqrt(2)))
    _close(trf_b, np.array([0.5]), rtol=1e-15)


def _cfg_inputs(seed, B=3, numels=(40, 12)):
    r = _rng(seed)
    zh = [r.normal(size=(B, n)) for n in numels]
    yc = [x + r.normal(0, 0.1, size=x.shape) for x in zh]
    yu = [x + r.normal(0, 0.1, size=x.shape) for x in zh]
    yF = [y + r.normal(0, 0.1, size=y.shape) for y in yc]
    return zh, yc, yu, yF


def pin_cfg_teacher(orc):
    """Guided teacher: scale 1 gives the conditional prediction and 0 the unconditional
    one; equal predictions make the scale irrelevant; a closed form with constant
    offsets (uncond = zhat0 + a, cond = zhat0 + b, fake = zhat0 + f) at the page's video
    and audio scales 3 and 5: c = |a + s (b - a)|, grad = 2 lam w (f - a - s (b - a)) / (c + eps);
    the stage-3 sum with guidance is the sCM terms plus the guided DMD terms."""
    zh, yc, yu, yF = _cfg_inputs(47)
    w, eps, lam = (1.0, 4.0), 1e-6, 0.25
    for scale, yT in ((1.0, yc), (0.0, yu)):
        a = orc.dmd_objective_cfg(zh, yc, yu, (scale, scale), yF, eps, w, lam)
        b = orc.dmd_objective(zh, yT, yF, eps, w, lam)
        _close(a["loss"], b["loss"], rtol=1e-14)
        _close(a["cdmd"], b["cdmd"], rtol=1e-14)
    a = orc.dmd_objective_cfg(zh, yc, yc, (3.0, 5.0), yF, eps, w, lam)
    b = orc.dmd_objective(zh, yc, yF, eps, w, lam)
    _close(a["loss"], b["loss"], rtol=1e-14)
    B, N = 2, 64
    r = _rng(53)
    offs = ((0.1, 0.3, 0.5), (-0.2, 0.05, 0.4))  # (a, b, f) per modality
    z = [r.normal(size=(B, N)) for _ in range(2)]
    out = orc.dmd_objective_cfg(z, [z[m] + offs[m][1] for m in range(2)],
                                [z[m] + offs[m][0] for m in range(2)], (3.0, 5.0),
                                [z[m] + offs[m][2] for m in range(2)], 1e-3, w, lam)
    loss = np.zeros(B)
    for m, (sc, (ao, bo, fo)) in enumerate(zip((3.0, 5.0), offs)):
        d = ao + sc * (bo - ao)
        c = abs(d)
        _close(out["cdmd"][:, m], np.full(B, c), rtol=1e-12)
        k = (fo - d) / (c + 1e-3)
        _close(out["grad_zhat0"][m], np.full((B, N), 2 * lam * w[m] * k), rtol=1e-10)
        loss += lam * w[m] * N * k * k
    _close(out["loss"], loss, rtol=1e-10)
    sz, xT, xS, tan, t = _scm_inputs(59)
    s3 = orc.stage3_objective_cfg(sz, xT, xS, tan, t, zh, yc, yu, (3.0, 5.0), yF,
                                  1.0, 0.9, 1e-6, 1e-6, w, 1.0, 0.25)
    a = orc.scm_objective(sz, xT, xS, tan, t, 1.0, 0.9, 1e-6, w, 1.0)
    b = orc.dmd_objective_cfg(zh, yc, yu, (3.0, 5.0), yF, 1e-6, w, 0.25)
    _close(s3["loss"], a["loss"] + b["loss"], rtol=1e-14)
    for m in range(2):
        _close(s3["grad_zhat0"][m], b["grad_zhat0"][m], rtol=0)


PINS = [pin_jvp_finite_difference, pin_jvp_autodiff, pin_direction_symbolic,
        pin_direction_closed_forms, pin_norm_and_loss, pin_zero_direction,
        pin_scm_gradient_autograd, pin_dmd_closed_form, pin_dmd_autograd,
        pin_stage3_composition, pin_bf16_rounding, pin_noise, pin_domain, pin_rf_wrapper,
        pin_cfg_teacher]


@pytest.mark.parametrize("pin", PINS, ids=[p.__name__ for p in PINS])
def test_oracle_pin(pin):
    pin(ORACLE)


# ---------------------------------------------------------------------------
# planted mistakes: every one must make at least one pin fail
# ---------------------------------------------------------------------------

def _fresh_oracle():
    spec = importlib.util.spec_from_file_location("oracle_mutant", ORACLE_FILE)
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    return mod


def _mut_jvp_tangent_sign(m):
    orig = m.joint_jvp
    m.joint_jvp = lambda z, Ft, FT, tan, t: orig(z, Ft, FT, -tan, t)


def _mut_jvp_no_ct(m):
    orig = m.joint_jvp
    m.joint_jvp = lambda z, Ft, FT, tan, t: orig(z, Ft, FT, tan, t) / (np.cos(t) * np.sin(t)).reshape(-1, 1)


def _mut_jvp_drop_explicit_z(m):
    def jvp(z, Ft, FT, tan, t):
        c, s = m._trig(t)
        return c * s * (-z - (c / s) * Ft - tan / s)
    m.joint_jvp = jvp


def _mut_direction(kind):
    def apply(m):
        def scm_direction(z_t, x0_teacher, x0_student, x0_tangent, t, beta, gamma):
            c, s = m._trig(t)
            F_T = m.trigflow_field(z_t, x0_teacher, t)
            F_theta = m.trigflow_field(z_t, x0_student, t)
            J = m.joint_jvp(z_t, F_theta, F_T, x0_tangent, t)
            gg = gamma if kind == "gamma_not_squared" else gamma ** 2
            coef = beta * c / np.sqrt(1.0 - gg * s ** 2)
            if kind == "no_cos_in_coef":
                coef = beta / np.sqrt(1.0 - gg * s ** 2)
            warm = 0.0 if kind == "drop_warmup" else gamma * c * s * z_t
            sign = -1.0 if kind == "flip_J" else 1.0
            return -coef * (F_theta - F_T) - warm - sign * J, F_theta, F_T
        m.scm_direction = scm_direction
    return apply


def _mut_norm_no_eps(m):
    m.l2_normalise = lambda g, eps: (g / np.sqrt(np.sum(g * g, axis=1))[:, None], np.sqrt(np.sum(g * g, axis=1)))


def _mut_norm_mean(m):
    m.l2_normalise = lambda g, eps: (g / (np.sqrt(np.mean(g * g, axis=1))[:, None] + eps), np.sqrt(np.mean(g * g, axis=1)))


def _mut_field_sign(m):
    m.trigflow_field = lambda z, x0, t: (x0 - m._trig(t)[0] * z) / m._trig(t)[1]


def _mut_dmd_scale_from_fake(m):
    orig = m.dmd_objective

    def dmd(zh, yT, yF, eps, w, lam=1.0, dtype="f64"):
        m.dmd_residual_scale = lambda a, b: np.mean(np.abs(a - b), axis=1) * 2.0
        try:
            return orig(zh, yT, yF, eps, w, lam, dtype)
        finally:
            m.dmd_residual_scale = ORACLE.dmd_residual_scale
    m.dmd_objective = dmd


def _mut_noise_swap(m):
    m.trigflow_noise = lambda z0, eps, t: [np.sin(np.asarray(t, dtype=np.float64)).reshape(-1, 1) * z
                                           + np.cos(np.asarray(t, dtype=np.float64)).reshape(-1, 1) * e
                                           for z, e in zip(z0, eps)]


def _mut_bf16_double_rounding(m):
    m.round_to_bf16_bits = lambda x: torch.from_numpy(np.asarray(x, np.float64).astype(np.float32)).to(
        torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


def _mut_scm_grad_no_inv_sin(m):
    orig = m.scm_objective

    def scm(*a, **k):
        out = orig(*a, **k)
        t = a[4]
        out["grad_x0_student"] = [g * np.sin(np.asarray(t)).reshape(-1, 1) for g in out["grad_x0_student"]]
        return out
    m.scm_objective = scm


def _mut_dmd_mean_loss(m):
    orig = m.dmd_objective

    def dmd(zh, yT, yF, eps, w, lam=1.0, dtype="f64"):
        out = orig(zh, yT, yF, eps, w, lam, dtype)
        out["loss"] = out["loss"] / np.asarray(zh[0]).shape[1]
        return out
    m.dmd_objective = dmd


def _mut_rf_norm_divisor(m):
    # divide by the rotation's norm sqrt(c^2 + s^2) = 1 instead of c + s
    m.trigflow_to_rf = lambda z, t: ([x.copy() for x in z],
                                     (np.sin(np.asarray(t, np.float64)) / 1.0).reshape(-1))


def _mut_rf_time_cos(m):
    orig = m.trigflow_to_rf

    def rf(z, t):
        zr, _ = orig(z, t)
        c, s = m._trig(t)
        return zr, (c / (c + s)).reshape(-1)
    m.trigflow_to_rf = rf


def _mut_cfg_swapped(m):
    m.cfg_prediction = lambda cond, uncond, scale: cond + scale * (uncond - cond)


def _mut_cfg_scale_order(m):
    orig = m.dmd_objective_cfg

    def cfg(zh, yc, yu, g, yF, *a, **k):
        return orig(zh, yc, yu, tuple(reversed(tuple(g))), yF, *a, **k)
    m.dmd_objective_cfg = cfg


MUTANTS = {
    "jvp_tangent_sign": _mut_jvp_tangent_sign,
    "jvp_no_ct": _mut_jvp_no_ct,
    "jvp_drop_explicit_z": _mut_jvp_drop_explicit_z,
    "direction_gamma_not_squared": _mut_direction("gamma_not_squared"),
    "direction_no_cos_in_coef": _mut_direction("no_cos_in_coef"),
    "direction_drop_warmup": _mut_direction("drop_warmup"),
    "direction_flip_J": _mut_direction("flip_J"),
    "norm_no_eps": _mut_norm_no_eps,
    "norm_mean_not_sum": _mut_norm_mean,
    "field_sign": _mut_field_sign,
    "dmd_scale_wrong": _mut_dmd_scale_from_fake,
    "dmd_mean_loss": _mut_dmd_mean_loss,
    "noise_swap_cos_sin": _mut_noise_swap,
    "bf16_double_rounding": _mut_bf16_double_rounding,
    "scm_grad_no_inv_sin": _mut_scm_grad_no_inv_sin,
    "rf_norm_divisor": _mut_rf_norm_divisor,
    "rf_time_cos": _mut_rf_time_cos,
    "cfg_swapped": _mut_cfg_swapped,
    "cfg_scale_order": _mut_cfg_scale_order,
}


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_pins_catch_planted_mistakes(name):
    mod = _fresh_oracle()
    MUTANTS[name](mod)
    failed = []
    for pin in PINS:
        try:
            with np.errstate(all="ignore"):
                pin(mod)
        except (AssertionError, FloatingPointError, ValueError):
            failed.append(pin.__name__)
    assert failed, f"planted mistake {name} was not caught by any pin"
