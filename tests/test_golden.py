"""The oracle against hand-derived values of the pages' equations (tests/golden/): closed
forms at exact angles, a matched student and teacher, a four-element DMD term, the guided
teacher at the printed guidance scales, quantisation codes with exact ties, and one row of
the fused normalisation. Each fixture cites the passage it follows. Planted mistakes in
fresh copies of the oracle modules must each fail one of these checks. CPU only."""

import importlib.util
import os

import numpy as np
import pytest

from golden_util import ANGLES, load, num, scalar

ORACLE = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "oracle")


def _fresh(name):
    spec = importlib.util.spec_from_file_location(f"golden_{name}", os.path.join(ORACLE, name + ".py"))
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    return mod


def _modules():
    return _fresh("t2va_oracle"), _fresh("w8a8_oracle"), _fresh("fused_ops_oracle")


def check_trigflow_noise_and_rf_wrapper(O, W8, F):
    g = load("trigflow_noise_rf.txt")
    z0, eps = scalar(g["z0"]), scalar(g["eps"])
    for key, n in ANGLES:
        t = np.array([np.pi / n])
        zt = O.trigflow_noise([np.array([[z0]])], [np.array([[eps]])], t)[0]
        zrf, trf = O.trigflow_to_rf([zt], t)
        assert abs(zt[0, 0] - scalar(g[key + ".z_t"])) <= 1e-15
        assert abs(zrf[0][0, 0] - scalar(g[key + ".z_rf"])) <= 1e-15
        assert abs(trf[0] - scalar(g[key + ".t_rf"])) <= 1e-15


def check_scm_matched_student(O, W8, F):
    g = load("scm_direction_closed_form.txt")
    z, x0, tan = num(g["z_t"])[None], num(g["x0"])[None], num(g["tangent"])[None]
    r = O.scm_objective([z], [x0], [x0.copy()], [tan], np.array([num(g["t"])]), scalar(g["beta"]),
                        scalar(g["gamma"]), scalar(g["eps_scm"]), [1.0])
    np.testing.assert_allclose(r["g"][0][0], num(g["g"]), rtol=1e-14, atol=1e-15)
    np.testing.assert_allclose(r["norm"][0, 0], scalar(g["norm"]), rtol=1e-14)
    np.testing.assert_allclose(r["loss"][0], scalar(g["loss"]), rtol=1e-14)
    np.testing.assert_allclose(r["grad_x0_student"][0][0], num(g["grad_x0_student"]), rtol=1e-14)


def check_dmd_residual_scale(O, W8, F):
    g = load("dmd_residual_scale.txt")
    r = O.dmd_objective([num(g["zhat0"])[None]], [num(g["x0_teacher_hat"])[None]], [num(g["x0_fake"])[None]],
                        scalar(g["eps_dmd"]), [1.0])
    assert r["cdmd"][0, 0] == scalar(g["cdmd"])
    np.testing.assert_allclose(r["loss"][0], scalar(g["loss"]), rtol=1e-15)
    np.testing.assert_allclose(r["grad_zhat0"][0][0], num(g["grad_zhat0"]), rtol=1e-15, atol=0)


def check_guided_teacher(O, W8, F):
    g = load("cfg_guided_teacher.txt")
    cond, uncond = num(g["cond"]), num(g["uncond"])
    assert np.array_equal(O.cfg_prediction(cond, uncond, scalar(g["scale_video"])), num(g["guided_video"]))
    assert np.array_equal(O.cfg_prediction(cond, uncond, scalar(g["scale_audio"])), num(g["guided_audio"]))
    r = O.dmd_objective_cfg([num(g["dmd.zhat0"])[None]], [num(g["dmd.cond"])[None]], [num(g["dmd.uncond"])[None]],
                            [scalar(g["scale_video"])], [num(g["dmd.x0_fake"])[None]], scalar(g["dmd.eps_dmd"]), [1.0])
    assert r["cdmd"][0, 0] == scalar(g["dmd.cdmd"])
    np.testing.assert_allclose(r["loss"][0], scalar(g["dmd.loss"]), rtol=1e-15)
    np.testing.assert_allclose(r["grad_zhat0"][0][0], num(g["dmd.grad_zhat0"]), rtol=1e-15)


def check_w8a8_codes_and_linear(O, W8, F):
    g = load("w8a8_quantise_and_linear.txt")
    for k in ("row1", "row2", "row3", "row4"):
        q, s = W8.quantize_rows(num(g[k]).astype(np.float32)[None])
        assert np.array_equal(q[0].astype(np.int64), num(g[k + ".codes"]).astype(np.int64)), k
        assert s[0] == np.float32(scalar(g[k + ".scale"])), k
    acc, y = W8.w8a8_linear(num(g["xq"]).astype(np.int8), num(g["sx"]).astype(np.float32),
                            num(g["wq"]).astype(np.int8), num(g["sw"]).astype(np.float32),
                            num(g["bias"]).astype(np.float32))
    assert np.array_equal(acc, num(g["acc"]).astype(np.int64))
    assert np.array_equal(y, num(g["y"]))


def check_residual_modnorm(O, W8, F):
    g = load("residual_modnorm.txt")
    vec = lambda k: num(g[k])[None]
    h2, y = F.residual_modnorm(vec("h"), vec("u"), vec("gate"), vec("scale"), vec("shift"), scalar(g["eps"]), 1,
                               lambda v: np.asarray(v, np.float64))
    assert np.array_equal(h2[0], num(g["h_new"]))
    np.testing.assert_allclose(y[0], num(g["y"]), rtol=1e-15, atol=0)


CHECKS = [check_trigflow_noise_and_rf_wrapper, check_scm_matched_student, check_dmd_residual_scale,
          check_guided_teacher, check_w8a8_codes_and_linear, check_residual_modnorm]


@pytest.mark.parametrize("check", CHECKS, ids=[c.__name__ for c in CHECKS])
def test_golden(check):
    check(*_modules())


# planted mistakes: each edits fresh copies of the oracle modules
def _swap_cos_sin(O, W8, F):
    orig = O._trig
    O._trig = lambda t: orig(t)[::-1]


def _rf_time_from_cos(O, W8, F):
    orig = O.trigflow_to_rf

    def f(z, t):
        zr, trf = orig(z, t)
        return zr, 1.0 - trf
    O.trigflow_to_rf = f


def _drop_gamma_term(O, W8, F):
    orig = O.scm_direction

    def f(z_t, x_T, x_S, x_dot, t, beta, gamma):
        g, Fs, Ft = orig(z_t, x_T, x_S, x_dot, t, beta, gamma)
        c, s = O._trig(t)
        return g + gamma * c * s * z_t, Fs, Ft
    O.scm_direction = f


def _jvp_sign(O, W8, F):
    orig = O.joint_jvp
    O.joint_jvp = lambda *a: -orig(*a)


def _eps_inside_root(O, W8, F):
    def f(g, eps):
        n = np.sqrt(np.sum(g * g, axis=1))
        return g / np.sqrt(n * n + eps)[:, None], n
    O.l2_normalise = f


def _scale_sum_not_mean(O, W8, F):
    O.dmd_residual_scale = lambda zh, y: np.sum(np.abs(zh - y), axis=1)


def _cfg_reversed(O, W8, F):
    O.cfg_prediction = lambda k, u, s: k + s * (u - k)


def _round_half_away(O, W8, F):
    def f(x, eps=W8.EPS):
        x32 = np.asarray(x, np.float32)
        s = W8.row_scales(x32, eps)
        q = np.clip(np.sign(x32) * np.floor(np.abs(x32 / s[:, None]) + 0.5), -127, 127)
        return q.astype(np.int8), s
    W8.quantize_rows = f


def _scale_over_128(O, W8, F):
    orig = W8.row_scales
    W8.row_scales = lambda x, eps=W8.EPS: (orig(x, eps) * np.float32(127.0) / np.float32(128.0)).astype(np.float32)


def _gate_on_h(O, W8, F):
    F.gated_residual = lambda h, u, gate: (1.0 if gate is None else np.asarray(gate)) * np.asarray(h) + np.asarray(u)


MUTANTS = {"cos_sin_swapped": _swap_cos_sin, "rf_time_from_cos": _rf_time_from_cos,
           "scm_gamma_term_dropped": _drop_gamma_term, "jvp_sign_flipped": _jvp_sign,
           "eps_inside_root": _eps_inside_root, "dmd_scale_sum_not_mean": _scale_sum_not_mean,
           "cfg_reversed": _cfg_reversed, "round_half_away_from_zero": _round_half_away,
           "scale_over_128": _scale_over_128, "gate_on_h": _gate_on_h}


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_golden_catches_planted_mistakes(name):
    mods = _modules()
    MUTANTS[name](*mods)
    failed = []
    for check in CHECKS:
        try:
            with np.errstate(all="ignore"):
                check(*mods)
        except (AssertionError, ValueError, IndexError, FloatingPointError):
            failed.append(check.__name__)
    assert failed, f"planted mistake {name} was not caught"
