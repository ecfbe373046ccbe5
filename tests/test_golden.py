"""The oracle against hand-derived values of the pages' equations (tests/golden/): closed
forms at exact angles, a matched student and teacher, a four-element DMD term, the guided
teacher at the printed guidance scales, quantisation codes with exact ties, and one row of
the fused normalisation. Each fixture cites the passage it follows. CPU only."""

import numpy as np

import oracle.fused_ops_oracle as F
import oracle.t2va_oracle as O
import oracle.w8a8_oracle as W8
from golden_util import ANGLES, load, num, scalar


def test_golden_trigflow_noise_and_rf_wrapper():
    g = load("trigflow_noise_rf.txt")
    z0, eps = scalar(g["z0"]), scalar(g["eps"])
    for key, n in ANGLES:
        t = np.array([np.pi / n])
        zt = O.trigflow_noise([np.array([[z0]])], [np.array([[eps]])], t)[0]
        zrf, trf = O.trigflow_to_rf([zt], t)
        assert abs(zt[0, 0] - scalar(g[key + ".z_t"])) <= 1e-15
        assert abs(zrf[0][0, 0] - scalar(g[key + ".z_rf"])) <= 1e-15
        assert abs(trf[0] - scalar(g[key + ".t_rf"])) <= 1e-15


def test_golden_scm_matched_student():
    g = load("scm_direction_closed_form.txt")
    z, x0, tan = num(g["z_t"])[None], num(g["x0"])[None], num(g["tangent"])[None]
    r = O.scm_objective([z], [x0], [x0.copy()], [tan], np.array([num(g["t"])]), scalar(g["beta"]),
                        scalar(g["gamma"]), scalar(g["eps_scm"]), [1.0])
    np.testing.assert_allclose(r["g"][0][0], num(g["g"]), rtol=1e-14, atol=1e-15)
    np.testing.assert_allclose(r["norm"][0, 0], scalar(g["norm"]), rtol=1e-14)
    np.testing.assert_allclose(r["loss"][0], scalar(g["loss"]), rtol=1e-14)
    np.testing.assert_allclose(r["grad_x0_student"][0][0], num(g["grad_x0_student"]), rtol=1e-14)


def test_golden_dmd_residual_scale():
    g = load("dmd_residual_scale.txt")
    r = O.dmd_objective([num(g["zhat0"])[None]], [num(g["x0_teacher_hat"])[None]], [num(g["x0_fake"])[None]],
                        scalar(g["eps_dmd"]), [1.0])
    assert r["cdmd"][0, 0] == scalar(g["cdmd"])
    np.testing.assert_allclose(r["loss"][0], scalar(g["loss"]), rtol=1e-15)
    np.testing.assert_allclose(r["grad_zhat0"][0][0], num(g["grad_zhat0"]), rtol=1e-15, atol=0)


def test_golden_guided_teacher():
    g = load("cfg_guided_teacher.txt")
    cond, uncond = num(g["cond"]), num(g["uncond"])
    assert np.array_equal(O.cfg_prediction(cond, uncond, scalar(g["scale_video"])), num(g["guided_video"]))
    assert np.array_equal(O.cfg_prediction(cond, uncond, scalar(g["scale_audio"])), num(g["guided_audio"]))
    r = O.dmd_objective_cfg([num(g["dmd.zhat0"])[None]], [num(g["dmd.cond"])[None]], [num(g["dmd.uncond"])[None]],
                            [scalar(g["scale_video"])], [num(g["dmd.x0_fake"])[None]], scalar(g["dmd.eps_dmd"]), [1.0])
    assert r["cdmd"][0, 0] == scalar(g["dmd.cdmd"])
    np.testing.assert_allclose(r["loss"][0], scalar(g["dmd.loss"]), rtol=1e-15)
    np.testing.assert_allclose(r["grad_zhat0"][0][0], num(g["dmd.grad_zhat0"]), rtol=1e-15)


def test_golden_w8a8_codes_and_linear():
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


def test_golden_residual_modnorm():
    g = load("residual_modnorm.txt")
    vec = lambda k: num(g[k])[None]
    h2, y = F.residual_modnorm(vec("h"), vec("u"), vec("gate"), vec("scale"), vec("shift"), scalar(g["eps"]), 1,
                               lambda v: np.asarray(v, np.float64))
    assert np.array_equal(h2[0], num(g["h_new"]))
    np.testing.assert_allclose(y[0], num(g["y"]), rtol=1e-15, atol=0)
