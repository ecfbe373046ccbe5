"""The seeded input generator: shapes, determinism, storage formats, distributions."""

import math

import numpy as np
import torch

import synthetic as S


def test_workload_shapes():
    assert S.workload("tiny_scm_f32").numels == [6144, 1024]
    assert S.workload("scm_512x768_bf16").numels == [786432, 16128]
    assert S.workload("stage3_1024x1792_bf16").numels == [3670016, 16128]
    for b in (1, 4, 16, 32):
        wl = S.workload(f"stage3_sweep_b{b}_bf16")
        assert wl.batch == b and wl.numels == [786432, 64512] and wl.weight == (1.0, 4.0)


def test_deterministic_and_seed_dependent():
    a = S.make_inputs(3, [100, 17], "bf16", S.STAGE3, seed=(5,))
    b = S.make_inputs(3, [100, 17], "bf16", S.STAGE3, seed=(5,))
    c = S.make_inputs(3, [100, 17], "bf16", S.STAGE3, seed=(6,))
    for f in ("z0", "eps", "x0_teacher", "x0_student", "x0_tangent", "zhat0", "x0_teacher_hat", "x0_fake"):
        for m in range(2):
            assert np.array_equal(getattr(a, f)[m], getattr(b, f)[m])
            assert getattr(a, f)[m].dtype == np.uint16 and getattr(a, f)[m].shape == (3, [100, 17][m])
    assert not np.array_equal(a.z0[0], c.z0[0])
    assert np.array_equal(a.t, b.t)


def test_bf16_encoding_matches_torch():
    x = np.random.default_rng(0).normal(size=10000).astype(np.float32)
    ref = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(S.bf16_bits_from_f32(x), ref)
    assert np.array_equal(S.f32_from_bf16_bits(ref), torch.from_numpy(ref.view(np.int16)).view(torch.bfloat16).float().numpy())


def test_distributions():
    inp = S.make_inputs(4, [200000], "f32", S.STAGE3, seed=(9,))
    z0, xt, xs, tan = inp.z0[0], inp.x0_teacher[0], inp.x0_student[0], inp.x0_tangent[0]
    assert abs(z0.std() - 1.0) < 0.01
    assert abs((xt - z0).std() - 0.1) < 0.002
    assert abs((xs - xt).std() - 0.05) < 0.001
    assert abs(tan.std() - 0.5) < 0.005
    assert abs((inp.x0_fake[0] - inp.x0_teacher_hat[0]).std() - 0.1) < 0.002
    t = S.make_inputs(20000, [1], "f32", S.SCM, seed=(1,)).t
    assert t.min() >= np.float32(1e-3) and t.max() <= np.float32(math.pi / 2 - 1e-3)
    tau = np.log(np.tan(t.astype(np.float64)))
    assert abs(tau.mean() + 0.8) < 0.05 and abs(tau.std() - 1.6) < 0.05


def test_fixed_timesteps_and_slicing():
    wl = S.workload("tiny_scm_f32")
    inp = S.make_workload_inputs(wl)
    assert np.array_equal(inp.t, np.array([0.3, 1.1], dtype=np.float32))
    sub = S.slice_samples(inp, [1])
    assert sub.batch == 1 and np.array_equal(sub.z0[0][0], inp.z0[0][1])
