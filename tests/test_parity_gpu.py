"""GPU parity: the CUDA library, called through its C ABI, against the float64 oracle
on the same seeded inputs, for every workload and the edge cases of the method.

Tolerances are stated in tests/t2va_gpu_util.py: per-sample loss / norm / c_DMD
relative 1e-5 (float32 inputs) or 1e-4 (bfloat16 inputs); gradients per sample
max |gpu - oracle| <= 1e-3 max |oracle|; noise within the float32 evaluation bound
(one output ulp where the two terms do not cancel), see test_noise_parity.
"""

import math

import numpy as np
import pytest
import torch

import joint_video_audio_02_b300 as t2va
import oracle
import synthetic as S
from joint_video_audio_02_b300.build import build
from t2va_gpu_util import (Params, alloc_like, compare, gpu_run, grads_like, oracle_run, select,
                           to_device, to_host, ulp_diff_bf16)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    build()
    t2va.load()


def _inputs(name, **kw):
    return S.make_workload_inputs(S.workload(name), **kw)


# --------------------------------------------------------------------------
# the workloads
# --------------------------------------------------------------------------

def _ulp(v: np.ndarray, dtype: str) -> np.ndarray:
    """Spacing of the output type at |v| (8 significant bits for bf16, 24 for f32)."""
    _, e = np.frexp(np.abs(v))
    bits = 8 if dtype == "bf16" else 24
    return np.ldexp(1.0, np.maximum(e - bits, -133 if dtype == "bf16" else -149))


@pytest.mark.parametrize("name", ["tiny_scm_f32", "scm_512x768_bf16", "stage3_1024x1792_bf16"])
def test_noise_parity(name):
    """Bound from the arithmetic: the kernel evaluates cos t z0 + sin t eps in float32
    (sin/cos within 2 ulp, one product, one fma) and rounds once to the output type, so
    |out - exact| <= 1 ulp_out(exact) + 8 * 2^-24 (|cos t z0| + |sin t eps|). Where the
    two terms do not nearly cancel this is one unit in the last place."""
    wl = S.workload(name)
    inp = _inputs(name)
    z0 = to_device(inp.z0, wl.dtype)
    eps = to_device(inp.eps, wl.dtype)
    zt = alloc_like(z0)
    t = torch.from_numpy(inp.t).cuda()
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    t2va.noise(z0, eps, zt, t, status=status)
    got = to_host(zt, wl.dtype)
    ref = oracle.noise(inp.z0, inp.eps, inp.t, wl.dtype)
    t64 = inp.t.astype(np.float64)[:, None]
    for m in range(len(got)):
        z = oracle.decode(inp.z0[m], wl.dtype)
        e = oracle.decode(inp.eps[m], wl.dtype)
        exact = np.cos(t64) * z + np.sin(t64) * e
        mag = np.abs(np.cos(t64) * z) + np.abs(np.sin(t64) * e)
        g = oracle.decode(got[m], wl.dtype)
        bound = _ulp(exact, wl.dtype) + 8 * 2.0 ** -24 * mag
        assert np.all(np.abs(g - exact) <= bound), f"modality {m}: worst {np.max(np.abs(g - exact) / bound):.2f} of bound"
        if wl.dtype == "bf16":
            d = ulp_diff_bf16(got[m], ref[m])
            assert (d > 0).mean() < 1e-3, f"modality {m}: {(d > 0).mean():.2e} of elements differ from the oracle"
    assert status.item() == 0


@pytest.mark.parametrize("name", ["tiny_scm_f32", "scm_512x768_bf16"])
def test_scm_parity(name):
    wl = S.workload(name)
    inp = _inputs(name)
    gpu = gpu_run(inp, Params.of(wl), S.SCM)
    ref = oracle_run(inp, Params.of(wl), S.SCM)
    assert gpu["status"] == 0
    compare(gpu, ref, wl.dtype, S.SCM)


@pytest.mark.parametrize("name", ["stage3_512x768_bf16", "stage3_1024x1792_bf16",
                                  "stage3_sweep_b1_bf16", "stage3_sweep_b4_bf16"])
def test_stage3_parity(name):
    wl = S.workload(name)
    inp = _inputs(name)
    gpu = gpu_run(inp, Params.of(wl), S.STAGE3)
    ref = oracle_run(inp, Params.of(wl), S.STAGE3)
    assert gpu["status"] == 0
    compare(gpu, ref, wl.dtype, S.STAGE3)


@pytest.mark.parametrize("batch", [16, 32])
def test_stage3_sweep_full_size_sampled(batch):
    """Full-size launch; the oracle recomputes a sample of the batch (first, middle, last)."""
    wl = S.workload(f"stage3_sweep_b{batch}_bf16")
    inp = _inputs(wl.name)
    gpu = gpu_run(inp, Params.of(wl), S.STAGE3)
    assert gpu["status"] == 0
    samples = [0, batch // 2, batch - 1]
    ref = oracle_run(S.slice_samples(inp, samples), Params.of(wl), S.STAGE3)
    compare(select(gpu, samples), ref, wl.dtype, S.STAGE3)
    assert np.all(np.isfinite(gpu["loss"]))


def test_dmd_parity():
    wl = S.workload("stage3_512x768_bf16")
    inp = _inputs(wl.name)
    gpu = gpu_run(inp, Params.of(wl), S.DMD)
    ref = oracle_run(inp, Params.of(wl), S.DMD)
    assert gpu["status"] == 0
    compare(gpu, ref, wl.dtype, S.DMD)


def test_stage3_two_1024x1792_samples():
    """Two 1024x1792 samples (7.4M elements, 922K vectors): 1800 chunks of one
    512-vector batch, about four waves of three CTAs per SM, and inputs (103 MB) that
    nearly fill L2 between the two passes."""
    inp = S.make_inputs(2, S.workload("stage3_1024x1792_bf16").numels, "bf16", S.STAGE3, seed=(103,))
    p = Params()
    compare(gpu_run(inp, p, S.STAGE3), oracle_run(inp, p, S.STAGE3), "bf16", S.STAGE3)


def test_stage3_one_12M_element_row():
    """One sample whose video row has 12M elements (1.5M vectors): the row needs more
    than the 1024 chunks a row may have at one batch per chunk, so its chunks hold
    three 512-vector batches (977 chunks); the call's inputs (168 MB) do not fit in
    L2, so the gradient pass reads them from HBM again."""
    inp = S.make_inputs(1, [12_000_000, 1000], "bf16", S.STAGE3, seed=(104,))
    p = Params(weight=(1.0, 2.0))
    compare(gpu_run(inp, p, S.STAGE3), oracle_run(inp, p, S.STAGE3), "bf16", S.STAGE3)


# the configs clamp t to [1e-3, pi/2 - 1e-3]; both ends, in float32 as the kernels get them
T_CLAMP = np.array([1e-3, math.pi / 2 - 1e-3], dtype=np.float32)


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
@pytest.mark.parametrize("mode", [S.SCM, S.STAGE3, S.STAGE3_CFG])
@pytest.mark.parametrize("gamma", [0.0, 0.5, 0.9, 1.0])
@pytest.mark.parametrize("beta", [0.8, 1.0, 1.2])
def test_clamp_boundary_timesteps(dtype, mode, gamma, beta):
    """One sample at t = 1e-3 and one at t = pi/2 - 1e-3. There the sCM direction's
    beta cos t / sqrt(1 - gamma^2 sin^2 t) term nearly cancels the c^2 term of J
    (t -> 0, beta = 1), the gradient's 1/sin t is 1000, and with gamma = 1 the square
    root itself shrinks to cos t = 1e-3: the float32 per-sample coefficients must stay
    within the stated tolerances of the float64 oracle at both ends."""
    inp = S.make_inputs(2, [20000, 333], dtype, S.STAGE3_CFG if mode == S.STAGE3_CFG else S.STAGE3,
                        seed=(310, int(gamma * 10), int(beta * 10)))
    p = Params(gamma=gamma, beta=beta)
    gpu = gpu_run(inp, p, mode, t_override=T_CLAMP)
    ref = oracle_run(inp, p, mode, t_override=T_CLAMP)
    assert gpu["status"] == 0
    compare(gpu, ref, dtype, mode)


# --------------------------------------------------------------------------
# edge cases
# --------------------------------------------------------------------------

RAGGED = [
    # (batch, numels, stride padding)
    (3, [1, 7], 0),
    (2, [9, 8191], 3),
    (5, [100003, 5], 1),
    (2, [0, 77], 0),
    (1, [12345], 0),
    (3, [1000, 17, 4096], 5),
    (2, [33, 64, 1, 250001], 7),
]


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
@pytest.mark.parametrize("mode", [S.SCM, S.DMD, S.STAGE3])
@pytest.mark.parametrize("case", RAGGED, ids=[f"B{b}-{'-'.join(map(str, n))}-p{p}" for b, n, p in RAGGED])
def test_ragged(dtype, mode, case):
    B, numels, pad = case
    inp = S.make_inputs(B, numels, dtype, S.STAGE3, seed=(200, B, len(numels), pad))
    p = Params(weight=tuple(1.0 + 0.5 * m for m in range(len(numels))), gamma=0.7, beta=1.2)
    gpu = gpu_run(inp, p, mode, stride_pad=pad)
    ref = oracle_run(inp, p, mode)
    assert gpu["status"] == 0
    compare(gpu, ref, dtype, mode)


def test_empty_batch():
    z = [torch.empty((0, 64), dtype=torch.bfloat16, device="cuda")]
    t = torch.empty((0,), device="cuda")
    t2va.noise(z, z, [torch.empty_like(z[0])], t)
    ws = t2va.new_workspace(1, 1)
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    loss = torch.empty((0,), device="cuda")
    g = [torch.empty((0, 64), device="cuda")]
    t2va.stage3_objective(z, z, z, z, t, z, z, z, beta=1, gamma=0.5, eps_scm=1e-6, eps_dmd=1e-6,
                          weight=[1.0], lambda_scm=1, lambda_dmd=1, grad_x0_student=g, grad_zhat0=g,
                          loss=loss, workspace=ws, status=st)
    torch.cuda.synchronize()
    assert st.item() == 0


@pytest.mark.parametrize("mode", [S.SCM, S.STAGE3])
def test_bad_timesteps(mode):
    """t outside (0, pi/2): that sample's outputs are NaN and the status bit is set;
    the other samples are unaffected."""
    inp = S.make_inputs(6, [5000, 300], "bf16", S.STAGE3, seed=(300,))
    t = np.array([0.5, 0.0, np.float32(math.pi / 2), np.nan, -0.3, 1.2], dtype=np.float32)
    p = Params()
    gpu = gpu_run(inp, p, mode, t_override=t)
    ref = oracle_run(inp, p, mode, t_override=t)
    assert gpu["status"] & t2va.STATUS_BAD_TIMESTEP
    assert np.array_equal(np.isnan(gpu["loss"]), [False, True, True, True, True, False])
    compare(gpu, ref, "bf16", mode)


def test_zero_direction_is_exactly_zero():
    """gamma = 1, student = teacher, zero tangent, fake = teacher: both directions vanish,
    so every norm, loss and gradient is exactly 0 (closed form)."""
    inp = S.make_inputs(3, [4099, 130], "bf16", S.STAGE3, seed=(301,))
    inp.x0_student = [a.copy() for a in inp.x0_teacher]
    inp.x0_tangent = [np.zeros_like(a) for a in inp.x0_tangent]
    inp.x0_fake = [a.copy() for a in inp.x0_teacher_hat]
    gpu = gpu_run(inp, Params(gamma=1.0, beta=0.8), S.STAGE3)
    assert gpu["status"] == 0
    for k in ("loss", "norm", "loss_scm", "loss_dmd"):
        assert np.all(gpu[k] == 0.0), k
    for g in gpu["grad_x0_student"] + gpu["grad_zhat0"]:
        assert np.all(g == 0.0)
    assert np.all(gpu["cdmd"] > 0)


def test_accumulate():
    inp = S.make_inputs(2, [20000, 333], "bf16", S.STAGE3, seed=(302,))
    p = Params()
    rng = np.random.default_rng(0)
    prior = {"grad_x0_student": [rng.normal(size=a.shape).astype(np.float32) for a in inp.z0],
             "grad_zhat0": [rng.normal(size=a.shape).astype(np.float32) for a in inp.z0]}
    gpu = gpu_run(inp, p, S.STAGE3, accumulate_into=prior)
    ref = oracle_run(inp, p, S.STAGE3)
    for k in ("grad_x0_student", "grad_zhat0"):
        ref[k] = [r + q.astype(np.float64) for r, q in zip(ref[k], prior[k])]
    compare(gpu, ref, "bf16", S.STAGE3)


def test_alias_sums_gradients():
    """grad_zhat0 given as the same buffer as grad_x0_student: the two gradients are summed."""
    inp = S.make_inputs(2, [20000, 333], "bf16", S.STAGE3, seed=(303,))
    p = Params()
    gpu = gpu_run(inp, p, S.STAGE3, alias=True)
    ref = oracle_run(inp, p, S.STAGE3)
    summed = [a + b for a, b in zip(ref["grad_x0_student"], ref["grad_zhat0"])]
    ref["grad_x0_student"] = summed
    ref["grad_zhat0"] = summed
    compare(gpu, ref, "bf16", S.STAGE3)


def test_reproducible_bitwise():
    inp = _inputs("stage3_512x768_bf16")
    p = Params.of(S.workload("stage3_512x768_bf16"))
    a = gpu_run(inp, p, S.STAGE3)
    b = gpu_run(inp, p, S.STAGE3)
    for k in ("loss", "norm", "cdmd"):
        assert np.array_equal(a[k], b[k])
    for k in ("grad_x0_student", "grad_zhat0"):
        for x, y in zip(a[k], b[k]):
            assert np.array_equal(x, y)


def test_cuda_graph_capture_matches_eager():
    wl = S.workload("stage3_512x768_bf16")
    inp = _inputs(wl.name)
    p = Params.of(wl)
    dt = wl.dtype
    z0, eps, xT, xS, tan, zh, yT, yF = (to_device(getattr(inp, f), dt) for f in (
        "z0", "eps", "x0_teacher", "x0_student", "x0_tangent", "zhat0", "x0_teacher_hat", "x0_fake"))
    t = torch.from_numpy(inp.t).cuda()
    zt = alloc_like(z0)
    gS, gD = grads_like(z0), grads_like(z0)
    loss = torch.zeros(wl.batch, device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    ws = t2va.new_workspace(wl.batch, 2)

    def step():
        t2va.noise(z0, eps, zt, t, status=st)
        t2va.stage3_objective(zt, xT, xS, tan, t, zh, yT, yF, beta=p.beta, gamma=p.gamma,
                              eps_scm=p.eps_scm, eps_dmd=p.eps_dmd, weight=p.weight,
                              lambda_scm=p.lambda_scm, lambda_dmd=p.lambda_dmd, grad_x0_student=gS,
                              grad_zhat0=gD, loss=loss, workspace=ws, status=st)

    step()
    torch.cuda.synchronize()
    eager = (loss.clone(), [g.clone() for g in gS], [g.clone() for g in gD])
    for g in gS + gD:
        g.zero_()
    loss.zero_()
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.stream(s):
        with torch.cuda.graph(graph, stream=s):
            step()
    torch.cuda.current_stream().wait_stream(s)
    for _ in range(3):
        graph.replay()
    torch.cuda.synchronize()
    assert st.item() == 0
    assert torch.equal(loss, eager[0])
    for a, b in zip(gS + gD, eager[1] + eager[2]):
        assert torch.equal(a, b)


def test_objective_right_after_the_noising_that_writes_its_input():
    """The noising kernel lets its dependents launch early, and the objective's first
    kernel starts pulling its inputs into L2 before its dependency wait. Here the
    noising overwrites z_t (holding the previous iteration's values) immediately before
    the objective reads it, on one stream with no synchronisation: the results must be
    bit-identical to the objective run on a settled copy of that z_t, and match the
    float64 oracle on it."""
    wl = S.workload("stage3_512x768_bf16")
    inp = _inputs(wl.name)
    p = Params.of(wl)
    dt = wl.dtype
    z0, eps, xT, xS, tan, zh, yT, yF = (to_device(getattr(inp, f), dt) for f in (
        "z0", "eps", "x0_teacher", "x0_student", "x0_tangent", "zhat0", "x0_teacher_hat", "x0_fake"))
    zt = alloc_like(z0)
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    ws = t2va.new_workspace(wl.batch, 2)

    def objective(z, t):
        gS, gD = grads_like(z0, float("nan")), grads_like(z0, float("nan"))
        loss, loss_s, loss_d = (torch.full((wl.batch,), float("nan"), device="cuda") for _ in range(3))
        norm = torch.full((wl.batch * 2,), float("nan"), device="cuda")
        cdmd = torch.full((wl.batch * 2,), float("nan"), device="cuda")
        t2va.stage3_objective(z, xT, xS, tan, t, zh, yT, yF, beta=p.beta, gamma=p.gamma,
                              eps_scm=p.eps_scm, eps_dmd=p.eps_dmd, weight=p.weight,
                              lambda_scm=p.lambda_scm, lambda_dmd=p.lambda_dmd, grad_x0_student=gS,
                              grad_zhat0=gD, loss=loss, loss_scm=loss_s, loss_dmd=loss_d, norm=norm,
                              cdmd=cdmd, workspace=ws, status=st)
        return (loss, loss_s, loss_d, norm, cdmd), gS, gD

    rng = np.random.default_rng(41)
    for it in range(4):
        t_host = rng.uniform(0.05, 1.5, wl.batch).astype(np.float32)
        t = torch.from_numpy(t_host).cuda()
        torch.cuda.synchronize()
        t2va.noise(z0, eps, zt, t, status=st)         # overwrites last iteration's z_t
        chained = objective(zt, t)                    # same stream, no synchronisation
        torch.cuda.synchronize()
        settled_zt = [z.clone() for z in zt]
        torch.cuda.synchronize()
        settled = objective(settled_zt, t)
        torch.cuda.synchronize()
        assert st.item() == 0
        for a, b in zip(chained[0], settled[0]):
            assert torch.equal(a, b), it
        for a, b in zip(chained[1] + chained[2], settled[1] + settled[2]):
            assert torch.equal(a, b), it
    # the last chained call against the oracle on the z_t the noising wrote
    zt_bits = [z.view(torch.int16).cpu().numpy().view(np.uint16) for z in zt]
    ref = oracle.stage3_objective(zt_bits, inp.x0_teacher, inp.x0_student, inp.x0_tangent, t_host,
                                  inp.zhat0, inp.x0_teacher_hat, inp.x0_fake, p.beta, p.gamma,
                                  p.eps_scm, p.eps_dmd, p.weight, p.lambda_scm, p.lambda_dmd, dt)
    (loss, loss_s, loss_d, norm, cdmd), gS, gD = chained
    compare({"loss": loss.cpu().numpy(), "loss_scm": loss_s.cpu().numpy(), "loss_dmd": loss_d.cpu().numpy(),
             "norm": norm.cpu().numpy().reshape(wl.batch, 2), "cdmd": cdmd.cpu().numpy().reshape(wl.batch, 2),
             "grad_x0_student": [g.cpu().numpy() for g in gS],
             "grad_zhat0": [g.cpu().numpy() for g in gD]}, ref, dt, S.STAGE3)


def test_noising_right_after_the_objective_that_writes_its_input():
    """The noising kernel also pulls its inputs into L2 before its dependency wait. Here
    its z0 and eps are the float32 gradients that the objective's second kernel (which
    lets its dependents launch early) writes immediately before, on one stream with no
    synchronisation: z_t must be bit-identical to the noising of a settled copy."""
    wl = S.workload("stage3_512x768_bf16")
    inp = _inputs(wl.name)
    p = Params.of(wl)
    dt = wl.dtype
    zt_in, xT, xS, tan, zh, yT, yF = (to_device(getattr(inp, f), dt) for f in (
        "z0", "x0_teacher", "x0_student", "x0_tangent", "zhat0", "x0_teacher_hat", "x0_fake"))
    t = torch.from_numpy(inp.t).cuda()
    gS, gD = grads_like(zt_in, float("nan")), grads_like(zt_in, float("nan"))
    out = grads_like(zt_in, float("nan"))
    loss = torch.zeros(wl.batch, device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    ws = t2va.new_workspace(wl.batch, 2)
    rng = np.random.default_rng(43)
    for it in range(4):
        w = [float(x) for x in rng.uniform(0.5, 2.0, 2)]
        t_noise = torch.from_numpy(rng.uniform(0.05, 1.5, wl.batch).astype(np.float32)).cuda()
        torch.cuda.synchronize()
        t2va.stage3_objective(zt_in, xT, xS, tan, t, zh, yT, yF, beta=p.beta, gamma=p.gamma,
                              eps_scm=p.eps_scm, eps_dmd=p.eps_dmd, weight=w,
                              lambda_scm=p.lambda_scm, lambda_dmd=p.lambda_dmd, grad_x0_student=gS,
                              grad_zhat0=gD, loss=loss, workspace=ws, status=st)
        t2va.noise(gS, gD, out, t_noise, status=st)   # same stream, no synchronisation
        torch.cuda.synchronize()
        chained = [o.clone() for o in out]
        settled_in = ([g.clone() for g in gS], [g.clone() for g in gD])
        torch.cuda.synchronize()
        t2va.noise(settled_in[0], settled_in[1], out, t_noise, status=st)
        torch.cuda.synchronize()
        assert st.item() == 0
        for a, b in zip(chained, out):
            assert torch.equal(a, b), it
            assert torch.isfinite(a).all(), it


# --------------------------------------------------------------------------
# the workspace: per-chunk partial sums written and read within one call
# --------------------------------------------------------------------------

def test_workspace_contents_do_not_matter():
    """The first kernel of a call writes every partial sum the second one reads, so a
    workspace full of garbage (never initialised, or left by a call with other sizes)
    gives bit-identical results."""
    inp = S.make_inputs(3, [50_003, 701], "bf16", S.STAGE3, seed=(400,))
    p = Params(weight=(1.0, 3.0))
    clean = gpu_run(inp, p, S.STAGE3)
    ws = torch.randint(0, 256, (t2va.workspace_bytes(3, 2),), dtype=torch.uint8, device="cuda")
    dirty = gpu_run(inp, p, S.STAGE3, workspace=ws)
    assert dirty["status"] == 0
    for k in ("loss", "norm", "cdmd"):
        assert np.array_equal(clean[k], dirty[k])
    for k in ("grad_x0_student", "grad_zhat0"):
        for x, y in zip(clean[k], dirty[k]):
            assert np.array_equal(x, y)
    # the same workspace for calls with other sizes, then this call again
    gpu_run(S.make_inputs(2, [777, 33], "bf16", S.STAGE3, seed=(401,)), p, S.STAGE3, workspace=ws)
    gpu_run(S.make_inputs(1, [9, 8191], "f32", S.STAGE3, seed=(402,)), p, S.SCM, workspace=ws)
    again = gpu_run(inp, p, S.STAGE3, workspace=ws)
    for k in ("loss", "loss_scm", "loss_dmd", "norm", "cdmd"):
        assert np.array_equal(clean[k], again[k]), k
    for k in ("grad_x0_student", "grad_zhat0"):
        for x, y in zip(clean[k], again[k]):
            assert np.array_equal(x, y)


def test_host_errors_on_device():
    inp = S.make_inputs(2, [64, 16], "bf16", S.STAGE3, seed=(402,))
    z = to_device(inp.z0, "bf16")
    t = torch.from_numpy(inp.t).cuda()
    ws = t2va.new_workspace(2, 2)
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    loss = torch.zeros(2, device="cuda")
    g = grads_like(z)
    small = ws[: ws.numel() // 2]
    with pytest.raises(t2va.T2VAError) as e:
        t2va.scm_objective(z, z, z, z, t, beta=1, gamma=0.5, eps_scm=1e-6, weight=[1, 1], lambda_scm=1,
                           grad_x0_student=g, loss=loss, workspace=small, status=st)
    assert e.value.code == 4
    with pytest.raises(t2va.T2VAError) as e:
        t2va.scm_objective(z, z, z, z, t, beta=1, gamma=1.5, eps_scm=1e-6, weight=[1, 1], lambda_scm=1,
                           grad_x0_student=g, loss=loss, workspace=ws, status=st)
    assert e.value.code == 1
    flat = torch.zeros(2 * 64 + 8, dtype=torch.bfloat16, device="cuda")
    mis = [flat[1:129].view(2, 64), z[1]]
    with pytest.raises(t2va.T2VAError) as e:
        t2va.noise(mis, mis, mis, t)
    assert e.value.code == 3
