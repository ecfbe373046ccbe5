"""GPU parity of the noising step fused with the TrigFlow -> rectified-flow wrapper
(t2va_noise_rf) against the float64 oracle.

Bounds from the arithmetic. The kernel computes, in float32, c = cos t and s = sin t
(each within 2 ulp), c + s (one rounding; no cancellation for t in [0, pi/2]), and the
coefficients c / (c + s), s / (c + s) (one rounding each): every coefficient is within
10 * 2^-24 of its exact value, relatively. Each output is then one product and one fma
of a coefficient pair with the stored inputs, rounded once to the output type, so
  |z_rf - exact| <= 1 ulp_out(exact) + 16 * 2^-24 (|c z0| + |s eps|) / (c + s),
  |t_rf - exact| <= 12 * 2^-24 exact.
The z_t output is the same arithmetic as t2va_noise and must match it bit for bit.
"""

import math

import numpy as np
import pytest
import torch

import joint_video_audio_02_b300 as t2va
import oracle
import synthetic as S
from joint_video_audio_02_b300.build import build
from t2va_gpu_util import alloc_like, to_device, to_host, ulp_diff_bf16

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    build()
    t2va.load()


def _ulp(v: np.ndarray, dtype: str) -> np.ndarray:
    _, e = np.frexp(np.abs(v))
    bits = 8 if dtype == "bf16" else 24
    return np.ldexp(1.0, np.maximum(e - bits, -133 if dtype == "bf16" else -149))


def _check_rf(inp: S.Inputs, got_zrf, got_trf, t: np.ndarray):
    dt = inp.dtype
    t64 = t.astype(np.float64)
    c, s = np.cos(t64)[:, None], np.sin(t64)[:, None]
    for m in range(len(got_zrf)):
        z = oracle.decode(inp.z0[m], dt)
        e = oracle.decode(inp.eps[m], dt)
        exact = (c * z + s * e) / (c + s)
        mag = (np.abs(c * z) + np.abs(s * e)) / (c + s)
        g = oracle.decode(got_zrf[m], dt)
        bound = _ulp(exact, dt) + 16 * 2.0 ** -24 * mag
        assert np.all(np.abs(g - exact) <= bound), \
            f"z_rf modality {m}: worst {np.max(np.abs(g - exact) / bound):.2f} of bound"
    if got_trf is not None:
        exact_t = np.sin(t64) / (np.cos(t64) + np.sin(t64))
        assert np.all(np.abs(got_trf.astype(np.float64) - exact_t) <= 12 * 2.0 ** -24 * exact_t), \
            "t_rf outside its bound"


@pytest.mark.parametrize("name", ["tiny_scm_f32", "scm_512x768_bf16", "stage3_1024x1792_bf16"])
def test_noise_rf_parity(name):
    wl = S.workload(name)
    inp = S.make_workload_inputs(wl)
    z0 = to_device(inp.z0, wl.dtype)
    eps = to_device(inp.eps, wl.dtype)
    t = torch.from_numpy(inp.t).cuda()
    zt, zrf = alloc_like(z0), alloc_like(z0)
    t_rf = torch.full((wl.batch,), float("nan"), device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    t2va.noise_rf(z0, eps, zt, zrf, t, t_rf=t_rf, status=status)
    plain = alloc_like(z0)
    t2va.noise(z0, eps, plain, t)
    torch.cuda.synchronize()
    assert status.item() == 0
    for a, b in zip(zt, plain):
        assert torch.equal(a, b), "z_t of the fused call differs from t2va_noise"
    got = to_host(zrf, wl.dtype)
    _check_rf(inp, got, t_rf.cpu().numpy(), inp.t)
    if wl.dtype == "bf16":
        # the rounded outputs differ from the oracle's only where the float32 error
        # crosses a rounding boundary (more than one ulp only where the two terms nearly
        # cancel, which the bound above allows)
        ref_zt, ref_zrf, ref_trf = oracle.noise_rf(inp.z0, inp.eps, inp.t, wl.dtype)
        for m in range(len(got)):
            d = ulp_diff_bf16(got[m], ref_zrf[m])
            assert (d > 0).mean() < 1e-3, \
                f"modality {m}: {(d > 0).mean():.2e} of elements differ from the oracle"


RAGGED = [(3, [1, 7], 0), (2, [9, 8191], 3), (5, [100003, 5], 1), (2, [33, 64, 1, 250001], 7)]


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
@pytest.mark.parametrize("case", RAGGED, ids=[f"B{b}-{'-'.join(map(str, n))}-p{p}" for b, n, p in RAGGED])
def test_noise_rf_ragged(dtype, case):
    """Heads and tails that are not whole 16-byte vectors, strided samples, one-chunk
    segments, the endpoints t = 0 and pi/2, and the RF output alone (zt = None)."""
    B, numels, pad = case
    inp = S.make_inputs(B, numels, dtype, S.SCM, seed=(500, B, len(numels), pad))
    t = inp.t.copy()
    t[0] = 0.0
    if B > 1:
        t[1] = np.float32(math.pi / 2)
    z0 = to_device(inp.z0, dtype, pad)
    eps = to_device(inp.eps, dtype, pad)
    tt = torch.from_numpy(t).cuda()
    zrf = alloc_like(z0, fill=7.0)
    t_rf = torch.full((B,), float("nan"), device="cuda")
    t2va.noise_rf(z0, eps, None, zrf, tt, t_rf=t_rf)
    torch.cuda.synchronize()
    _check_rf(inp, to_host(zrf, dtype), t_rf.cpu().numpy(), t)
    # the padding between strided samples is untouched
    if pad and B > 1:
        for x in zrf:
            gap = x.as_strided((B, x.stride(0) - x.shape[1]), (x.stride(0), 1), x.shape[1])
            assert torch.all(gap == 7.0)


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
@pytest.mark.parametrize("case", RAGGED, ids=[f"B{b}-{'-'.join(map(str, n))}-p{p}" for b, n, p in RAGGED])
def test_noise_zt_ragged_both_kernels(dtype, case):
    """z_t on the same ragged geometries, from the z_t-only kernel and from the kernel that
    writes z_t and z_rf together (their own instantiations, with their own register caps):
    z_t within the float32 evaluation bound of cos t z0 + sin t eps (one output ulp plus
    8 * 2^-24 of the magnitudes, as in the noise parity test), the two kernels' z_t equal
    bit for bit, z_rf within its bound, and the padding between strided samples untouched."""
    B, numels, pad = case
    inp = S.make_inputs(B, numels, dtype, S.SCM, seed=(503, B, len(numels), pad))
    z0 = to_device(inp.z0, dtype, pad)
    eps = to_device(inp.eps, dtype, pad)
    t = torch.from_numpy(inp.t).cuda()
    zt = alloc_like(z0, fill=7.0)
    zt2 = alloc_like(z0, fill=7.0)
    zrf = alloc_like(z0, fill=7.0)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    t2va.noise(z0, eps, zt, t, status=status)
    t2va.noise_rf(z0, eps, zt2, zrf, t, status=status)
    torch.cuda.synchronize()
    assert status.item() == 0
    got = to_host(zt, dtype)
    t64 = inp.t.astype(np.float64)[:, None]
    for m in range(len(got)):
        z = oracle.decode(inp.z0[m], dtype)
        e = oracle.decode(inp.eps[m], dtype)
        exact = np.cos(t64) * z + np.sin(t64) * e
        mag = np.abs(np.cos(t64) * z) + np.abs(np.sin(t64) * e)
        g = oracle.decode(got[m], dtype)
        bound = _ulp(exact, dtype) + 8 * 2.0 ** -24 * mag
        assert np.all(np.abs(g - exact) <= bound), \
            f"z_t modality {m}: worst {np.max(np.abs(g - exact) / bound):.2f} of bound"
    for a, b in zip(zt, zt2):
        assert torch.equal(a, b)
    _check_rf(inp, to_host(zrf, dtype), None, inp.t)
    if pad and B > 1:
        for x in zt + zt2 + zrf:
            gap = x.as_strided((B, x.stride(0) - x.shape[1]), (x.stride(0), 1), x.shape[1])
            assert torch.all(gap == 7.0)


def test_noise_rf_in_place_and_empty_modality():
    """z_rf written over z0 (in place), and t_rf written even when no modality has an
    element (the launch then has one CTA per sample)."""
    inp = S.make_inputs(4, [1000, 77], "bf16", S.SCM, seed=(501,))
    z0 = to_device(inp.z0, "bf16")
    eps = to_device(inp.eps, "bf16")
    t = torch.from_numpy(inp.t).cuda()
    ref = alloc_like(z0)
    t2va.noise_rf(z0, eps, None, ref, t)
    t2va.noise_rf(z0, eps, None, z0, t)
    torch.cuda.synchronize()
    for a, b in zip(z0, ref):
        assert torch.equal(a, b)
    empty = [torch.empty((4, 0), dtype=torch.bfloat16, device="cuda")]
    t_rf = torch.full((4,), float("nan"), device="cuda")
    t2va.noise_rf(empty, empty, None, [torch.empty((4, 0), dtype=torch.bfloat16, device="cuda")], t,
                  t_rf=t_rf)
    torch.cuda.synchronize()
    t64 = inp.t.astype(np.float64)
    exact = np.sin(t64) / (np.cos(t64) + np.sin(t64))
    assert np.all(np.abs(t_rf.cpu().numpy() - exact) <= 12 * 2.0 ** -24 * exact)


def test_noise_rf_errors():
    inp = S.make_inputs(2, [64, 16], "bf16", S.SCM, seed=(502,))
    z = to_device(inp.z0, "bf16")
    t = torch.from_numpy(inp.t).cuda()
    with pytest.raises(t2va.T2VAError) as e:
        t2va.noise_rf(z, z, z, z, t)          # z_t and z_rf the same buffers
    assert e.value.code == 1
    flat = torch.zeros(2 * 64 + 8, dtype=torch.bfloat16, device="cuda")
    mis = [flat[1:129].view(2, 64), z[1]]
    with pytest.raises(t2va.T2VAError) as e:
        t2va.noise_rf(z, z, None, mis, t)
    assert e.value.code == 3
