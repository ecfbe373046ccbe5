"""GPU parity of the fused gated residual + modulated RMS normalisation
(t2va_residual_modnorm) against oracle/fused_ops_oracle.py.

Bound from the arithmetic. The kernel sums D squares in float32 (sequential fmas per
thread over D / 128 terms, then a 32-lane tree and the row's four warps), so the mean
square is within (D / 128 + 9) * 2^-24 of its exact value, relatively; the reciprocal
square root is correctly rounded after one rounded addition of eps; then one product, one
rounded 1 + scale and one fma. So
  |y - exact| <= 1 ulp_out(exact) + ((D / 128 + 9) / 2 + 5) * 2^-24 * (|h' r (1 + scale)| + |shift|).
With power-of-two gates h + gate * u is exact in float32, so the stored h' is the exactly
rounded h' and must match the oracle bit for bit; with other gates the bfloat16 h' is
rounded twice (to float32 by the fma, then to bfloat16) and may differ by one unit.
"""

import numpy as np
import pytest
import torch

import joint_video_audio_02_b300 as t2va
import oracle
import oracle.fused_ops_oracle as F
from joint_video_audio_02_b300.build import build

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    build()
    t2va.load()


def _round(dtype):
    if dtype == torch.bfloat16:
        return lambda v: oracle.decode(oracle.round_to_bf16_bits(np.asarray(v, np.float64)), "bf16")
    return lambda v: np.asarray(v, np.float64).astype(np.float32).astype(np.float64)


def _ulp(v, dtype):
    _, e = np.frexp(np.abs(v))
    bits = 8 if dtype == torch.bfloat16 else 24
    return np.ldexp(1.0, np.maximum(e - bits, -133 if dtype == torch.bfloat16 else -149))


def _case(seed, rows, D, samples, dtype, residual, pow2_gate=True, mods=True):
    r = np.random.default_rng(seed)
    h = (r.standard_normal((rows, D)) * np.exp(r.uniform(-2, 2, (rows, 1)))).astype(np.float32)
    u = r.standard_normal((rows, D)).astype(np.float32) if residual else None
    if residual:
        gate = (r.choice([0.25, 0.5, 1.0, 2.0], (samples, D)) if pow2_gate else r.uniform(-1, 1, (samples, D))).astype(np.float32)
    else:
        gate = None
    scale = r.uniform(-0.5, 0.5, (samples, D)).astype(np.float32) if mods else None
    shift = r.uniform(-0.3, 0.3, (samples, D)).astype(np.float32) if mods else None
    th = torch.from_numpy(h).to(dtype)
    tu = torch.from_numpy(u).to(dtype) if residual else None
    return th, tu, gate, scale, shift


def _run(th, tu, gate, scale, shift, eps, rps, store_h, in_place=False):
    dev = lambda a: None if a is None else torch.from_numpy(a).cuda()
    h = th.cuda()
    u = None if tu is None else tu.cuda()
    y = torch.empty_like(h)
    h_out = (h if in_place else torch.empty_like(h)) if store_h else None
    t2va.residual_modnorm(h, y, u=u, gate=dev(gate), scale=dev(scale), shift=dev(shift), eps=eps,
                          h_out=h_out, rows_per_sample=rps)
    torch.cuda.synchronize()
    return (None if h_out is None else h_out.float().cpu().numpy().astype(np.float64)), y.float().cpu().numpy().astype(np.float64)


def _check_y(y, h2, scale, shift, eps, rps, dtype):
    rows, D = h2.shape
    ms = np.mean(h2 * h2, axis=1, keepdims=True)
    rr = 1.0 / np.sqrt(ms + eps)
    sc = F.per_row(scale, rows, rps)
    sh = F.per_row(shift, rows, rps)
    mag = np.abs(h2 * rr * (1.0 + (0.0 if sc is None else sc))) + (0.0 if sh is None else np.abs(sh))
    _, exact = F.residual_modnorm(h2, None, None, scale, shift, eps, rps, None)
    bound = _ulp(exact, dtype) + ((D / 128 + 9) / 2 + 5) * 2.0 ** -24 * mag + 1e-30
    err = np.abs(y - exact)
    assert np.all(err <= bound), f"worst {np.max(err / bound):.2f} of bound"


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
@pytest.mark.parametrize("rows,D,samples", [(3, 8, 1), (7, 64, 7), (130, 4096, 2), (5, 12288, 5), (9, 1024, 3)])
def test_modnorm_without_residual(dtype, rows, D, samples):
    th, _, _, scale, shift = _case(rows * 31 + D, rows, D, samples, dtype, residual=False)
    rps = -(-rows // samples)
    _, y = _run(th, None, None, scale, shift, 1e-6, rps, store_h=False)
    h2 = th.float().numpy().astype(np.float64)
    _check_y(y, h2, scale, shift, 1e-6, rps, dtype)
    # no modulation at all: the plain normalisation
    _, y0 = _run(th, None, None, None, None, 1e-6, rps, store_h=False)
    _check_y(y0, h2, None, None, 1e-6, rps, dtype)


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
@pytest.mark.parametrize("rows,D,samples", [(4, 64, 2), (130, 4096, 1), (6, 12288, 3)])
def test_residual_modnorm_exact_residual(dtype, rows, D, samples):
    """Power-of-two gates: the stored h' is the exactly rounded h + gate u, bit for bit,
    and y is within the bound of the normalisation of that stored h'."""
    th, tu, gate, scale, shift = _case(rows * 7 + D, rows, D, samples, dtype, residual=True)
    rps = -(-rows // samples)
    h_out, y = _run(th, tu, gate, scale, shift, 1e-6, rps, store_h=True)
    ref_h2, _ = F.residual_modnorm(th.float().numpy(), tu.float().numpy(), gate, scale, shift, 1e-6, rps, _round(dtype))
    assert np.array_equal(h_out, ref_h2)
    _check_y(y, ref_h2, scale, shift, 1e-6, rps, dtype)
    # not storing h' (long rows then form it again in the second pass) gives the same y
    _, y2 = _run(th, tu, gate, scale, shift, 1e-6, rps, store_h=False)
    assert np.array_equal(y, y2)
    # in place: h' written over h
    h_in, y3 = _run(th, tu, gate, scale, shift, 1e-6, rps, store_h=True, in_place=True)
    assert np.array_equal(h_in, h_out) and np.array_equal(y3, y)


def test_residual_modnorm_general_gate():
    """Other gates: the bfloat16 h' is within one unit of the exactly rounded value (in a
    small fraction of elements), and y within the bound of the normalisation of the stored
    h' plus the effect of that unit."""
    dtype = torch.bfloat16
    th, tu, gate, scale, shift = _case(77, 64, 4096, 2, dtype, residual=True, pow2_gate=False)
    h_out, y = _run(th, tu, gate, scale, shift, 1e-6, 32, store_h=True)
    ref_h2, ref_y = F.residual_modnorm(th.float().numpy(), tu.float().numpy(), gate, scale, shift, 1e-6, 32, _round(dtype))
    diff = np.abs(h_out - ref_h2)
    assert np.all(diff <= _ulp(ref_h2, dtype) * 1.0 + 1e-30)
    assert (diff > 0).mean() < 1e-2
    ms = np.mean(ref_h2 * ref_h2, axis=1, keepdims=True)
    rr = 1.0 / np.sqrt(ms + 1e-6)
    sc = F.per_row(scale, 64, 32)
    mag = np.abs(ref_h2 * rr * (1 + sc)) + np.abs(F.per_row(shift, 64, 32))
    bound = 2 * _ulp(ref_y, dtype) + 1e-5 * mag + diff * rr * np.abs(1 + sc)
    assert np.all(np.abs(y - ref_y) <= bound)


def test_residual_modnorm_bench_size_sampled():
    """The benchmark's launch: 28,672 token rows x 4096 (the 1024x1792 video tokens), bf16,
    one sample's gate in [0, 1), scale and shift, h' stored. Rows sampled across the grid:
    h' within one unit of the exactly rounded value, y within the bound of the
    normalisation of the oracle's h' plus the effect of that unit."""
    rows, D = 28672, 4096
    r = np.random.default_rng(5)
    th = torch.from_numpy(r.standard_normal((rows, D), dtype=np.float32)).to(torch.bfloat16)
    tu = torch.from_numpy(r.standard_normal((rows, D), dtype=np.float32)).to(torch.bfloat16)
    gate = r.uniform(0, 1, (1, D)).astype(np.float32)
    scale = (r.uniform(0, 1, (1, D)) - 0.5).astype(np.float32)
    shift = (r.uniform(0, 1, (1, D)) - 0.5).astype(np.float32)
    h, u = th.cuda(), tu.cuda()
    y, h_out = torch.empty_like(h), torch.empty_like(h)
    dev = lambda a: torch.from_numpy(a).cuda()
    t2va.residual_modnorm(h, y, u=u, gate=dev(gate), scale=dev(scale), shift=dev(shift), eps=1e-6, h_out=h_out)
    torch.cuda.synchronize()
    rs = np.unique(np.concatenate([np.arange(0, rows, 487), [1, rows - 2, rows - 1]]))
    ri = torch.from_numpy(rs).cuda()
    got_h = h_out[ri].float().cpu().numpy().astype(np.float64)
    got_y = y[ri].float().cpu().numpy().astype(np.float64)
    n = len(rs)
    ref_h2, ref_y = F.residual_modnorm(th[rs].float().numpy(), tu[rs].float().numpy(), gate, scale, shift, 1e-6, n,
                                       _round(torch.bfloat16))
    diff = np.abs(got_h - ref_h2)
    assert np.all(diff <= _ulp(ref_h2, torch.bfloat16) + 1e-30)
    assert (diff > 0).mean() < 1e-2
    ms = np.mean(ref_h2 * ref_h2, axis=1, keepdims=True)
    rr = 1.0 / np.sqrt(ms + 1e-6)
    sc, sh = F.per_row(scale, n, n), F.per_row(shift, n, n)
    mag = np.abs(ref_h2 * rr * (1 + sc)) + np.abs(sh)
    bound = 2 * _ulp(ref_y, torch.bfloat16) + 1e-5 * mag + diff * rr * np.abs(1 + sc)
    assert np.all(np.abs(got_y - ref_y) <= bound)


def test_residual_modnorm_errors():
    h = torch.zeros((4, 128), dtype=torch.bfloat16, device="cuda")
    with pytest.raises(t2va.T2VAError) as e:
        t2va.residual_modnorm(h, h)                               # y is h
    assert e.value.code == 1
    with pytest.raises(t2va.T2VAError) as e:
        t2va.residual_modnorm(h, torch.empty_like(h), h_out=torch.empty_like(h))   # h' without u
    assert e.value.code == 1
