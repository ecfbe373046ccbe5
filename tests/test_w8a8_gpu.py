"""GPU parity of the post-scale W8A8 linear (t2va_quantize_rows, t2va_w8a8_linear)
against the oracle in oracle/w8a8_oracle.py, for both contractions: int8 codes on the
warp-level INT8 MMA, and the same codes stored as bfloat16 integers on the tcgen05
tensor cores (float32 sums over K chunks of 1024, below 2^24, added as int32).

Codes and scales are integers and float32 values decided in float32 on both sides, so
they must match bit for bit. The integer sums are exact: with float32 output and unit
scales y equals the sum exactly while |sum| < 2^24. The epilogue
y = fma(float(acc), sx * sw, b) rounds float(acc) (once, only past 2^24), sx * sw and the
fma, so |y - exact| <= 4 * 2^-24 (|sx sw acc| + |b|), plus one output ulp for bfloat16.
"""

import time

import numpy as np
import pytest
import torch

import joint_video_audio_02_b300 as t2va
import oracle.w8a8_oracle as W8
from joint_video_audio_02_b300.build import build

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    build()
    t2va.load()


def _ulp_bf16(v):
    _, e = np.frexp(np.abs(v))
    return np.ldexp(1.0, np.maximum(e - 8, -133))


def _rows(seed, M, K, dtype):
    r = np.random.default_rng(seed)
    x = (r.standard_normal((M, K)) * np.exp(r.uniform(-4, 4, (M, 1)))).astype(np.float32)
    x[0, :] = 0.0                                   # an all-zero row: the eps scale
    if M > 1:
        x[1, :] = 0.0
        x[1, : min(K, 8)] = np.array([127.0, 2.5, 3.5, -2.5, 0.5, -0.5, 1.5, 126.5], np.float32)[: min(K, 8)]
    if M > 2:
        x[2, :] *= 1e-9                             # below eps
    t = torch.from_numpy(x)
    if dtype == torch.bfloat16:
        t = t.to(torch.bfloat16)
    return t


CODES = [torch.int8, torch.bfloat16]


@pytest.mark.parametrize("code", CODES, ids=["int8", "bf16codes"])
@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
@pytest.mark.parametrize("M,K,pad", [(3, 8, 0), (5, 4096, 0), (7, 12352, 0), (6, 1024, 16), (130, 256, 8)])
def test_quantize_rows_bit_exact(code, dtype, M, K, pad):
    if dtype == torch.float32 and K % 4:
        pytest.skip("float32 rows are whole 16-byte vectors")
    x_host = _rows(M * 1000 + K, M, K, dtype)
    xbuf = torch.zeros((M, K + pad), dtype=dtype, device="cuda")
    xbuf[:, :K] = x_host.cuda()
    x = xbuf[:, :K]
    qbuf = torch.full((M, K + 16 * (pad > 0)), 99, dtype=code, device="cuda")
    q = qbuf[:, :K]
    s = torch.empty(M, device="cuda")
    t2va.quantize_rows(x, q, s)
    torch.cuda.synchronize()
    ref_q, ref_s = W8.quantize_rows(x_host.float().numpy())
    assert np.array_equal(s.cpu().numpy().view(np.uint32), ref_s.view(np.uint32))
    got = q.cpu().float().numpy() if code == torch.bfloat16 else q.cpu().numpy()
    assert np.array_equal(got, ref_q.astype(got.dtype))
    if pad:
        assert torch.all(qbuf[:, K:] == 99)


def test_quantize_codes_at_rounding_boundaries():
    """Values at and within 3 ulps of (k + 1/2) s for random scales: the kernel forms the
    quotient only near such boundaries, and its codes must still be those of the float32
    quotient rounded half to even."""
    r = np.random.default_rng(31)
    M, K = 64, 1024
    amax = r.uniform(0.1, 100.0, M).astype(np.float32)
    s = (amax / np.float32(127)).astype(np.float32)
    k = r.integers(-126, 126, (M, K)).astype(np.float32)
    x = ((k + np.float32(0.5)) * s[:, None]).astype(np.float32)
    xi = x.view(np.int32)
    xi += r.integers(-3, 4, (M, K)).astype(np.int32)
    x[:, 0] = amax                                   # the row maximum, so the scale is s
    xd = torch.from_numpy(x).cuda()
    q = torch.empty((M, K), dtype=torch.int8, device="cuda")
    sc = torch.empty(M, device="cuda")
    t2va.quantize_rows(xd, q, sc)
    torch.cuda.synchronize()
    ref_q, ref_s = W8.quantize_rows(x)
    assert np.array_equal(sc.cpu().numpy(), ref_s)
    assert np.array_equal(q.cpu().numpy(), ref_q)


def _codes(seed, R, K, extreme=False):
    r = np.random.default_rng(seed)
    q = r.integers(-127, 128, (R, K)).astype(np.int8)
    if extreme:
        q[0, :] = 127
        q[1, :] = -127
    return q


def _check_linear(y, acc, sx, sw, b, out_dtype):
    exact = (sx.astype(np.float64)[:, None] * sw.astype(np.float64)[None, :]) * acc
    mag = np.abs(exact)
    if b is not None:
        exact = exact + b.astype(np.float64)[None, :]
        mag = mag + np.abs(b.astype(np.float64))[None, :]
    bound = 4 * 2.0 ** -24 * mag + 1e-30
    if out_dtype == torch.bfloat16:
        bound = bound + _ulp_bf16(exact)
    err = np.abs(y.astype(np.float64) - exact)
    assert np.all(err <= bound), f"worst {np.max(err / bound):.2f} of bound"


def _dev_codes(q, code):
    t = torch.from_numpy(q).cuda()
    return t.to(torch.bfloat16) if code == torch.bfloat16 else t


@pytest.mark.parametrize("code", CODES, ids=["int8", "bf16codes"])
@pytest.mark.parametrize("out_dtype", [torch.float32, torch.bfloat16])
@pytest.mark.parametrize("M,N,K,bias", [(128, 128, 128, True), (256, 384, 512, False),
                                        (384, 256, 4096, True), (128, 640, 1152, True),
                                        (256, 128, 8192, False), (128, 256, 8192, True),
                                        (256, 512, 2048, False)])
def test_w8a8_linear_parity(code, out_dtype, M, N, K, bias):
    xq = _codes(M + K, M, K, extreme=True)
    wq = _codes(N + K + 1, N, K, extreme=True)
    r = np.random.default_rng(K)
    sx = r.uniform(1e-4, 0.05, M).astype(np.float32)
    sw = r.uniform(1e-4, 0.05, N).astype(np.float32)
    b = r.standard_normal(N).astype(np.float32) if bias else None
    y = torch.empty((M, N), dtype=out_dtype, device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    t2va.w8a8_linear(_dev_codes(xq, code), torch.from_numpy(sx).cuda(), _dev_codes(wq, code),
                     torch.from_numpy(sw).cuda(), y, None if b is None else torch.from_numpy(b).cuda(),
                     status=st)
    torch.cuda.synchronize()
    assert st.item() == 0
    acc, _ = W8.w8a8_linear(xq, sx, wq, sw, b)
    _check_linear(y.float().cpu().numpy(), acc, sx, sw, b, out_dtype)


@pytest.mark.parametrize("out_dtype", [torch.float32, torch.bfloat16])
def test_w8a8_wide_tiles_more_than_one_per_sm(out_dtype):
    """N divisible by 256 takes the persistent 128 x 256 tensor-core kernel. 20 x 8 = 160
    tiles on at most 148 CTAs: some CTAs run two tiles, their accumulators continuing the
    ring across tiles, and K = 1152 ends each tile with a partial chunk. Rows sampled in
    every TMEM lane quadrant of every row tile, all columns (both halves of each tile),
    against the oracle's exact sums."""
    M, N, K = 2560, 2048, 1152
    xq = _codes(71, M, K, extreme=True)
    wq = _codes(72, N, K, extreme=True)
    r = np.random.default_rng(73)
    sx = r.uniform(1e-4, 0.05, M).astype(np.float32)
    sw = r.uniform(1e-4, 0.05, N).astype(np.float32)
    b = r.standard_normal(N).astype(np.float32)
    y = torch.empty((M, N), dtype=out_dtype, device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    t2va.w8a8_linear(_dev_codes(xq, torch.bfloat16), torch.from_numpy(sx).cuda(), _dev_codes(wq, torch.bfloat16),
                     torch.from_numpy(sw).cuda(), y, torch.from_numpy(b).cuda(), status=st)
    torch.cuda.synchronize()
    assert st.item() == 0
    rows = np.array([t * 128 + o for t in range(M // 128) for o in (0, 1, 45, 70, 127)])
    acc, _ = W8.w8a8_linear(xq[rows], sx[rows], wq, sw, b)
    _check_linear(y.float().cpu().numpy()[rows], acc, sx[rows], sw, b, out_dtype)


@pytest.mark.parametrize("code", CODES, ids=["int8", "bf16codes"])
def test_w8a8_integer_sum_exact(code):
    """Unit scales, no bias, float32 output: y is the integer sum itself while |sum| < 2^24,
    so every output must equal the oracle's sum exactly, tile edges included. K = 1024
    holds one full chunk of the tensor-core path at its largest possible magnitude,
    1024 x 127 x 127 = 16,516,096 (just below 2^24); K = 3072 adds chunks of opposite
    sign that must cancel exactly."""
    one = lambda n: torch.ones(n, device="cuda")
    for K in (1024, 3072):
        M, N = 256, 256
        xq, wq = _codes(11 + K, M, K, extreme=True), _codes(12 + K, N, K, extreme=True)
        if K == 3072:
            wq[2, :1024], wq[2, 1024:2048], wq[2, 2048:] = 127, -127, 0   # +16.5M, -16.5M, 0
            xq[0, :] = 127
        y = torch.empty((M, N), device="cuda")
        st = torch.zeros(1, dtype=torch.int32, device="cuda")
        t2va.w8a8_linear(_dev_codes(xq, code), one(M), _dev_codes(wq, code), one(N), y, status=st)
        torch.cuda.synchronize()
        assert st.item() == 0
        acc = W8.int_dot(xq, wq)
        ok = np.abs(acc) < 2 ** 24
        assert np.array_equal(y.cpu().numpy().astype(np.int64)[ok], acc[ok])
        if K == 1024:
            assert int(acc[0, 0]) == K * 127 * 127 and int(acc[1, 0]) == -K * 127 * 127
        else:
            assert int(acc[0, 2]) == 0 and float(y[0, 2]) == 0.0


@pytest.mark.parametrize("code", CODES, ids=["int8", "bf16codes"])
def test_w8a8_forward_matches_oracle(code):
    """bf16 activations -> quantise -> linear against pre-quantised weights, the whole
    operator, against the oracle's codes, scales and exact output."""
    M, N, K = 256, 384, 2048
    r = np.random.default_rng(21)
    x = torch.from_numpy(r.standard_normal((M, K)).astype(np.float32)).to(torch.bfloat16)
    w = r.standard_normal((N, K)).astype(np.float32) * 0.02
    wq, sw = W8.quantize_rows(w)
    b = r.standard_normal(N).astype(np.float32) * 0.1
    xd = x.cuda()
    q = torch.empty((M, K), dtype=code, device="cuda")
    sx = torch.empty(M, device="cuda")
    t2va.quantize_rows(xd, q, sx)
    y = torch.empty((M, N), dtype=torch.bfloat16, device="cuda")
    t2va.w8a8_linear(q, sx, _dev_codes(wq, code), torch.from_numpy(sw).cuda(), y,
                     torch.from_numpy(b).cuda())
    torch.cuda.synchronize()
    ref_xq, ref_sx, acc, _ = W8.w8a8_forward(x.float().numpy(), wq, sw, b)
    assert np.array_equal(q.cpu().float().numpy().astype(np.int64), ref_xq.astype(np.int64))
    assert np.array_equal(sx.cpu().numpy(), ref_sx)
    _check_linear(y.float().cpu().numpy(), acc, ref_sx, sw, b, torch.bfloat16)


def test_w8a8_bench_size_sampled():
    """The operator at the benchmark's size and launch: x [28672, 4096] bf16 (the
    1024x1792 video tokens) quantised per row on the device to bf16 codes, weights
    [4096, 4096] quantised once by the oracle, bias, bf16 out, through the persistent
    128 x 256 tensor-core kernel. Rows sampled from every other row tile, in every TMEM
    lane quadrant: their codes and scales bit for bit, their outputs within the bound of
    the oracle's exact sums."""
    M, N, K = 28672, 4096, 4096
    r = np.random.default_rng(31)
    tx = torch.from_numpy(r.standard_normal((M, K), dtype=np.float32)).to(torch.bfloat16)
    w = r.standard_normal((N, K), dtype=np.float32) * 0.02
    wq, sw = W8.quantize_rows(w)
    b = (r.standard_normal(N) * 0.1).astype(np.float32)
    q = torch.empty((M, K), dtype=torch.bfloat16, device="cuda")
    sx = torch.empty(M, device="cuda")
    t2va.quantize_rows(tx.cuda(), q, sx)
    y = torch.empty((M, N), dtype=torch.bfloat16, device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    t2va.w8a8_linear(q, sx, _dev_codes(wq, torch.bfloat16), torch.from_numpy(sw).cuda(), y,
                     torch.from_numpy(b).cuda(), status=st)
    torch.cuda.synchronize()
    assert st.item() == 0
    rows = np.array([t * 128 + (37 * t) % 128 for t in range(0, M // 128, 2)])
    ref_xq, ref_sx, acc, _ = W8.w8a8_forward(tx[rows].float().numpy(), wq, sw, b)
    ri = torch.from_numpy(rows).cuda()
    assert np.array_equal(q[ri].float().cpu().numpy().astype(np.int64), ref_xq.astype(np.int64))
    assert np.array_equal(sx[ri].cpu().numpy(), ref_sx)
    _check_linear(y[ri].float().cpu().numpy(), acc, ref_sx, sw, b, torch.bfloat16)


def test_w8a8_guard():
    z = torch.zeros((100, 128), dtype=torch.int8, device="cuda")
    with pytest.raises(t2va.T2VAError) as e:
        t2va.w8a8_linear(z, torch.ones(100, device="cuda"), torch.zeros((128, 128), dtype=torch.int8, device="cuda"),
                         torch.ones(128, device="cuda"), torch.empty((100, 128), device="cuda"))
    assert e.value.code == 1


def test_bounded_wait_runs_out_and_context_survives():
    """The tensor-core kernel's waits are bounded: in the self-test launch one wait is on a
    barrier nothing arrives on. It must end by itself with T2VA_STATUS_TIMEOUT, free its
    resources, and leave the context usable; a later launch given the flagged status word
    does nothing, and one given a clear word computes as usual."""
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    t0 = time.time()
    t2va.selftest_wait_timeout(st)
    torch.cuda.synchronize()
    assert st.item() & t2va.STATUS_TIMEOUT
    assert time.time() - t0 < 60
    M = N = K = 128
    xq, wq = _codes(41, M, K, extreme=True), _codes(42, N, K)
    one = lambda n: torch.ones(n, device="cuda")
    y = torch.full((M, N), -1.0, device="cuda")
    t2va.w8a8_linear(_dev_codes(xq, torch.bfloat16), one(M), _dev_codes(wq, torch.bfloat16), one(N), y, status=st)
    torch.cuda.synchronize()
    assert torch.all(y == -1.0)                      # skipped: the word still holds the timeout
    yw = torch.full((M, 2 * N), -1.0, device="cuda")  # N = 256: the wide kernel skips as well
    wq2 = np.concatenate([wq, wq])
    t2va.w8a8_linear(_dev_codes(xq, torch.bfloat16), one(M), _dev_codes(wq2, torch.bfloat16), one(2 * N), yw,
                     status=st)
    torch.cuda.synchronize()
    assert torch.all(yw == -1.0)
    st.zero_()
    t2va.w8a8_linear(_dev_codes(xq, torch.bfloat16), one(M), _dev_codes(wq, torch.bfloat16), one(N), y, status=st)
    torch.cuda.synchronize()
    assert st.item() == 0
    assert np.array_equal(y.cpu().numpy().astype(np.int64), W8.int_dot(xq, wq))
    t2va.w8a8_linear(_dev_codes(xq, torch.bfloat16), one(M), _dev_codes(wq2, torch.bfloat16), one(2 * N), yw,
                     status=st)
    torch.cuda.synchronize()
    assert st.item() == 0
    assert np.array_equal(yw.cpu().numpy().astype(np.int64), W8.int_dot(xq, wq2))
