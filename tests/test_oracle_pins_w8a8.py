"""Pins of the W8A8 oracle (oracle/w8a8_oracle.py) against facts that do not come from
its own formulas: hand-made codes with exact scales, half-way ties, the dequantisation
error bound, pure-Python integer sums on small shapes, a closed form of the linear,
and planted mistakes that must each make a pin fail. CPU only."""

import importlib.util
import os

import numpy as np
import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
ORACLE_FILE = os.path.join(ROOT, "oracle", "w8a8_oracle.py")


def _load():
    spec = importlib.util.spec_from_file_location("w8a8_oracle_pinned", ORACLE_FILE)
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    return mod


W8 = _load()


def pin_codes_exact_scale(o):
    """amax = 127 gives s = 1 exactly, so the codes are the rounded values: ties go to
    even (2.5 -> 2, 3.5 -> 4, -2.5 -> -2), the largest element maps to +-127."""
    x = np.array([[127.0, 2.5, 3.5, -2.5, 0.49, -0.51, 126.5, -127.0]], np.float32)
    q, s = o.quantize_rows(x)
    assert s.dtype == np.float32 and s[0] == np.float32(1.0)
    assert q.dtype == np.int8
    assert q.tolist() == [[127, 2, 4, -2, 0, -1, 126, -127]]


def pin_scale_and_eps(o):
    """s = max(amax, 1e-4) / 127 in float32; an all-zero row and a row below eps both
    take the eps scale and give zero codes; scales are per row."""
    x = np.zeros((3, 16), np.float32)
    x[1, 3] = 5e-5
    x[2, :] = np.linspace(-3.0, 1.0, 16, dtype=np.float32)
    q, s = o.quantize_rows(x)
    eps_s = np.float32(1e-4) / np.float32(127)
    assert s[0] == eps_s and s[1] == eps_s
    assert np.all(q[0] == 0)
    assert q[1, 3] == int(np.rint(np.float32(5e-5) / eps_s))
    assert s[2] == np.float32(3.0) / np.float32(127)
    assert q[2, 0] == -127


def pin_dequant_bound(o):
    """|x - q s| <= s/2 (plus float32 rounding) on random rows of several scales."""
    r = np.random.default_rng(3)
    x = (r.standard_normal((64, 256)) * np.exp(r.uniform(-6, 6, (64, 1)))).astype(np.float32)
    q, s = o.quantize_rows(x)
    err = np.abs(x.astype(np.float64) - q.astype(np.float64) * s[:, None].astype(np.float64))
    assert np.all(err <= s[:, None] * (0.5 + 1e-5))
    assert np.all(np.abs(q).max(axis=1) == 127)


def pin_int_sum_brute_force(o):
    """acc_ij = sum_k xq_ik wq_jk by Python integer loops, non-square shapes so that a
    transposed operand cannot pass; y = sx_i sw_j acc_ij + b_j."""
    r = np.random.default_rng(5)
    M, N, K = 5, 3, 7
    xq = r.integers(-127, 128, (M, K)).astype(np.int8)
    wq = r.integers(-127, 128, (N, K)).astype(np.int8)
    sx = r.uniform(0.01, 1.0, M).astype(np.float32)
    sw = r.uniform(0.01, 1.0, N).astype(np.float32)
    b = r.standard_normal(N).astype(np.float32)
    acc, y = o.w8a8_linear(xq, sx, wq, sw, b)
    for i in range(M):
        for j in range(N):
            ref = sum(int(xq[i, k]) * int(wq[j, k]) for k in range(K))
            assert int(acc[i, j]) == ref
            assert abs(y[i, j] - (float(sx[i]) * float(sw[j]) * ref + float(b[j]))) <= 1e-12 * (1 + abs(y[i, j]))


def pin_int_sum_extremes(o):
    """All codes +-127 over K = 4096: the sum reaches 4096 * 16129 = 66,064,384 and stays
    exact (above float32's exact-integer range)."""
    K = 4096
    xq = np.full((2, K), 127, np.int8)
    xq[1, ::2] = -127
    wq = np.full((1, K), 127, np.int8)
    acc, _ = o.w8a8_linear(xq, np.ones(2, np.float32), wq, np.ones(1, np.float32))
    assert int(acc[0, 0]) == K * 127 * 127 and int(acc[1, 0]) == 0


def pin_forward_closed_form(o):
    """x_i = a_i * u with u's entries in {-1, 0, 1} and amax 127-multiples: codes are
    exactly 127 u, so y_ij = a_i s_j^w 127 (u . wq_j) / 127 + b_j = a_i s_j^w (u . wq_j) + b_j."""
    K = 128
    u = np.tile(np.array([1, -1, 0, 1], np.float32), K // 4)
    a = np.array([0.5, 2.0, 64.0], np.float32)
    x = a[:, None] * u[None, :]
    r = np.random.default_rng(7)
    wq = r.integers(-127, 128, (4, K)).astype(np.int8)
    sw = r.uniform(0.01, 0.1, 4).astype(np.float32)
    b = np.arange(4, dtype=np.float32)
    xq, sx, acc, y = o.w8a8_forward(x, wq, sw, b)
    assert np.array_equal(xq.astype(np.int64), 127 * np.tile(u.astype(np.int64), (3, 1)))
    dots = np.array([[int(np.dot(u.astype(np.int64), wq[j].astype(np.int64))) for j in range(4)]])
    ref = a[:, None].astype(np.float64) * sw[None, :].astype(np.float64) * dots + b[None, :]
    np.testing.assert_allclose(y, ref, rtol=1e-6)


PINS = [pin_codes_exact_scale, pin_scale_and_eps, pin_dequant_bound, pin_int_sum_brute_force,
        pin_int_sum_extremes, pin_forward_closed_form]


@pytest.mark.parametrize("pin", PINS, ids=[p.__name__ for p in PINS])
def test_w8a8_oracle_pin(pin):
    pin(W8)


def _mut_round_half_away(m):
    orig_scales = m.row_scales

    def q(x, eps=m.EPS):
        x32 = np.asarray(x, np.float32)
        s = orig_scales(x32, eps)
        v = x32 / s[:, None]
        return np.clip(np.sign(v) * np.floor(np.abs(v) + 0.5), -127, 127).astype(np.int8), s
    m.quantize_rows = q


def _mut_no_eps(m):
    m.row_scales = lambda x, eps=m.EPS: (np.max(np.abs(np.asarray(x, np.float32)), axis=1)
                                         / np.float32(127)).astype(np.float32)


def _mut_scale_255(m):
    m.row_scales = lambda x, eps=m.EPS: (np.maximum(np.max(np.abs(np.asarray(x, np.float32)), axis=1),
                                                    np.float32(eps)) / np.float32(255)).astype(np.float32)


def _mut_transposed_w(m):
    m.int_dot = lambda xq, wq: np.asarray(xq, np.int64) @ np.asarray(wq, np.int64).reshape(
        np.asarray(wq).shape[1], np.asarray(wq).shape[0])


def _mut_int16_wrap(m):
    m.int_dot = lambda xq, wq: (np.asarray(xq, np.int64) @ np.asarray(wq, np.int64).T).astype(np.int16).astype(np.int64)


def _mut_no_bias(m):
    orig = m.w8a8_linear
    m.w8a8_linear = lambda xq, sx, wq, sw, bias=None: orig(xq, sx, wq, sw, None)


def _mut_truncate(m):
    orig_scales = m.row_scales

    def q(x, eps=m.EPS):
        x32 = np.asarray(x, np.float32)
        s = orig_scales(x32, eps)
        return np.clip(np.trunc(x32 / s[:, None]), -127, 127).astype(np.int8), s
    m.quantize_rows = q


MUTANTS = {"round_half_away": _mut_round_half_away, "no_eps": _mut_no_eps, "scale_255": _mut_scale_255,
           "transposed_w": _mut_transposed_w, "int16_accumulator": _mut_int16_wrap,
           "bias_dropped": _mut_no_bias, "truncate": _mut_truncate}


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_w8a8_pins_catch_planted_mistakes(name):
    mod = _load()
    MUTANTS[name](mod)
    failed = []
    for pin in PINS:
        try:
            with np.errstate(all="ignore"):
                pin(mod)
        except (AssertionError, ValueError, FloatingPointError, IndexError):
            failed.append(pin.__name__)
    assert failed, f"planted mistake {name} was not caught"
