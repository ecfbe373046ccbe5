"""The C-ABI library: builds, loads, exports every declared symbol, and rejects bad
arguments on the host before touching the device (runs without a GPU)."""

import ctypes
import os
import re

import pytest

import joint_video_audio_02_b300 as t2va
from joint_video_audio_02_b300 import binding
from joint_video_audio_02_b300.build import build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADERS = [os.path.join(ROOT, "include", f) for f in os.listdir(os.path.join(ROOT, "include")) if f.endswith(".h")]


def declared_functions():
    names = set()
    for h in HEADERS:
        src = open(h).read()
        src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
        for m in re.finditer(r"\b(t2va_\w+)\s*\(", src):
            names.add(m.group(1))
    return sorted(names)


@pytest.fixture(scope="module")
def lib():
    build()
    return binding.load()


def test_exports_every_declared_symbol(lib):
    names = declared_functions()
    assert names, "no declarations found"
    for n in names:
        assert hasattr(lib, n), f"{n} declared in include/ but not exported"
    assert set(names) == set(binding.EXPORTED)


def test_version_and_error_strings(lib):
    assert lib.t2va_abi_version() == 3
    for code in range(0, 7):
        assert len(t2va.error_string(code)) > 5


def _seg(n, s):
    segs = (binding.Segment * len(n))()
    for i, (a, b) in enumerate(zip(n, s)):
        segs[i].numel, segs[i].sample_stride = a, b
    return segs


def _p(*vals):
    return (ctypes.c_void_p * len(vals))(*vals)


def test_host_validation_without_device(lib):
    ok = 0x10000  # 16-byte aligned fake addresses: never dereferenced, every call below fails first
    segs = _seg([64, 16], [64, 16])
    ptrs = _p(ok, ok)
    # negative batch, bad modality count, bad geometry
    assert lib.t2va_noise(-1, 2, segs, 1, ptrs, ptrs, ptrs, ok, None, None) == 1
    assert lib.t2va_noise(2, 0, segs, 1, ptrs, ptrs, ptrs, ok, None, None) == 1
    assert lib.t2va_noise(2, 5, segs, 1, ptrs, ptrs, ptrs, ok, None, None) == 1
    assert lib.t2va_noise(2, 2, _seg([64, 16], [32, 16]), 1, ptrs, ptrs, ptrs, ok, None, None) == 1
    # unsupported dtype, misaligned and null pointers
    assert lib.t2va_noise(2, 2, segs, 7, ptrs, ptrs, ptrs, ok, None, None) == 2
    assert lib.t2va_noise(2, 2, segs, 1, _p(ok + 8, ok), ptrs, ptrs, ok, None, None) == 3
    assert lib.t2va_noise(2, 2, segs, 1, _p(0, ok), ptrs, ptrs, ok, None, None) == 1
    assert lib.t2va_noise(2, 2, segs, 1, ptrs, ptrs, ptrs, 0, None, None) == 1
    # empty batch is a no-op success
    assert lib.t2va_noise(0, 2, segs, 1, ptrs, ptrs, ptrs, ok, None, None) == 0
    w = (ctypes.c_float * 2)(1.0, 1.0)
    wbad = (ctypes.c_float * 2)(1.0, -1.0)
    args = lambda beta, gamma, eps, wt: (2, 2, segs, 1, ptrs, ptrs, ptrs, ptrs, ok, beta, gamma, eps, wt,
                                         1.0, ptrs, 0, ok, None, ok, 1 << 20, ok, None)
    assert lib.t2va_scm_objective(*args(1.0, 1.5, 1e-6, w)) == 1      # gamma > 1
    assert lib.t2va_scm_objective(*args(1.0, 0.5, 0.0, w)) == 1       # eps <= 0
    assert lib.t2va_scm_objective(*args(float("nan"), 0.5, 1e-6, w)) == 1
    assert lib.t2va_scm_objective(*args(1.0, 0.5, 1e-6, wbad)) == 1   # negative weight
    assert lib.t2va_dmd_objective(2, 2, segs, 1, ptrs, ptrs, ptrs, -1.0, w, 1.0, ptrs, 0, ok, None,
                                  ok, 1 << 20, ok, None) == 1
    # the fused RF noising: z_rf required, z_t optional but never the z_rf buffer
    assert lib.t2va_noise_rf(2, 2, segs, 1, ptrs, ptrs, None, None, ok, None, None, None) == 1
    assert lib.t2va_noise_rf(2, 2, segs, 1, ptrs, ptrs, ptrs, ptrs, ok, None, None, None) == 1
    assert lib.t2va_noise_rf(2, 2, segs, 1, ptrs, ptrs, None, _p(ok + 8, ok), ok, None, None, None) == 3
    assert lib.t2va_noise_rf(2, 2, segs, 1, ptrs, ptrs, None, ptrs, ok, ok + 2, None, None) == 3
    assert lib.t2va_noise_rf(0, 2, segs, 1, ptrs, ptrs, None, ptrs, ok, None, None, None) == 0
    # the guided stage-3 objective: the unconditional prediction and finite scales required
    g_ok = (ctypes.c_float * 2)(3.0, 5.0)
    g_bad = (ctypes.c_float * 2)(3.0, float("inf"))
    cfg = lambda uncond, g: (2, 2, segs, 1, ptrs, ptrs, ptrs, ptrs, ok, ptrs, ptrs, uncond, g, ptrs,
                             1.0, 0.5, 1e-6, 1e-6, w, 1.0, 1.0, ptrs, ptrs, 0, ok, None, None, None,
                             None, ok, 1 << 20, ok, None)
    assert lib.t2va_stage3_objective_cfg(*cfg(None, g_ok)) == 1
    assert lib.t2va_stage3_objective_cfg(*cfg(ptrs, None)) == 1
    assert lib.t2va_stage3_objective_cfg(*cfg(ptrs, g_bad)) == 1
    assert lib.t2va_stage3_objective_cfg(*cfg(_p(ok + 8, ok), g_ok)) == 3
    # W8A8: the paper's shape guard and the alignment rules are host checks
    a16 = 0x20000
    I8, BF = 2, 1
    assert lib.t2va_quantize_rows(4, 100, 1, a16, 100, 1e-4, I8, a16, 112, a16, None) == 1   # cols % 8
    assert lib.t2va_quantize_rows(4, 128, 1, a16, 128, 0.0, I8, a16, 128, a16, None) == 1    # eps <= 0
    assert lib.t2va_quantize_rows(4, 128, 1, a16, 120, 1e-4, I8, a16, 128, a16, None) == 1   # ld_x < cols
    assert lib.t2va_quantize_rows(4, 128, 1, a16 + 8, 128, 1e-4, I8, a16, 128, a16, None) == 3
    assert lib.t2va_quantize_rows(4, 128, 1, a16, 128, 1e-4, 0, a16, 128, a16, None) == 2    # float32 codes
    assert lib.t2va_quantize_rows(0, 128, 1, None, 128, 1e-4, BF, None, 128, None, None) == 0
    for M, N, K in ((100, 128, 128), (128, 96, 128), (128, 128, 192), (128, 128, 0), (128, 128, 131200)):
        for code in (I8, BF):
            assert lib.t2va_w8a8_linear(M, N, K, code, a16, a16, a16, a16, None, 0, a16, None, None) == 1
    assert lib.t2va_w8a8_linear(128, 128, 128, I8, a16 + 4, a16, a16, a16, None, 0, a16, None, None) == 3
    assert lib.t2va_w8a8_linear(128, 128, 128, BF, a16, a16, a16, a16, None, 0, a16 + 8, None, None) == 3
    assert lib.t2va_w8a8_linear(128, 128, 128, I8, a16, a16, a16, a16, None, 7, a16, None, None) == 2
    assert lib.t2va_w8a8_linear(128, 128, 128, 0, a16, a16, a16, a16, None, 0, a16, None, None) == 2
    assert lib.t2va_w8a8_linear(0, 128, 128, I8, None, None, None, None, None, 0, None, None, None) == 0
    # the fused residual + modulated normalisation
    assert lib.t2va_residual_modnorm(4, 100, 1, 1, a16, a16, None, None, None, 1e-6, None, a16 + 64, None) == 1  # D % 8
    assert lib.t2va_residual_modnorm(4, 128, 0, 1, a16, a16, None, None, None, 1e-6, None, a16 + 64, None) == 1  # rows/sample
    assert lib.t2va_residual_modnorm(4, 128, 1, 1, a16, None, a16, None, None, 1e-6, None, a16 + 64, None) == 1  # gate w/o u
    assert lib.t2va_residual_modnorm(4, 128, 1, 1, a16, None, None, None, None, 1e-6, a16, a16 + 64, None) == 1  # h' w/o u
    assert lib.t2va_residual_modnorm(4, 128, 1, 1, a16, a16 + 32, None, None, None, 1e-6, None, a16, None) == 1  # y is h
    assert lib.t2va_residual_modnorm(4, 128, 1, 1, a16, None, None, None, None, -1.0, None, a16 + 64, None) == 1
    assert lib.t2va_residual_modnorm(4, 128, 1, 1, a16 + 8, None, None, None, None, 1e-6, None, a16 + 64, None) == 3
    assert lib.t2va_residual_modnorm(4, 128, 1, 5, a16, None, None, None, None, 1e-6, None, a16 + 64, None) == 2
    assert lib.t2va_residual_modnorm(0, 128, 1, 1, None, None, None, None, None, 1e-6, None, None, None) == 0
    assert lib.t2va_selftest_wait_timeout(None, None) == 1
    assert lib.t2va_selftest_wait_timeout(a16 + 2, None) == 3
    # workspace checks come after the argument checks and need no device either
    assert lib.t2va_workspace_init(None, 1024, 0, None) == 4
    assert lib.t2va_workspace_init(ok + 4, 1024, 0, None) == 4


def test_load_fails_loudly_without_library(tmp_path):
    missing = str(tmp_path / "libt2va.so")
    saved = binding._LIB
    binding._LIB = None
    try:
        with pytest.raises(RuntimeError, match="not found"):
            binding.load(missing)
    finally:
        binding._LIB = saved
