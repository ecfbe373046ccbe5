"""The objective's launch plan (t2va_objective_plan_query), checked on the CPU.

Both kernels of an objective call launch one CTA per chunk of every (sample, modality)
row; the plan fixes the chunk length, the chunks per row, and which chunk of a sample
writes its per-sample outputs. These tests check, for many geometries and SM counts,
the properties the kernels rely on (every vector of every row in exactly one chunk, at
most 1024 chunks per row, so the workspace holds every partial sum) and the ones the
performance rests on (one wave whenever the chunks can be kept to 2048 vectors: three
CTAs per SM less one slot per nine SMs, left free for the next kernel, with the shortest
such chunks; the per-sample outputs on the row end with the fewest vectors).
"""

import numpy as np
import pytest

import joint_video_audio_02_b300 as t2va
import synthetic as S
from joint_video_audio_02_b300 import binding
from joint_video_audio_02_b300.build import build

MAX_CHUNKS = 1024        # chunks per row the workspace holds (16 bytes each)
ONE_WAVE_MAX_VEC = 2048  # longest chunk of a one-wave plan
BATCH_VEC = 512          # vectors of one CTA batch (256 threads x 2)


@pytest.fixture(scope="module", autouse=True)
def _lib():
    build()
    t2va.load()


def _ve(dtype):
    return 8 if dtype == "bf16" else 4


def _check(batch, numels, dtype, sms):
    p = t2va.objective_plan(batch, numels, dtype, sms)
    ve = _ve(dtype)
    vpc = p["vectors_per_chunk"]
    nvec = [-(-n // ve) for n in numels]       # vectors of a row, rounded up
    chunks = p["chunks"]
    assert p["threads"] == 256
    assert vpc > 0 and vpc % 32 == 0
    assert p["grid"] == batch * sum(chunks)
    for m, (c, nv) in enumerate(zip(chunks, nvec)):
        assert 1 <= c <= MAX_CHUNKS, (m, c)
        assert c * vpc >= nv, "a row's vectors are not all covered"
        assert (c - 1) * vpc < max(nv, 1), "a chunk beyond the row's end"
    resident = 3 * sms
    wave = resident - sms // 9          # the slots a one-wave plan may fill
    total = batch * sum(nvec)
    assert p["one_wave"] == (p["grid"] <= resident)
    if total <= wave * ONE_WAVE_MAX_VEC:
        # one wave, with the shortest multiple of 32 that needs no more CTAs than that
        assert p["grid"] <= wave or vpc == ONE_WAVE_MAX_VEC
        if vpc > 32:
            shorter = vpc - 32
            g = batch * sum(max(1, -(-nv // shorter)) for nv in nvec)
            assert g > wave, "a shorter chunk would also fit in one wave"
    else:
        assert vpc % BATCH_VEC == 0
    # the per-sample outputs: a row's last chunk, the one with the fewest vectors
    om, oc = p["outputs_modality"], p["outputs_chunk"]
    assert 0 <= om < len(numels) and oc == chunks[om] - 1
    last = [nv - (c - 1) * vpc for c, nv in zip(chunks, nvec)]
    assert last[om] == min(last) and om == last.index(min(last))
    return p


@pytest.mark.parametrize("name", sorted(S.WORKLOADS))
def test_plan_of_every_workload(name):
    wl = S.workload(name)
    for sms in (148, 132, 16, 1):
        _check(wl.batch, wl.numels, wl.dtype, sms)


def test_plans_of_the_benchmark_shapes():
    """The plans the measurements are quoted on: 512x768 batch 4 and one 1024x1792 sample."""
    p = _check(4, [786432, 16128], "bf16", 148)
    assert (p["grid"], p["vectors_per_chunk"], p["chunks"]) == (424, 960, [103, 3])
    assert (p["outputs_modality"], p["outputs_chunk"]) == (1, 2)   # the audio row's 96-vector end
    p = _check(1, [3670016, 16128], "bf16", 148)
    assert (p["grid"], p["vectors_per_chunk"], p["chunks"]) == (424, 1088, [422, 2])
    assert p["one_wave"]


def test_plans_of_random_geometries():
    rng = np.random.default_rng(7)
    for _ in range(400):
        M = int(rng.integers(1, 5))
        batch = int(rng.integers(1, 65))
        numels = [int(x) for x in np.exp(rng.uniform(0, np.log(2e7), M)).astype(np.int64)]
        if rng.random() < 0.1:
            numels[int(rng.integers(0, M))] = 0
        dtype = "bf16" if rng.random() < 0.5 else "f32"
        sms = int(rng.choice([148, 132, 74, 8, 1]))
        _check(batch, numels, dtype, sms)


def test_rows_too_long_for_one_batch_per_chunk():
    """A 12M-element row needs more than 1024 one-batch chunks: its chunks grow to several
    512-vector batches so that the row still fits the workspace's 1024 entries."""
    p = _check(1, [12_000_000, 1000], "bf16", 148)
    assert p["vectors_per_chunk"] % BATCH_VEC == 0 and p["vectors_per_chunk"] >= 3 * BATCH_VEC
    p = _check(1, [400_000_000], "f32", 148)
    assert p["chunks"][0] <= MAX_CHUNKS


def test_plan_query_errors():
    with pytest.raises(t2va.T2VAError) as e:
        t2va.objective_plan(4, [100, 10], "bf16", 0)
    assert e.value.code == 1
    with pytest.raises(t2va.T2VAError) as e:
        t2va.objective_plan(4, [100, 10], "f16", 148)
    assert e.value.code == 2
    with pytest.raises(t2va.T2VAError) as e:
        t2va.objective_plan(4, [100, -1], "bf16", 148)
    assert e.value.code == 1
    with pytest.raises(t2va.T2VAError) as e:   # a stride shorter than the sample
        t2va.objective_plan(2, [100], "bf16", 148, sample_strides=[50])
    assert e.value.code == 1
    lib = binding.load()
    segs = (binding.Segment * 1)()
    segs[0].numel, segs[0].sample_stride = 10, 10
    assert lib.t2va_objective_plan_query(1, 1, segs, 1, 148, None) == 1
