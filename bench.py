"""Benchmark of the joint video-audio distillation objective on B300.

One step = one pass of the whole hot path over one batch of synthetic inputs:
TrigFlow noising of (z0, eps) and of (zhat0, eps'), then the fused stage-3
sCM + DMD objective (forward + gradient), all through the C ABI. The default
workload is the 512x768 stage-3 shape (B=4, video [128,16,16,24], audio
[126,128], bf16 inputs, float32 gradients). The workload stage3_cfg_rf_512x768_bf16
extends the step with the rectified-flow wrapper in the noising (z_rf and t_rf
written beside z_t) and a guided DMD teacher (conditional and unconditional
predictions read in place of one).

Prints one JSON line. `value` is the whole-job throughput in GB/s of algorithmic
HBM bytes (each input read once, each output written once) with inputs resident
in device memory; `roofline` describes the dominant kernel (the fused objective),
timed live as back-to-back launches of a captured graph with CUDA events around
the region on the launching stream; `e2e` is the
same metric with host buffers (pinned host -> device copies of the inputs and
device -> host copies of the gradients and losses inside the timed region);
`cpu_baseline` is the float64 CPU oracle timed on a bounded sample.

`--impl reference` times the CPU oracle itself as the reference arm.
"""

from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import statistics
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import synthetic as S  # noqa: E402

METRIC = "fused joint sCM+DMD objective GB/s (fwd+grad) and % of B300 HBM peak"
UNIT = "GB/s"
DEFAULT_WORKLOAD = "stage3_512x768_bf16"
FALLBACK_HBM_GBS = 6400.0
OBJECTIVE_SOURCES = ["joint_video_audio_02_b300/csrc/t2va_objective.cu",
                     "joint_video_audio_02_b300/csrc/t2va_internal.cuh"]
TRAFFIC_FILE = "profiles/stage3_objective_512x768_traffic.txt"


# ---------------------------------------------------------------------------
# algorithmic bytes
# ---------------------------------------------------------------------------

def elem_size(dtype: str) -> int:
    return {"bf16": 2, "f32": 4}[dtype]


def bytes_per_element(call: str, dtype: str) -> int:
    """Each input read once, each output written once; gradients are float32."""
    e = elem_size(dtype)
    return {"noise": 3 * e, "noise_rf": 4 * e, "scm": 4 * e + 4, "dmd": 3 * e + 4,
            "stage3": 7 * e + 2 * 4, "stage3_cfg": 8 * e + 2 * 4}[call]


def is_stage3(wl: S.Workload) -> bool:
    return wl.mode in (S.STAGE3, S.STAGE3_CFG)


def step_bytes(wl: S.Workload) -> dict:
    n = wl.batch * sum(wl.numels)
    out = {"elements": n}
    nz = bytes_per_element("noise_rf" if wl.rf_wrapper else "noise", wl.dtype)
    if is_stage3(wl):
        out["noise"] = 2 * n * nz + (2 * 4 * wl.batch if wl.rf_wrapper else 0)
        out["objective"] = n * bytes_per_element(wl.mode, wl.dtype)
    elif wl.mode == S.SCM:
        out["noise"] = n * nz + (4 * wl.batch if wl.rf_wrapper else 0)
        out["objective"] = n * bytes_per_element("scm", wl.dtype)
    else:
        out["noise"] = 0
        out["objective"] = n * bytes_per_element("dmd", wl.dtype)
    out["step"] = out["noise"] + out["objective"]
    return out


def input_fields(wl: S.Workload) -> list:
    """The host inputs of one step, per modality (the timesteps apart)."""
    f = ["z0", "eps", "x0_teacher", "x0_student", "x0_tangent"]
    if is_stage3(wl):
        f += ["zhat0", "eps_hat", "x0_teacher_hat", "x0_fake"]
    if wl.mode == S.STAGE3_CFG:
        f += ["x0_teacher_hat_uncond"]
    return f


def measured_peak():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(p) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


def objective_source_hash() -> str:
    h = hashlib.sha256()
    for rel in OBJECTIVE_SOURCES:
        with open(os.path.join(ROOT, rel), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def committed_traffic(workload: str):
    """DRAM bytes per launch of the objective kernel from the committed ncu summary,
    if it was taken on the current kernel source and this workload; else None."""
    try:
        kv = {}
        with open(os.path.join(ROOT, TRAFFIC_FILE)) as f:
            for line in f:
                if ":" in line:
                    k, v = line.split(":", 1)
                    kv[k.strip()] = v.strip()
        if kv.get("kernel_source_sha256") != objective_source_hash() or kv.get("workload") != workload:
            return None
        return float(kv["dram_bytes_per_launch"])
    except Exception:
        return None


# ---------------------------------------------------------------------------
# multi-rank host logic (one process per GPU; samples are sharded by rank)
# ---------------------------------------------------------------------------

def rank_seed_offset(rank: int, input_set: int) -> int:
    """Seed key suffix of input set `input_set` on `rank`: every rank draws its own samples."""
    return 1000 * rank + input_set


def max_over_ranks(ms: float, dist, device) -> float:
    """The slowest rank's time: the whole job ends when its last rank ends."""
    if dist is None:
        return float(ms)
    import torch
    tt = torch.tensor([float(ms)], device=device, dtype=torch.float64)
    dist.all_reduce(tt, op=dist.ReduceOp.MAX)
    return float(tt.item())


def whole_job_gbs(world: int, bytes_per_step_per_rank: int, steps: int, ms: float) -> float:
    """Algorithmic bytes of all ranks' steps over the (max-over-ranks) time, in GB/s."""
    return world * bytes_per_step_per_rank * steps / (ms * 1e-3) / 1e9


# ---------------------------------------------------------------------------
# clocks during the timed region
# ---------------------------------------------------------------------------

class ClockSampler:
    """SM clock and clock-event reasons sampled in a background thread (NVML, looked up
    by the CUDA device's UUID), or by an `nvidia-smi -lms` subprocess if NVML fails."""

    REASONS = {
        0x1: "gpu_idle", 0x2: "applications_clocks_setting", 0x4: "sw_power_cap",
        0x8: "hw_slowdown", 0x10: "sync_boost", 0x20: "sw_thermal_slowdown",
        0x40: "hw_thermal_slowdown", 0x80: "hw_power_brake_slowdown", 0x100: "display_clock_setting",
    }
    SMI_FIELDS = "timestamp,clocks.sm,clocks.max.sm,clocks_event_reasons.active"

    def __init__(self, uuid: str, period_s: float = 0.005):
        self.samples = []          # (wall time, sm MHz, reason bits)
        self.period = period_s
        self.stop_evt = threading.Event()
        self.error = ""
        self.max_mhz = None
        self.uuid = uuid
        self.proc = None
        try:
            import pynvml
            pynvml.nvmlInit()
            self.nv = pynvml
            self.h = pynvml.nvmlDeviceGetHandleByUUID(uuid)
            self.max_mhz = pynvml.nvmlDeviceGetMaxClockInfo(self.h, pynvml.NVML_CLOCK_SM)
            pynvml.nvmlDeviceGetCurrentClocksEventReasons(self.h)
            self.mode = "nvml"
        except Exception as e:  # fall back to nvidia-smi
            self.error = f"nvml: {type(e).__name__}: {e}"[:160]
            self.mode = "smi"
        self.thread = threading.Thread(target=self._run, daemon=True)

    def _run(self):
        while not self.stop_evt.is_set():
            try:
                mhz = self.nv.nvmlDeviceGetClockInfo(self.h, self.nv.NVML_CLOCK_SM)
                rs = self.nv.nvmlDeviceGetCurrentClocksEventReasons(self.h)
                self.samples.append((time.time(), mhz, int(rs)))
            except Exception:
                pass
            time.sleep(self.period)

    def start(self):
        if self.mode == "nvml":
            self.thread.start()
            return
        import subprocess
        import tempfile
        self.smi_out = tempfile.NamedTemporaryFile("w+", suffix=".csv", delete=False)
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", self.uuid, f"--query-gpu={self.SMI_FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "50"],
                stdout=self.smi_out, stderr=subprocess.DEVNULL)
            time.sleep(0.5)
        except Exception as e:
            self.error += f"; smi: {e}"[:160]
            self.proc = None

    def stop(self):
        self.stop_evt.set()
        if self.mode == "nvml":
            self.thread.join()
            return
        if self.proc is None:
            return
        import datetime
        self.proc.terminate()
        self.proc.wait()
        self.smi_out.seek(0)
        for line in self.smi_out:
            parts = [x.strip() for x in line.split(",")]
            if len(parts) < 4:
                continue
            try:
                ts = datetime.datetime.strptime(parts[0], "%Y/%m/%d %H:%M:%S.%f").timestamp()
                self.samples.append((ts, float(parts[1]), int(parts[3], 16)))
                self.max_mhz = float(parts[2])
            except Exception:
                continue
        os.unlink(self.smi_out.name)

    def summary(self, t0: float, t1: float) -> dict:
        if not self.samples:
            return {"sm_mhz": None, "sm_max_mhz": self.max_mhz, "reasons": ["no_samples"],
                    "samples": 0, "source": self.mode, "note": self.error}
        inside = [x for x in self.samples if t0 <= x[0] <= t1]
        n_inside = len(inside)
        if not inside:   # region shorter than the sampling period: nearest sample
            mid = 0.5 * (t0 + t1)
            inside = [min(self.samples, key=lambda x: abs(x[0] - mid))]
        bits = 0
        for x in inside:
            bits |= x[2]
        reasons = sorted({name for b, name in self.REASONS.items() if bits & b and b != 0x1})
        out = {"sm_mhz": statistics.median([x[1] for x in inside]), "sm_max_mhz": self.max_mhz,
               "reasons": reasons, "samples": n_inside, "source": self.mode}
        if self.error:
            out["note"] = self.error
        return out


# ---------------------------------------------------------------------------
# GPU arm
# ---------------------------------------------------------------------------

EXTRA_SHAPES = ["stage3_1024x1792_bf16", "stage3_sweep_b1_bf16", "stage3_sweep_b4_bf16",
                "stage3_sweep_b16_bf16", "stage3_sweep_b32_bf16", "scm_512x768_bf16"]


def objective_rooflines(names, dev, cap_stream, n_launch, l2, peak):
    """The objective alone at other shapes, timed as the roofline kernel is: a CUDA graph
    of `n_launch` back-to-back calls over input sets that together exceed 3x L2, replayed
    once untimed and then timed with CUDA events on the launching stream. The inputs
    are drawn on the device (N(0, 1), t uniform in [0.05, 1.45]): the kernels' work does
    not depend on the values."""
    import torch

    import joint_video_audio_02_b300 as t2va

    out = {}
    for name in names:
        w = S.workload(name)
        tdt = torch.bfloat16 if w.dtype == "bf16" else torch.float32
        n_el = w.batch * sum(w.numels)
        scm_only = w.mode == S.SCM
        nbytes = n_el * bytes_per_element("scm" if scm_only else "stage3", w.dtype)
        R = max(2, math.ceil(3 * l2 / (nbytes + 2 * n_el * elem_size(w.dtype))))
        g = torch.Generator(device=dev)
        g.manual_seed(1234)
        sets = []
        for _ in range(R):
            d = {f: [torch.randn(w.batch, n, device=dev, generator=g).to(tdt) for n in w.numels]
                 for f in ("zt", "xT", "xS", "tan", "zh", "yT", "yF")}
            d["gS"] = [torch.empty(w.batch, n, device=dev) for n in w.numels]
            d["gD"] = [torch.empty(w.batch, n, device=dev) for n in w.numels]
            d["t"] = torch.rand(w.batch, device=dev, generator=g) * 1.4 + 0.05
            d["loss"] = torch.empty(w.batch, device=dev)
            sets.append(d)
        ws = t2va.new_workspace(w.batch, w.num_modalities)
        st = torch.zeros(1, dtype=torch.int32, device=dev)

        def call(d):
            if scm_only:
                t2va.scm_objective(d["zt"], d["xT"], d["xS"], d["tan"], d["t"], beta=w.beta,
                                   gamma=w.gamma, eps_scm=w.eps_scm, weight=w.weight,
                                   lambda_scm=w.lambda_scm, grad_x0_student=d["gS"], loss=d["loss"],
                                   workspace=ws, status=st, stream=cap_stream)
                return
            t2va.stage3_objective(d["zt"], d["xT"], d["xS"], d["tan"], d["t"], d["zh"], d["yT"], d["yF"],
                                  beta=w.beta, gamma=w.gamma, eps_scm=w.eps_scm, eps_dmd=w.eps_dmd,
                                  weight=w.weight, lambda_scm=w.lambda_scm, lambda_dmd=w.lambda_dmd,
                                  grad_x0_student=d["gS"], grad_zhat0=d["gD"], loss=d["loss"],
                                  workspace=ws, status=st, stream=cap_stream)

        with torch.cuda.stream(cap_stream):
            for d in sets:
                call(d)
        cap_stream.synchronize()
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.stream(cap_stream):
            with torch.cuda.graph(graph, stream=cap_stream):
                for i in range(n_launch):
                    call(sets[i % R])
        reps = max(1, min(10, 2000 // n_launch))
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        with torch.cuda.stream(cap_stream):
            graph.replay()
            e0.record(cap_stream)
            for _ in range(reps):
                graph.replay()
            e1.record(cap_stream)
        cap_stream.synchronize()
        if int(st.item()) != 0:
            raise RuntimeError(f"device status {int(st.item())} at {name}")
        us = e0.elapsed_time(e1) * 1e3 / (reps * n_launch)
        gbs = nbytes / (us * 1e-6) / 1e9
        out[name] = {"elements": n_el, "algorithmic_bytes_per_launch": nbytes, "mean_launch_us": round(us, 3),
                     "achieved": round(gbs, 2), "unit": "GB/s", "frac": round(gbs / peak, 4),
                     "launches_timed": reps * n_launch, "input_sets": R}
        del graph, sets, ws
        torch.cuda.empty_cache()
    return out


def run_gpu(args, wl: S.Workload, rank: int, world: int, dist):
    import torch

    import joint_video_audio_02_b300 as t2va
    from joint_video_audio_02_b300.build import build

    build()
    t2va.load()
    dev = torch.device("cuda", torch.cuda.current_device())
    props = torch.cuda.get_device_properties(dev)
    l2 = int(getattr(props, "L2_cache_size", 126 * 2 ** 20))
    nb = step_bytes(wl)
    M = wl.num_modalities
    dt = wl.dtype
    tdt = torch.bfloat16 if dt == "bf16" else torch.float32

    # rotating input sets: together at least 3x the L2 size, so no step finds its inputs in L2
    set_bytes = nb["step"] + 2 * wl.batch * sum(wl.numels) * elem_size(dt)
    R = max(2, math.ceil(3 * l2 / set_bytes))
    fields_in = input_fields(wl)

    def to_dev(a):
        if dt == "bf16":
            return torch.from_numpy(a.view(np.int16)).view(torch.bfloat16).to(dev)
        return torch.from_numpy(a).to(dev)

    sets = []
    host0 = None
    for r in range(R):
        inp = S.make_workload_inputs(wl, seed_offset=rank_seed_offset(rank, r))
        if r == 0:
            host0 = inp
        d = {f: [to_dev(a) for a in getattr(inp, f)] for f in fields_in}
        d["t"] = torch.from_numpy(inp.t).to(dev)
        d["zt"] = [torch.empty_like(x) for x in d["z0"]]
        d["gS"] = [torch.empty(x.shape, dtype=torch.float32, device=dev) for x in d["z0"]]
        if is_stage3(wl):
            d["zht"] = [torch.empty_like(x) for x in d["zhat0"]]
            d["gD"] = [torch.empty(x.shape, dtype=torch.float32, device=dev) for x in d["z0"]]
        if wl.rf_wrapper:
            d["zrf"] = [torch.empty_like(x) for x in d["z0"]]
            d["t_rf"] = torch.empty(wl.batch, device=dev)
            if is_stage3(wl):
                d["zhrf"] = [torch.empty_like(x) for x in d["zhat0"]]
        d["loss"] = torch.empty(wl.batch, device=dev)
        d["norm"] = torch.empty(wl.batch * M, device=dev)
        d["cdmd"] = torch.empty(wl.batch * M, device=dev)
        sets.append(d)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    ws = t2va.new_workspace(wl.batch, M)
    torch.cuda.synchronize()

    def objective(d, stream=None):
        if wl.mode == S.STAGE3_CFG:
            t2va.stage3_objective_cfg(
                d["zt"], d["x0_teacher"], d["x0_student"], d["x0_tangent"], d["t"], d["zhat0"],
                d["x0_teacher_hat"], d["x0_teacher_hat_uncond"], d["x0_fake"], guidance=wl.guidance,
                beta=wl.beta, gamma=wl.gamma, eps_scm=wl.eps_scm, eps_dmd=wl.eps_dmd,
                weight=wl.weight, lambda_scm=wl.lambda_scm, lambda_dmd=wl.lambda_dmd,
                grad_x0_student=d["gS"], grad_zhat0=d["gD"], loss=d["loss"], norm=d["norm"],
                cdmd=d["cdmd"], workspace=ws, status=status, stream=stream)
        elif wl.mode == S.STAGE3:
            t2va.stage3_objective(d["zt"], d["x0_teacher"], d["x0_student"], d["x0_tangent"], d["t"],
                                  d["zhat0"], d["x0_teacher_hat"], d["x0_fake"], beta=wl.beta,
                                  gamma=wl.gamma, eps_scm=wl.eps_scm, eps_dmd=wl.eps_dmd,
                                  weight=wl.weight, lambda_scm=wl.lambda_scm, lambda_dmd=wl.lambda_dmd,
                                  grad_x0_student=d["gS"], grad_zhat0=d["gD"], loss=d["loss"],
                                  norm=d["norm"], cdmd=d["cdmd"], workspace=ws, status=status,
                                  stream=stream)
        else:
            t2va.scm_objective(d["zt"], d["x0_teacher"], d["x0_student"], d["x0_tangent"], d["t"],
                               beta=wl.beta, gamma=wl.gamma, eps_scm=wl.eps_scm, weight=wl.weight,
                               lambda_scm=wl.lambda_scm, grad_x0_student=d["gS"], loss=d["loss"],
                               norm=d["norm"], workspace=ws, status=status, stream=stream)

    def noise(d, stream=None):
        # both noisings (z0 -> z_t and the on-policy zhat0 -> zhat_t) share the per-sample t,
        # so they go to the library as one call over four latents
        z0, eps, zt = d["z0"], d["eps"], d["zt"]
        if is_stage3(wl):
            z0, eps, zt = z0 + d["zhat0"], eps + d["eps_hat"], zt + d["zht"]
        if wl.rf_wrapper:
            zrf = d["zrf"] + (d["zhrf"] if is_stage3(wl) else [])
            t2va.noise_rf(z0, eps, zt, zrf, d["t"], t_rf=d["t_rf"], status=status, stream=stream)
        else:
            t2va.noise(z0, eps, zt, d["t"], status=status, stream=stream)

    launches_per_step = 3   # t2va_noise + the objective's two kernels

    # CUDA graphs of whole steps, with no event nodes inside: an event node between two
    # kernels of a graph costs about 3 us of its own, which would be charged to the step
    K, W = args.steps, args.warmup
    S_steps = min(K, 1000)
    cap_stream = torch.cuda.Stream(device=dev)
    cap_stream.wait_stream(torch.cuda.current_stream())

    side = torch.cuda.Stream(device=dev)

    def capture(nsteps, offset=0, objective_only=False, noise_only=False):
        """A graph of `nsteps` steps. Whole steps are scheduled on two streams: the noising
        on a side stream, the objective on the capture stream. objective(i) waits for
        noise(i); noise(i) waits for the objective that last read its buffer set, i - R.
        So the noising of the next steps overlaps the objective of this one (their inputs
        and outputs are disjoint buffer sets), and every step does all of its work."""
        g = torch.cuda.CUDAGraph()
        with torch.cuda.stream(cap_stream):
            with torch.cuda.graph(g, stream=cap_stream):
                if not objective_only and not noise_only:
                    side.wait_stream(cap_stream)
                    ev_n = [torch.cuda.Event() for _ in range(nsteps)]
                    ev_o = [torch.cuda.Event() for _ in range(nsteps)]
                    for i in range(nsteps):
                        d = sets[(offset + i) % R]
                        with torch.cuda.stream(side):
                            if i >= R:
                                side.wait_event(ev_o[i - R])
                            noise(d, side)
                            ev_n[i].record(side)
                        cap_stream.wait_event(ev_n[i])
                        objective(d, cap_stream)
                        ev_o[i].record(cap_stream)
                    cap_stream.wait_stream(side)
                else:
                    for i in range(nsteps):
                        d = sets[(offset + i) % R]
                        if not objective_only:
                            noise(d, cap_stream)
                        if not noise_only:
                            objective(d, cap_stream)
        return g

    # eager warm-up of every set once (also first-call attribute setup), then capture
    with torch.cuda.stream(cap_stream):
        for d in sets:
            noise(d, cap_stream)
            objective(d, cap_stream)
    cap_stream.synchronize()
    g_main = capture(S_steps)
    reps, rem = divmod(K, S_steps)
    g_rem = capture(rem, offset=S_steps) if rem else None
    g_warm = capture(max(W, 3))
    # the dominant kernel alone: back-to-back objective launches over the same rotating sets,
    # in graphs of at least 500 launches whatever K is, so that a graph's fixed launch cost
    # is not spread over a handful of launches (at --steps 20 it added 0.3 us to each)
    S_leg = max(S_steps, 500)
    g_obj = capture(S_leg, objective_only=True)
    g_noise = capture(S_leg, noise_only=True)
    torch.cuda.synchronize()

    # The clock sampler runs from before the clock ramp to after the per-kernel legs, so
    # that even a short timed region lies inside a window with samples.
    sampler = ClockSampler("GPU-" + str(props.uuid))
    sampler.start()
    # clock ramp (the GPU leaves its idle clocks only under sustained load), then W warm-up steps
    ramp_t0 = time.time()
    with torch.cuda.stream(cap_stream):
        while time.time() - ramp_t0 < args.clock_ramp_seconds:
            g_main.replay()
            cap_stream.synchronize()
    cap_stream.synchronize()
    if dist is not None:
        dist.barrier()
    torch.cuda.synchronize()
    t_start = torch.cuda.Event(enable_timing=True)
    t_end = torch.cuda.Event(enable_timing=True)
    h0 = time.time()
    with torch.cuda.stream(cap_stream):
        # The W warm-up steps are replayed, not waited for, right before the start
        # event: the GPU is busy with them while the host submits the timed graphs, so
        # no submission latency falls inside the timed region.
        g_warm.replay()
        t_start.record(cap_stream)
        for _ in range(reps):
            g_main.replay()
        if g_rem is not None:
            g_rem.replay()
        t_end.record(cap_stream)
    cap_stream.synchronize()
    torch.cuda.synchronize()
    h1 = time.time()
    if dist is not None:
        dist.barrier()
    elapsed_ms = t_start.elapsed_time(t_end)
    st = int(status.item())
    if st != 0:
        raise RuntimeError(f"device status {st} during the benchmark")

    # the objective's mean launch duration: CUDA events on the launching stream around
    # `obj_reps` replays of S_leg back-to-back launches (inputs rotate over R sets), about
    # 5000 launches in all
    obj_reps = max(1, 5000 // S_leg)
    o_start = torch.cuda.Event(enable_timing=True)
    o_end = torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(cap_stream):
        g_obj.replay()
        o_start.record(cap_stream)
        for _ in range(obj_reps):
            g_obj.replay()
        o_end.record(cap_stream)
    cap_stream.synchronize()
    obj_mean_ms = o_start.elapsed_time(o_end) / (obj_reps * S_leg)
    # the same for the noising kernel
    with torch.cuda.stream(cap_stream):
        g_noise.replay()
        o_start.record(cap_stream)
        for _ in range(obj_reps):
            g_noise.replay()
        o_end.record(cap_stream)
    cap_stream.synchronize()
    noise_mean_ms = o_start.elapsed_time(o_end) / (obj_reps * S_leg)
    if int(status.item()) != 0:
        raise RuntimeError(f"device status {int(status.item())} during the benchmark")
    peak, peak_kind = measured_peak()
    extra = None
    if wl.name == DEFAULT_WORKLOAD and not args.no_extra_shapes:
        extra = objective_rooflines(EXTRA_SHAPES, dev, cap_stream, 100, l2, peak)
    h2 = time.time()
    time.sleep(0.02)
    sampler.stop()

    elapsed_ms = max_over_ranks(elapsed_ms, dist, dev)
    ms_per_step = elapsed_ms / K
    value = whole_job_gbs(world, nb["step"], K, elapsed_ms)
    obj_gbs = nb["objective"] / (obj_mean_ms * 1e-3) / 1e9
    clocks = sampler.summary(ramp_t0, h2)
    clocks["window"] = ("clock ramp, warm-up, timed steps and the per-kernel legs "
                        f"({h2 - ramp_t0:.2f} s; timed steps {h1 - h0:.4f} s)")

    # end to end through the public API with host buffers
    e2e = run_e2e(args, wl, host0, status, noise, objective, dev, nb, world, dist)

    result = {
        "metric": METRIC, "value": round(value, 2), "unit": UNIT, "n_gpus": world, "steps": K,
        "warmup": W, "ms_per_step": ms_per_step, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": dt, "data": "synthetic",
        "config": {"workload": wl.name, "global_batch": wl.batch * world, "per_gpu_batch": wl.batch,
                   "latent_shapes": [list(s) for s in wl.shapes], "mode": wl.mode,
                   "rf_wrapper": wl.rf_wrapper,
                   **({"guidance": list(wl.guidance)} if wl.mode == S.STAGE3_CFG else {}),
                   "elements_per_step": nb["elements"] * world,
                   "algorithmic_bytes_per_step": nb["step"] * world,
                   "parallelism": f"replicas x{world} (samples sharded by rank, no collective)",
                   "l2": f"rotating {R} input sets ({R * set_bytes / 2**20:.0f} MiB >= 3x L2 "
                         f"{l2 / 2**20:.0f} MiB): no step finds its inputs in L2",
                   "timing": "CUDA graph replay of whole steps (no event nodes inside); CUDA events "
                             "on the launching stream around the timed region",
                   "schedule": "noising on a side stream, objective on the main stream: objective(i) "
                               "after noise(i), noise(i) after objective(i - R) (buffer-set reuse), "
                               "so the next steps' noising overlaps this step's objective",
                   "clock_ramp_s": args.clock_ramp_seconds,
                   "value_covers": "the whole step: both noisings and the objective; the objective "
                                   "alone is roofline.achieved"},
        "elements_per_s": nb["elements"] * world * K / (elapsed_ms * 1e-3),
        "hbm_fraction_of_step": round(value / world / peak, 4),
        "roofline": {"kernel": {S.STAGE3: "t2va stage-3 objective",
                                S.STAGE3_CFG: "t2va guided stage-3 objective",
                                S.SCM: "t2va sCM objective"}.get(wl.mode, "t2va objective")
                               + " call (k_sums + k_grads)",
                     "bound": "hbm", "achieved": round(obj_gbs, 2), "peak": peak, "unit": "GB/s",
                     "frac": round(obj_gbs / peak, 4), "peak_source": f"{peak_kind} (MEASURED_PEAKS.json hbm_gbs)"
                     if peak_kind == "measured" else "fallback 6400 GB/s",
                     "traffic": committed_traffic(wl.name),
                     "algorithmic_bytes_per_launch": nb["objective"],
                     "mean_launch_us": round(obj_mean_ms * 1e3, 3),
                     "launches_timed": obj_reps * S_leg,
                     "launch_timing": "back-to-back objective launches in a CUDA graph, CUDA events "
                                      "around the region on the launching stream; includes the "
                                      "launch-to-launch gap",
                     "frac_of_nominal_8TBps": round(obj_gbs / 8000.0, 4)},
        "noise_kernel": {"kernel": "t2va_noise_rf (k_noise, z_t and z_rf)" if wl.rf_wrapper
                                   else "t2va_noise (k_noise)",
                         "achieved": round(nb["noise"] / (noise_mean_ms * 1e-3) / 1e9, 2),
                         "unit": "GB/s", "frac": round(nb["noise"] / (noise_mean_ms * 1e-3) / 1e9 / peak, 4),
                         "algorithmic_bytes_per_launch": nb["noise"],
                         "mean_launch_us": round(noise_mean_ms * 1e3, 3),
                         "launch_timing": "as for the roofline kernel"},
        "clocks": clocks,
        "e2e": e2e,
        "gpu_launches": launches_per_step * K,
    }
    if extra is not None:
        result["objective_at_other_shapes"] = extra
    return result


def _packed(fields_shapes, dev, pinned=False):
    """One byte block holding every (name, shape, dtype) tensor at a 256-byte aligned
    offset, and the tensor views into it."""
    import torch
    offs, total = [], 0
    for _, shape, dt in fields_shapes:
        n = int(np.prod(shape)) * torch.empty((), dtype=dt).element_size()
        offs.append((total, n))
        total += (n + 255) // 256 * 256
    if dev is None:
        block = torch.empty(total, dtype=torch.uint8, pin_memory=pinned)
    else:
        block = torch.empty(total, dtype=torch.uint8, device=dev)
    views = [block[o:o + n].view(dt).view(shape) for (o, n), (_, shape, dt) in zip(offs, fields_shapes)]
    return block, views


def run_e2e(args, wl, host0, status, noise, objective, dev, nb, world, dist):
    """The same steps with host buffers, through the public API: every step copies its
    inputs in from pinned host memory and its results, the float32 gradients and the
    per-sample losses, back to pinned host memory. Each direction is one copy per step:
    a step's inputs are packed in one pinned block and land in one device block whose
    views the library is called with, and the gradients and losses are written into one
    device block that is read back whole. Steps are pipelined the way a data loader
    feeds a training loop: two device buffer sets alternate, and the copies in, the
    compute and the copies out run on three streams ordered by events, so step i+1's
    inputs arrive while step i computes and step i-1's results drain. The host's time to
    submit a step is reported beside the device time."""
    import torch

    steps = max(4, min(args.steps, args.e2e_steps))
    tdt = torch.bfloat16 if wl.dtype == "bf16" else torch.float32
    M = wl.num_modalities
    fields = input_fields(wl)
    in_spec = [(f"{f}{m}", getattr(host0, f)[m].shape, tdt) for f in fields for m in range(M)]
    in_spec.append(("t", host0.t.shape, torch.float32))
    hblock, hviews = _packed(in_spec, None, pinned=True)
    for (name, _, _), v in zip(in_spec, hviews):
        if name == "t":
            v.copy_(torch.from_numpy(host0.t))
        else:
            f, m = name[:-1], int(name[-1])
            a = getattr(host0, f)[m]
            src = torch.from_numpy(a.view(np.int16)).view(torch.bfloat16) if wl.dtype == "bf16" else torch.from_numpy(a)
            v.copy_(src)
    shapes = [getattr(host0, "z0")[m].shape for m in range(M)]
    out_spec = [(f"gS{m}", shapes[m], torch.float32) for m in range(M)]
    if is_stage3(wl):
        out_spec += [(f"gD{m}", shapes[m], torch.float32) for m in range(M)]
    out_spec.append(("loss", (wl.batch,), torch.float32))
    sets = []
    for _ in range(2):
        iblock, iviews = _packed(in_spec, dev)
        oblock, oviews = _packed(out_spec, dev)
        d = {}
        for (name, _, _), v in zip(in_spec, iviews):
            if name == "t":
                d["t"] = v
            else:
                d.setdefault(name[:-1], []).append(v)
        for (name, _, _), v in zip(out_spec, oviews):
            if name == "loss":
                d["loss"] = v
            else:
                d.setdefault(name[:-1], []).append(v)
        d["zt"] = [torch.empty_like(x) for x in d["z0"]]
        if is_stage3(wl):
            d["zht"] = [torch.empty_like(x) for x in d["zhat0"]]
        if wl.rf_wrapper:
            d["zrf"] = [torch.empty_like(x) for x in d["z0"]]
            d["t_rf"] = torch.empty(wl.batch, device=dev)
            if is_stage3(wl):
                d["zhrf"] = [torch.empty_like(x) for x in d["zhat0"]]
        d["norm"] = torch.empty(wl.batch * M, device=dev)
        d["cdmd"] = torch.empty(wl.batch * M, device=dev)
        sets.append((iblock, oblock, d))
    h2d = hblock.numel()
    host_out = [_packed(out_spec, None, pinned=True)[0] for _ in sets]
    d2h = host_out[0].numel()
    s_in, s_cmp, s_out = (torch.cuda.Stream(device=dev) for _ in range(3))
    ev_in = [torch.cuda.Event() for _ in sets]
    ev_cmp = [torch.cuda.Event() for _ in sets]
    ev_out = [torch.cuda.Event() for _ in sets]

    def step(i):
        k = i % len(sets)
        iblock, oblock, d = sets[k]
        with torch.cuda.stream(s_in):
            if i >= len(sets):
                s_in.wait_event(ev_cmp[k])    # the compute that last read these inputs is done
            iblock.copy_(hblock, non_blocking=True)
            ev_in[k].record(s_in)
        with torch.cuda.stream(s_cmp):
            s_cmp.wait_event(ev_in[k])
            if i >= len(sets):
                s_cmp.wait_event(ev_out[k])   # the copy-out that last read these outputs is done
            noise(d, s_cmp)
            objective(d, s_cmp)
            ev_cmp[k].record(s_cmp)
        with torch.cuda.stream(s_out):
            s_out.wait_event(ev_cmp[k])
            host_out[k].copy_(oblock, non_blocking=True)
            ev_out[k].record(s_out)

    for i in range(len(sets)):
        step(i)
    torch.cuda.synchronize()
    if dist is not None:
        dist.barrier()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(s_in)
    t_host = time.perf_counter()
    for i in range(steps):
        step(i)
    e1.record(s_out)
    host_ms = (time.perf_counter() - t_host) * 1e3 / steps
    torch.cuda.synchronize()
    ms = max_over_ranks(e0.elapsed_time(e1), dist, dev)
    assert int(status.item()) == 0
    return {"value": round(whole_job_gbs(world, nb["step"], steps, ms), 3), "unit": UNIT,
            "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "steps": steps,
            "ms_per_step": ms / steps,
            "host_submit_ms_per_step": round(host_ms, 4),
            "link_gbs_per_step": round((h2d + d2h) / (ms / steps * 1e-3) / 1e9, 2),
            "pipeline": "2 device buffer sets; copy-in, compute and copy-out streams; one "
                        "pinned-block copy per direction per step",
            "read_back": "float32 gradients (every modality, both terms) and per-sample losses"}


# ---------------------------------------------------------------------------
# CPU oracle (baseline leg and reference arm)
# ---------------------------------------------------------------------------

def oracle_pass(wl: S.Workload, inp: S.Inputs):
    import oracle
    dt = wl.dtype
    if wl.rf_wrapper:
        zt = oracle.noise_rf(inp.z0, inp.eps, inp.t, dt)[0]
        if is_stage3(wl):
            oracle.noise_rf(inp.zhat0, inp.eps_hat, inp.t, dt)
    else:
        zt = oracle.noise(inp.z0, inp.eps, inp.t, dt)
        if is_stage3(wl):
            oracle.noise(inp.zhat0, inp.eps_hat, inp.t, dt)
    if wl.mode == S.STAGE3_CFG:
        oracle.stage3_objective_cfg(zt, inp.x0_teacher, inp.x0_student, inp.x0_tangent, inp.t,
                                    inp.zhat0, inp.x0_teacher_hat, inp.x0_teacher_hat_uncond,
                                    wl.guidance, inp.x0_fake, wl.beta, wl.gamma, wl.eps_scm,
                                    wl.eps_dmd, wl.weight, wl.lambda_scm, wl.lambda_dmd, dt)
    elif wl.mode == S.STAGE3:
        oracle.stage3_objective(zt, inp.x0_teacher, inp.x0_student, inp.x0_tangent, inp.t,
                                inp.zhat0, inp.x0_teacher_hat, inp.x0_fake, wl.beta, wl.gamma,
                                wl.eps_scm, wl.eps_dmd, wl.weight, wl.lambda_scm, wl.lambda_dmd, dt)
    else:
        oracle.scm_objective(zt, inp.x0_teacher, inp.x0_student, inp.x0_tangent, inp.t, wl.beta,
                             wl.gamma, wl.eps_scm, wl.weight, wl.lambda_scm, dt)


def bounded_sample(wl: S.Workload, frac: float) -> S.Workload:
    """The workload cut to one sample whose latents keep `frac` of each modality's elements."""
    import dataclasses
    numels = [max(16, int(n * frac)) for n in wl.numels]
    return dataclasses.replace(wl, batch=1, shapes=tuple((n,) for n in numels), t_fixed=None)


def cpu_baseline(wl: S.Workload, budget_s: float) -> dict:
    """The oracle, as it stands, on sample 0 of the workload, repeated for about budget_s."""
    one = bounded_sample(wl, 1.0)
    inp = S.make_workload_inputs(one)
    nbytes = step_bytes(one)["step"]
    reps, t0 = 0, time.perf_counter()
    while True:
        oracle_pass(one, inp)
        reps += 1
        if time.perf_counter() - t0 >= budget_s:
            break
    dt = time.perf_counter() - t0
    return {"value": round(nbytes * reps / dt / 1e9, 4), "unit": UNIT, "cores": 1, "kind": "oracle",
            "sample": f"sample 0 of {wl.batch} ({sum(one.numels):,} elements: noising + objective), "
                      f"{reps} passes in {dt:.1f} s; numpy float64, single thread"}


def _oracle_worker(job):
    """One process of the all-core baseline: the oracle on one sample, repeated for
    about `budget` seconds; returns (algorithmic bytes processed, seconds)."""
    name, sample, budget = job
    wl = S.workload(name)
    one = bounded_sample(wl, 1.0)
    inp = S.make_workload_inputs(one, seed_offset=sample)
    nbytes = step_bytes(one)["step"]
    oracle_pass(one, inp)  # first pass untimed (imports, caches)
    reps, t0 = 0, time.perf_counter()
    while True:
        oracle_pass(one, inp)
        reps += 1
        if time.perf_counter() - t0 >= budget:
            break
    return nbytes * reps, time.perf_counter() - t0


def cpu_baseline_all_cores(wl: S.Workload, budget_s: float, max_workers: int = 64) -> dict:
    """The same oracle over every host core: one single-threaded process per core, each
    on its own sample of the workload (samples are independent), started with `spawn`
    (the parent has a CUDA context). Aggregate rate = all bytes / the longest worker."""
    import multiprocessing as mp
    cores = max(1, min(os.cpu_count() or 1, max_workers))
    saved = {k: os.environ.get(k) for k in ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS")}
    for k in saved:
        os.environ[k] = "1"
    try:
        with mp.get_context("spawn").Pool(cores) as pool:
            res = pool.map(_oracle_worker, [(wl.name, i, budget_s) for i in range(cores)])
    finally:
        for k, v in saved.items():
            if v is None:
                os.environ.pop(k, None)
            else:
                os.environ[k] = v
    total = sum(r[0] for r in res)
    secs = max(r[1] for r in res)
    return {"value": round(total / secs / 1e9, 4), "unit": UNIT, "cores": cores, "kind": "oracle",
            "sample": f"{cores} processes, one per core (of {os.cpu_count()}), each repeating the oracle "
                      f"on one sample of the workload ({sum(wl.numels):,} elements: noising + objective) "
                      f"for about {budget_s:.0f} s; numpy float64, one thread per process"}


def run_reference(args, wl: S.Workload, world: int):
    """The oracle as the reference arm: each step a bounded sample of the workload."""
    probe = bounded_sample(wl, 0.05)
    pinp = S.make_workload_inputs(probe)
    t0 = time.perf_counter()
    oracle_pass(probe, pinp)
    rate = sum(probe.numels) / max(time.perf_counter() - t0, 1e-6)   # elements / s
    budget = min(120.0, max(20.0, 3.0 * (args.steps + args.warmup)))
    per_step = budget / max(1, args.steps + args.warmup)
    frac = min(1.0, per_step * rate / sum(wl.numels))
    one = bounded_sample(wl, frac)
    inp = S.make_workload_inputs(one)
    for _ in range(args.warmup):
        oracle_pass(one, inp)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        oracle_pass(one, inp)
    dt = time.perf_counter() - t0
    nbytes = step_bytes(one)["step"]
    value = nbytes * args.steps / dt / 1e9
    sample = (f"per step: one sample holding {frac:.4f} of each latent of the workload "
              f"({sum(one.numels):,} elements), noising + objective")
    return {"impl": "reference", "metric": METRIC, "value": round(value, 4), "unit": UNIT, "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": dt / args.steps * 1e3,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic",
            "config": {"workload": wl.name, "global_batch": wl.batch, "per_gpu_batch": wl.batch,
                       "latent_shapes": [list(s) for s in wl.shapes], "mode": wl.mode,
                       "reference": "float64 CPU oracle (numpy), the parity reference of this library"},
            "cpu_baseline": {"value": round(value, 4), "unit": UNIT, "cores": 1, "kind": "oracle",
                             "sample": sample},
            "e2e": {"value": round(value, 4), "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}


# ---------------------------------------------------------------------------
# W8A8 linear (second workload): per-row quantisation of the activations + the INT8
# contraction with the post-scale epilogue
# ---------------------------------------------------------------------------

# (M, N, K): M = video tokens of the 1024x1792 (28,672) and 512x768 (6,144) latents;
# N = K = 4096, a projection width assumed for the 14B video backbone (not printed)
# the "tc" workloads store the codes as bfloat16 integers and contract them on the
# tcgen05 tensor cores; the others use int8 codes and the warp-level INT8 MMA
W8A8_WORKLOADS = {"w8a8_28672x4096x4096_bf16": (28672, 4096, 4096, "int8"),
                  "w8a8_6144x4096x4096_bf16": (6144, 4096, 4096, "int8"),
                  "w8a8tc_28672x4096x4096_bf16": (28672, 4096, 4096, "bf16"),
                  "w8a8tc_6144x4096x4096_bf16": (6144, 4096, 4096, "bf16")}
W8A8_METRIC = "W8A8 linear TOPS (per-row int8 quantisation + exact int8 GEMM, bf16 out)"


def w8a8_cpu_baseline(M_sample: int, N: int, K: int, budget_s: float) -> dict:
    """The oracle on a bounded sample: M_sample rows against the full weight matrix."""
    import oracle.w8a8_oracle as W8
    r = np.random.default_rng(0)
    x = r.standard_normal((M_sample, K)).astype(np.float32)
    wq = r.integers(-127, 128, (N, K)).astype(np.int8)
    sw = r.uniform(1e-4, 1e-3, N).astype(np.float32)
    b = r.standard_normal(N).astype(np.float32)
    reps, t0 = 0, time.perf_counter()
    while True:
        W8.w8a8_forward(x, wq, sw, b)
        reps += 1
        if time.perf_counter() - t0 >= budget_s:
            break
    dt = time.perf_counter() - t0
    return {"value": round(2.0 * M_sample * N * K * reps / dt / 1e12, 6), "unit": "TOPS", "cores": 1,
            "kind": "oracle", "sample": f"{M_sample} rows x N={N} x K={K}, {reps} passes in {dt:.1f} s; "
                                        "numpy int64 matmul + float64 epilogue, single thread"}


def run_w8a8(args, name: str):
    import torch

    import joint_video_audio_02_b300 as t2va
    from joint_video_audio_02_b300.build import build

    build()
    t2va.load()
    M, N, K, codes = W8A8_WORKLOADS[name]
    cdt = torch.bfloat16 if codes == "bf16" else torch.int8
    dev = torch.device("cuda", torch.cuda.current_device())
    props = torch.cuda.get_device_properties(dev)
    g = torch.Generator(device=dev).manual_seed(1234)
    x = torch.randn((M, K), generator=g, device=dev).to(torch.bfloat16)
    w = torch.randn((N, K), generator=g, device=dev) * 0.02
    bias = torch.randn(N, generator=g, device=dev) * 0.1
    wq = torch.empty((N, K), dtype=cdt, device=dev)
    sw = torch.empty(N, device=dev)
    t2va.quantize_rows(w, wq, sw)                     # static weight quantisation, once
    xq = torch.empty((M, K), dtype=cdt, device=dev)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    sx = torch.empty(M, device=dev)
    y = torch.empty((M, N), dtype=torch.bfloat16, device=dev)
    st = torch.cuda.Stream(device=dev)

    def quant():
        t2va.quantize_rows(x, xq, sx, stream=st)

    def linear():
        t2va.w8a8_linear(xq, sx, wq, sw, y, bias, status=status, stream=st)

    with torch.cuda.stream(st):
        quant()
        linear()
    st.synchronize()
    K_steps, W = args.steps, args.warmup
    S_steps = max(1, min(K_steps, 50))

    def graph(fn_list, n):
        gr = torch.cuda.CUDAGraph()
        with torch.cuda.stream(st):
            with torch.cuda.graph(gr, stream=st):
                for _ in range(n):
                    for fn in fn_list:
                        fn()
        return gr

    g_step, g_q, g_l = graph([quant, linear], S_steps), graph([quant], S_steps), graph([linear], S_steps)
    reps = max(1, K_steps // S_steps)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)

    def timed(gr):
        with torch.cuda.stream(st):
            for _ in range(max(1, W // S_steps)):
                gr.replay()
            st.synchronize()
            e0.record(st)
            for _ in range(reps):
                gr.replay()
            e1.record(st)
        st.synchronize()
        return e0.elapsed_time(e1) / (reps * S_steps)

    t_ramp = time.time()
    with torch.cuda.stream(st):
        while time.time() - t_ramp < args.clock_ramp_seconds:
            g_step.replay()
            st.synchronize()
    sampler = ClockSampler("GPU-" + str(props.uuid))
    sampler.start()
    time.sleep(0.05)
    h0 = time.time()
    ms_step = timed(g_step)
    h1 = time.time()
    time.sleep(0.02)
    sampler.stop()
    ms_q, ms_l = timed(g_q), timed(g_l)
    if int(status.item()) != 0:
        raise RuntimeError(f"device status {int(status.item())} during the benchmark")
    flops = 2.0 * M * N * K
    q_bytes = M * K * 2 + M * K * (2 if codes == "bf16" else 1) + 4 * M
    peak_bf16, peak_bf16_sustained = None, None
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            pk = json.load(f)
        peak_bf16 = float(pk["bf16_tflops"])
        peak_bf16_sustained = float(pk["bf16_tflops_sustained"]) if "bf16_tflops_sustained" in pk else None
    except Exception:
        peak_bf16, peak_bf16_sustained = 1800.0, 1400.0
    peak_hbm, _ = measured_peak()

    # end to end: bf16 activations from pinned host memory, bf16 output back to the host
    hx = x.cpu().pin_memory()
    hy = torch.empty((M, N), dtype=torch.bfloat16, pin_memory=True)
    steps_e2e = max(3, min(K_steps, args.e2e_steps))
    with torch.cuda.stream(st):
        x.copy_(hx, non_blocking=True)
        quant()
        linear()
        hy.copy_(y, non_blocking=True)
        st.synchronize()
        e0.record(st)
        for _ in range(steps_e2e):
            x.copy_(hx, non_blocking=True)
            quant()
            linear()
            hy.copy_(y, non_blocking=True)
        e1.record(st)
    st.synchronize()
    ms_e2e = e0.elapsed_time(e1) / steps_e2e
    result = {
        "metric": W8A8_METRIC, "value": round(flops / (ms_step * 1e-3) / 1e12, 2), "unit": "TOPS",
        "n_gpus": 1, "steps": reps * S_steps, "warmup": W, "ms_per_step": ms_step,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "int8",
        "data": "synthetic",
        "config": {"workload": name, "M": M, "N": N, "K": K, "codes": codes, "x": "bf16 N(0,1)", "w": "N(0, 0.02^2), "
                   "quantised once per output channel", "out": "bf16", "bias": True,
                   "l2": "activations 235 MB / 50 MB and outputs larger than L2 at M = 28672 / 6144; "
                         "the 16.8 MB int8 weights stay in L2 by design",
                   "timing": "CUDA graphs of back-to-back steps, CUDA events on the launching stream"},
        "roofline": {"kernel": ("k_w8a8_tc_wide (tcgen05.mma kind::f16 M128 N256, TMA, TMEM)" if N % 256 == 0
                                else "k_w8a8_tc (tcgen05.mma kind::f16 M128 N128, TMA, TMEM)") if codes == "bf16"
                               else "k_w8a8_gemm (mma.sync m16n8k32 s8)", "bound": "tensor",
                     "achieved": round(flops / (ms_l * 1e-3) / 1e12, 2), "peak": peak_bf16,
                     "unit": "TOPS", "frac": round(flops / (ms_l * 1e-3) / 1e12 / peak_bf16, 4),
                     "peak_source": "measured dense bf16 TFLOP/s (MEASURED_PEAKS.json bf16_tflops): the "
                                    "tensor-core path runs bf16 MMAs; sm_103a has no INT8 tcgen05.mma",
                     "traffic": None, "mean_launch_us": round(ms_l * 1e3, 2),
                     # the GEMMs run back to back after a clock ramp, near the 1.1 kW power
                     # limit: the measured sustained cuBLAS rate is the other bound
                     "peak_sustained": peak_bf16_sustained,
                     "frac_of_sustained": (round(flops / (ms_l * 1e-3) / 1e12 / peak_bf16_sustained, 4)
                                           if peak_bf16_sustained else None)},
        "quantize_kernel": {"kernel": "k_quantize_rows", "achieved": round(q_bytes / (ms_q * 1e-3) / 1e9, 1),
                            "unit": "GB/s", "frac": round(q_bytes / (ms_q * 1e-3) / 1e9 / peak_hbm, 4),
                            "algorithmic_bytes_per_launch": q_bytes, "mean_launch_us": round(ms_q * 1e3, 2)},
        "clocks": sampler.summary(h0, h1),
        "e2e": {"value": round(flops / (ms_e2e * 1e-3) / 1e12, 2), "unit": "TOPS",
                "h2d_bytes_per_step": M * K * 2, "d2h_bytes_per_step": M * N * 2, "steps": steps_e2e,
                "ms_per_step": ms_e2e},
        "gpu_launches": 2 * reps * S_steps,
    }
    if not args.no_cpu_baseline:
        result["cpu_baseline"] = w8a8_cpu_baseline(64, N, K, args.cpu_baseline_seconds)
    return result


# ---------------------------------------------------------------------------
# fused gated residual + modulated RMS normalisation (inference-side, memory-bound)
# ---------------------------------------------------------------------------

# rows = video tokens of the 1024x1792 latent (28,672), D = 4096 (assumed width)
FUSED_WORKLOADS = {"modnorm_28672x4096_bf16": (28672, 4096)}
FUSED_METRIC = "fused gated residual + modulated RMSNorm GB/s and % of B300 HBM peak"


def fused_cpu_baseline(D: int, budget_s: float) -> dict:
    import oracle.fused_ops_oracle as F
    r = np.random.default_rng(0)
    rows = 64
    h, u = r.standard_normal((rows, D)), r.standard_normal((rows, D))
    g, sc, sh = (r.standard_normal((1, D)) for _ in range(3))
    reps, t0 = 0, time.perf_counter()
    while True:
        F.residual_modnorm(h, u, g, sc, sh, 1e-6, rows, lambda v: v)
        reps += 1
        if time.perf_counter() - t0 >= budget_s:
            break
    dt = time.perf_counter() - t0
    return {"value": round(rows * D * 8 * reps / dt / 1e9, 4), "unit": "GB/s", "cores": 1, "kind": "oracle",
            "sample": f"{rows} rows x D={D}, {reps} passes in {dt:.1f} s; numpy float64, single thread"}


def run_fused(args, name: str):
    import torch

    import joint_video_audio_02_b300 as t2va
    from joint_video_audio_02_b300.build import build

    build()
    t2va.load()
    rows, D = FUSED_WORKLOADS[name]
    dev = torch.device("cuda", torch.cuda.current_device())
    props = torch.cuda.get_device_properties(dev)
    g = torch.Generator(device=dev).manual_seed(99)
    # rotating sets larger than L2 together: no launch finds its inputs in L2
    l2 = int(getattr(props, "L2_cache_size", 126 * 2 ** 20))
    set_bytes = rows * D * 2 * 4
    R = max(2, math.ceil(3 * l2 / set_bytes))
    sets = []
    for _ in range(R):
        sets.append({"h": torch.randn((rows, D), generator=g, device=dev).to(torch.bfloat16),
                     "u": torch.randn((rows, D), generator=g, device=dev).to(torch.bfloat16),
                     "h_out": torch.empty((rows, D), dtype=torch.bfloat16, device=dev),
                     "y": torch.empty((rows, D), dtype=torch.bfloat16, device=dev)})
    gate = torch.rand((1, D), generator=g, device=dev)
    scale = torch.rand((1, D), generator=g, device=dev) - 0.5
    shift = torch.rand((1, D), generator=g, device=dev) - 0.5
    st = torch.cuda.Stream(device=dev)

    def step(d):
        t2va.residual_modnorm(d["h"], d["y"], u=d["u"], gate=gate, scale=scale, shift=shift, eps=1e-6,
                              h_out=d["h_out"], stream=st)

    with torch.cuda.stream(st):
        for d in sets:
            step(d)
    st.synchronize()
    S_steps = max(R, min(args.steps, 200))
    gr = torch.cuda.CUDAGraph()
    with torch.cuda.stream(st):
        with torch.cuda.graph(gr, stream=st):
            for i in range(S_steps):
                step(sets[i % R])
    reps = max(1, args.steps // S_steps)
    t_ramp = time.time()
    with torch.cuda.stream(st):
        while time.time() - t_ramp < args.clock_ramp_seconds:
            gr.replay()
            st.synchronize()
        for _ in range(max(1, args.warmup // S_steps)):
            gr.replay()
    st.synchronize()
    sampler = ClockSampler("GPU-" + str(props.uuid))
    sampler.start()
    time.sleep(0.05)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    h0 = time.time()
    with torch.cuda.stream(st):
        e0.record(st)
        for _ in range(reps):
            gr.replay()
        e1.record(st)
    st.synchronize()
    h1 = time.time()
    time.sleep(0.02)
    sampler.stop()
    ms = e0.elapsed_time(e1) / (reps * S_steps)
    nbytes = rows * D * 2 * 4 + 3 * D * 4          # h, u read; h', y written; three vectors
    gbs = nbytes / (ms * 1e-3) / 1e9
    peak, peak_kind = measured_peak()
    # end to end: h and u from pinned host memory, h' and y back to the host
    hh = sets[0]["h"].cpu().pin_memory()
    hu = sets[0]["u"].cpu().pin_memory()
    ho = torch.empty((rows, D), dtype=torch.bfloat16, pin_memory=True)
    hy = torch.empty((rows, D), dtype=torch.bfloat16, pin_memory=True)
    d = sets[0]
    steps_e2e = max(3, min(args.steps, args.e2e_steps))
    with torch.cuda.stream(st):
        e0.record(st)
        for _ in range(steps_e2e):
            d["h"].copy_(hh, non_blocking=True)
            d["u"].copy_(hu, non_blocking=True)
            step(d)
            ho.copy_(d["h_out"], non_blocking=True)
            hy.copy_(d["y"], non_blocking=True)
        e1.record(st)
    st.synchronize()
    ms_e2e = e0.elapsed_time(e1) / steps_e2e
    result = {
        "metric": FUSED_METRIC, "value": round(gbs, 2), "unit": "GB/s", "n_gpus": 1,
        "steps": reps * S_steps, "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": name, "rows": rows, "D": D, "samples": 1, "inputs": "h, u ~ N(0,1) bf16; gate "
                   "U(0,1), scale and shift U(-0.5,0.5) float32", "outputs": "h' and y, bf16",
                   "l2": f"rotating {R} sets ({R * set_bytes / 2**20:.0f} MiB >= 3x L2)",
                   "timing": "CUDA graph of back-to-back launches, CUDA events on the launching stream"},
        "roofline": {"kernel": "k_residual_modnorm", "bound": "hbm", "achieved": round(gbs, 2), "peak": peak,
                     "unit": "GB/s", "frac": round(gbs / peak, 4), "traffic": None,
                     "algorithmic_bytes_per_launch": nbytes, "mean_launch_us": round(ms * 1e3, 2),
                     "peak_source": f"{peak_kind} (MEASURED_PEAKS.json hbm_gbs)"},
        "clocks": sampler.summary(h0, h1),
        "e2e": {"value": round(nbytes / (ms_e2e * 1e-3) / 1e9, 2), "unit": "GB/s",
                "h2d_bytes_per_step": rows * D * 4, "d2h_bytes_per_step": rows * D * 4, "steps": steps_e2e,
                "ms_per_step": ms_e2e},
        "gpu_launches": reps * S_steps,
    }
    if not args.no_cpu_baseline:
        result["cpu_baseline"] = fused_cpu_baseline(D, args.cpu_baseline_seconds)
    return result


def main():
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20000)
    ap.add_argument("--warmup", type=int, default=50)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD,
                    choices=sorted(S.WORKLOADS) + sorted(W8A8_WORKLOADS) + sorted(FUSED_WORKLOADS))
    ap.add_argument("--e2e-steps", type=int, default=20)
    ap.add_argument("--clock-ramp-seconds", type=float, default=0.5,
                    help="untimed load before the warm-up steps so the GPU leaves its idle clocks")
    ap.add_argument("--cpu-baseline-seconds", type=float, default=12.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-extra-shapes", action="store_true",
                    help="skip the objective-only rooflines at the 1024x1792, sweep and sCM-only shapes")
    args = ap.parse_args()
    if args.warmup < 0 or args.steps < 1:
        ap.error("--steps >= 1 and --warmup >= 0")

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if args.workload in FUSED_WORKLOADS:
        if args.impl == "reference":
            base = fused_cpu_baseline(FUSED_WORKLOADS[args.workload][1], 10.0)
            rows, D = FUSED_WORKLOADS[args.workload]
            print(json.dumps({"impl": "reference", "metric": FUSED_METRIC, "value": base["value"], "unit": "GB/s",
                              "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
                              "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
                              "dtype": "f64", "data": "synthetic",
                              "config": {"workload": args.workload, "rows": rows, "D": D},
                              "cpu_baseline": base,
                              "e2e": {"value": base["value"], "unit": "GB/s", "h2d_bytes_per_step": 0,
                                      "d2h_bytes_per_step": 0}}), flush=True)
            return
        import torch
        torch.cuda.set_device(local)
        if rank == 0:
            print(json.dumps(run_fused(args, args.workload)), flush=True)
        return
    if args.workload in W8A8_WORKLOADS:
        if args.impl == "reference":
            M, N, K, _ = W8A8_WORKLOADS[args.workload]
            base = w8a8_cpu_baseline(16, N, K, 10.0)
            print(json.dumps({"impl": "reference", "metric": W8A8_METRIC, "value": base["value"],
                              "unit": "TOPS", "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
                              "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
                              "dtype": "int64", "data": "synthetic",
                              "config": {"workload": args.workload, "M": M, "N": N, "K": K},
                              "cpu_baseline": base,
                              "e2e": {"value": base["value"], "unit": "TOPS", "h2d_bytes_per_step": 0,
                                      "d2h_bytes_per_step": 0}}), flush=True)
            return
        import torch
        torch.cuda.set_device(local)
        if rank == 0:
            print(json.dumps(run_w8a8(args, args.workload)), flush=True)
        return
    wl = S.workload(args.workload)

    if args.impl == "reference":
        if rank == 0:
            print(json.dumps(run_reference(args, wl, world)), flush=True)
        return

    import torch
    torch.cuda.set_device(local)
    dist = None
    if world > 1:
        import torch.distributed as tdist
        os.environ.setdefault("MASTER_ADDR", "127.0.0.1")
        tdist.init_process_group("nccl", rank=rank, world_size=world,
                                  device_id=torch.device("cuda", local))
        dist = tdist
    result = run_gpu(args, wl, rank, world, dist)
    if rank == 0:
        if world == 1 and not args.no_cpu_baseline:
            result["cpu_baseline"] = cpu_baseline_all_cores(wl, args.cpu_baseline_seconds)
            result["cpu_baseline_1core"] = cpu_baseline(wl, args.cpu_baseline_seconds)
        else:
            result["cpu_baseline"] = None
        print(json.dumps(result), flush=True)
    if dist is not None:
        dist.barrier()
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
