"""The multi-rank path on CPU: world size 2 over gloo.

The objective's every reduction is per (sample, modality), so the path shards by
sample with no collective on the data path. These tests check the two things the
sharded benchmark relies on, with real torch.distributed ranks on 127.0.0.1:

* each rank's shard gives exactly the per-sample results of the whole batch
  (sample independence, checked with the float64 oracle on both ranks);
* the timing reduction takes the slowest rank, and the whole-job figure counts
  every rank's bytes once.
"""

import os
import socket

import numpy as np
import pytest
import torch.multiprocessing as mp

import synthetic as S


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, outdir):
    import torch
    import torch.distributed as dist

    import bench
    import oracle

    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        # one batch of 4 samples, split 2 + 2 by rank
        B, numels = 4, [96, 40]
        full = S.make_inputs(B, numels, "bf16", S.STAGE3, seed=(77,))
        per = B // world
        mine = S.slice_samples(full, range(rank * per, (rank + 1) * per))
        p = dict(beta=1.0, gamma=0.9, eps_scm=1e-6, eps_dmd=1e-6, weight=(1.0, 4.0),
                 lambda_scm=1.0, lambda_dmd=0.25)

        def run(inp):
            zt = oracle.noise(inp.z0, inp.eps, inp.t, "bf16")
            return oracle.stage3_objective(zt, inp.x0_teacher, inp.x0_student, inp.x0_tangent,
                                           inp.t, inp.zhat0, inp.x0_teacher_hat, inp.x0_fake,
                                           p["beta"], p["gamma"], p["eps_scm"], p["eps_dmd"],
                                           p["weight"], p["lambda_scm"], p["lambda_dmd"], "bf16")

        out = run(mine)
        loss = torch.from_numpy(out["loss"])
        gathered = [torch.zeros_like(loss) for _ in range(world)]
        dist.all_gather(gathered, loss)
        gnorm = torch.tensor([float(np.sum(g ** 2)) for g in out["grad_x0_student"]],
                             dtype=torch.float64)
        gn_all = [torch.zeros_like(gnorm) for _ in range(world)]
        dist.all_gather(gn_all, gnorm)

        # the slowest rank's time (rank r reports 10 + 5 r ms)
        ms = bench.max_over_ranks(10.0 + 5.0 * rank, dist, "cpu")
        np.save(os.path.join(outdir, f"rank{rank}.npy"),
                np.array([*torch.cat(gathered).tolist(), ms], dtype=np.float64))
        if rank == 0:
            np.save(os.path.join(outdir, "gnorm.npy"), torch.stack(gn_all).numpy())
        # every rank draws its own samples in the benchmark
        offs = [bench.rank_seed_offset(r, i) for r in range(world) for i in range(8)]
        assert len(set(offs)) == len(offs)
    finally:
        dist.destroy_process_group()


def test_two_rank_shards_match_whole_batch(tmp_path):
    import oracle

    world = 2
    mp.start_processes(_worker, args=(world, _free_port(), str(tmp_path)), nprocs=world,
                       join=True, start_method="spawn")
    r0 = np.load(tmp_path / "rank0.npy")
    r1 = np.load(tmp_path / "rank1.npy")
    np.testing.assert_array_equal(r0, r1)        # all_gather gives both ranks the same view
    assert r0[-1] == 15.0                         # max over ranks, not rank 0's own time

    B, numels = 4, [96, 40]
    full = S.make_inputs(B, numels, "bf16", S.STAGE3, seed=(77,))
    zt = oracle.noise(full.z0, full.eps, full.t, "bf16")
    whole = oracle.stage3_objective(zt, full.x0_teacher, full.x0_student, full.x0_tangent, full.t,
                                    full.zhat0, full.x0_teacher_hat, full.x0_fake, 1.0, 0.9,
                                    1e-6, 1e-6, (1.0, 4.0), 1.0, 0.25, "bf16")
    np.testing.assert_array_equal(r0[:-1], whole["loss"])    # sharding changes no bit

    gn = np.load(tmp_path / "gnorm.npy")                      # [rank, modality]
    for m in range(2):
        g = whole["grad_x0_student"][m]
        expect = np.array([np.sum(g[:2] ** 2), np.sum(g[2:] ** 2)])
        np.testing.assert_allclose(gn[:, m], expect, rtol=1e-15)


def test_whole_job_value_counts_every_rank():
    import bench

    # two ranks, 1 MB per step each, 100 steps, slowest rank 10 ms: 2 * 1e6 * 100 / 0.01 s
    assert bench.whole_job_gbs(2, 10 ** 6, 100, 10.0) == pytest.approx(20.0)
    assert bench.max_over_ranks(3.5, None, "cpu") == 3.5
