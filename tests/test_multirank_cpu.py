"""The N > 1 host path on CPU: two gloo ranks.

Groups are independent, so the path shards by groups with no collective in the data
path: each rank draws its own groups (bench.rank_seed), the job's time is the slowest
rank's (bench.max_over_ranks), and the job's value counts every rank's tokens
(bench.job_value).  Under torchrun the reference arm runs on rank 0 alone."""
import json
import os
import socket
import subprocess
import sys

import numpy as np
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402
import oracle  # noqa: E402
from causal_linear_attention_gb300.inputs import make_inputs  # noqa: E402

G, C, D, EPS = 3, 20, 16, 1e-6


def free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def worker(rank, world, port, result_path):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        # the slowest rank's time is the job's time, on every rank
        t = bench.max_over_ranks(0.5 + rank, world)
        # each rank's own groups, processed with no collective
        x = make_inputs(G, C, D, dtype="f32", seed=bench.rank_seed(rank), carry=True)
        o, S, z = oracle.fwd(x.q, x.k, x.v, x.S0, x.z0, eps=EPS)
        parts = [None] * world
        dist.all_gather_object(parts, (x.q.numpy(), x.k.numpy(), x.v.numpy(), x.S0.numpy(), x.z0.numpy(),
                                       np.asarray(o), np.asarray(S), np.asarray(z)))
        bench.barrier(world)
        if rank == 0:
            np.save(result_path, np.array([t], dtype=np.float64))
            cat = [np.concatenate([p[i] for p in parts]) for i in range(8)]
            o2, S2, z2 = oracle.fwd(*(torch.from_numpy(a) for a in cat[:5]), eps=EPS)
            ok = (np.array_equal(np.asarray(o2), cat[5]) and np.array_equal(np.asarray(S2), cat[6])
                  and np.array_equal(np.asarray(z2), cat[7]))
            np.save(result_path + ".ok.npy", np.array([ok]))
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_shard_groups_without_a_collective(tmp_path):
    oracle.build()
    path = str(tmp_path / "t.npy")
    mp.start_processes(worker, args=(2, free_port(), path), nprocs=2, join=True, start_method="spawn")
    assert np.load(path)[0] == 1.5
    # the per-rank results, side by side, equal one run over all the groups
    assert bool(np.load(path + ".ok.npy")[0])


def test_ranks_draw_different_groups():
    a = make_inputs(2, 8, 16, dtype="bf16", seed=bench.rank_seed(0))
    b = make_inputs(2, 8, 16, dtype="bf16", seed=bench.rank_seed(1))
    assert not torch.equal(a.q, b.q)


def test_job_value_counts_every_rank():
    assert bench.job_value(1, 160, 128, 10, 2.0) == 160 * 128 * 10 / 2.0
    assert bench.job_value(4, 160, 128, 10, 2.0) == 4 * bench.job_value(1, 160, 128, 10, 2.0)
    assert bench.max_over_ranks(3.25, 1) == 3.25


def test_reference_arm_under_torchrun_prints_one_line_from_rank_zero():
    oracle.build()
    env = dict(os.environ, OMP_NUM_THREADS="2")
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", "2", "--master-addr",
           "127.0.0.1", "--master-port", str(free_port()), os.path.join(ROOT, "bench.py"), "--impl", "reference",
           "--gpus", "2", "--steps", "1", "--warmup", "3", "--ref-seconds", "2"]
    r = subprocess.run(cmd, cwd=ROOT, env=env, capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["n_gpus"] == 2 and d["value"] > 0
    assert d["cpu_baseline"]["kind"] == "oracle" and d["e2e"]["h2d_bytes_per_step"] == 0
