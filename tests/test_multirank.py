"""The multi-rank host logic of bench.py on two gloo ranks (CPU, no GPU).

`bench.py --gpus N` runs one pack per rank with no collective on the data path
(replicas: KV groups, sequences and packs are independent), then takes the max
of the ranks' step times and reports the whole job's ms per pack.  Its
reference arm runs on rank 0 only.  These tests run those same functions in
two spawned processes joined by a gloo process group on 127.0.0.1."""
import json
import os
import socket
import types

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

WORLD = 2


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, outdir, mode):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    import bench
    import workloads as W

    dist.init_process_group("gloo", rank=rank, world_size=world)
    res = {}
    try:
        assert bench.dist_env() == (rank, world, rank)
        if mode == "timing":
            local = [1.25, 3.5][rank]                 # ms per step on this rank
            slowest = bench.slowest_rank_ms(local, world)
            shape = W.PrefillShape("tiny", (40, 25), 16, 1, 1)
            x = W.make_prefill(shape, seed=bench.rank_seed(7, rank))
            res = {"slowest": slowest, "value": bench.job_ms_per_pack(slowest, world),
                   "seed": bench.rank_seed(7, rank),
                   "q_sum": float(x["q"].float().sum())}
        else:
            args = types.SimpleNamespace(seed=0, steps=1, warmup=0, gpus=world, pool=8,
                                         ref_budget_s=2.0)
            res = {"line": bench.run_reference(args)}
        dist.barrier()
    finally:
        dist.destroy_process_group()
    with open(os.path.join(outdir, f"{rank}.json"), "w") as f:
        json.dump(res, f)


def _run(tmp_path, mode):
    mp.spawn(_rank_main, args=(WORLD, _free_port(), str(tmp_path), mode), nprocs=WORLD,
             join=True)
    return [json.load(open(tmp_path / f"{r}.json")) for r in range(WORLD)]


def test_slowest_rank_sets_the_job_time(tmp_path):
    r0, r1 = _run(tmp_path, "timing")
    # every rank sees the max of the step times; the job completes 2 packs per step
    assert r0["slowest"] == r1["slowest"] == 3.5
    assert r0["value"] == r1["value"] == pytest.approx(1.75)
    # each rank draws its own pack (weak scaling)
    assert r0["seed"] != r1["seed"]
    assert r0["q_sum"] != r1["q_sum"]


def test_reference_arm_runs_on_rank_zero_only(tmp_path):
    r0, r1 = _run(tmp_path, "reference")
    assert r1["line"] is None
    line = r0["line"]
    assert line["impl"] == "reference" and line["n_gpus"] == WORLD
    assert line["unit"] == "ms" and line["value"] > 0
    assert line["cpu_baseline"]["kind"] == "oracle" and line["cpu_baseline"]["cores"] >= 1
    assert line["e2e"]["h2d_bytes_per_step"] == 0
    # the same workload dict as the GPU arm prints
    import bench
    import workloads as W
    assert line["config"] == bench.config_dict(W.config(1, 0), 8, WORLD)
