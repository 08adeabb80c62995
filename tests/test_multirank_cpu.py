"""The multi-GPU (replica) path of bench.py, exercised with world_size-2 gloo on CPU.

Every (b, h) slice is independent, so N GPUs run N replicas with no
collective on the data path; only timing crosses ranks.  Two spawned gloo
ranks check: the max-over-ranks reduction of step times, the whole-job
throughput formula, that each rank draws its own batch, and that the
reference arm leaves all work to rank 0.
"""

import json
import os
import socket
import sys

import pytest
import torch
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, outdir):
    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    import torch.distributed as dist
    import bench
    import workloads
    dist.init_process_group("gloo", rank=rank, world_size=world)
    ms = [2.5, 4.0][rank]                        # per-rank step times
    got = bench.max_over_ranks(ms, torch.device("cpu"))
    q, _, _, _ = workloads.make_inputs(1, 1, 8, 64, workloads.replica_seed(workloads.TINY, rank))
    digest = float(q.float().sum())
    gathered = [None] * world
    dist.all_gather_object(gathered, digest)
    dist.barrier()
    with open(os.path.join(outdir, f"r{rank}.json"), "w") as f:
        json.dump({"max": got, "digests": gathered}, f)
    dist.destroy_process_group()


def test_two_gloo_ranks_reduce_time_and_draw_distinct_batches(tmp_path):
    port = _free_port()
    mp.start_processes(_worker, args=(2, port, str(tmp_path)), nprocs=2, start_method="spawn", join=True)
    res = [json.load(open(tmp_path / f"r{r}.json")) for r in range(2)]
    assert res[0]["max"] == res[1]["max"] == 4.0
    assert res[0]["digests"] == res[1]["digests"]
    assert res[0]["digests"][0] != res[0]["digests"][1]


def test_whole_job_throughput_formula():
    import bench
    # 2 ranks x 1e12 FLOP per step in 4 ms -> 500 TFLOP/s for the whole job
    assert abs(bench.whole_job_tflops(2, 1e12, 4.0) - 500.0) < 1e-9
    assert bench.max_over_ranks(3.0, torch.device("cpu")) == 3.0   # not distributed


def test_rank0_replica_is_the_workload_itself():
    import workloads
    w = workloads.TINY
    assert workloads.replica_seed(w, 0) == w.seed
    a = workloads.workload_inputs(w)[0]
    b = workloads.workload_inputs(w, rank=0)[0]
    assert torch.equal(a, b)


def test_reference_arm_leaves_other_ranks_idle(monkeypatch, capsys):
    import bench
    import workloads
    monkeypatch.setenv("RANK", "1")
    monkeypatch.setenv("WORLD_SIZE", "2")

    class Args:
        steps, warmup, ref_seconds = 1, 0, 0.01
    bench.run_reference(Args, workloads.TINY)
    assert capsys.readouterr().out == ""
