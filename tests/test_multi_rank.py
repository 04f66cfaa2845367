"""The multi-GPU bench path on CPU: two gloo ranks, each with its own replica
of the workload (weak scaling), and the max-over-ranks timing reduction.  No
data-path collective exists on the hot path: the ranks share no data."""

import os
import socket

import numpy as np
import torch
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _rank_main(rank, world, port, q):
    import bench
    from workloads import WORKLOADS, generate
    dist.init_process_group("gloo", init_method="tcp://127.0.0.1:%d" % port, rank=rank,
                            world_size=world)
    w = WORKLOADS["llama3_8b_128k_b1"]
    wr = bench.replica_workload(w, rank)
    g = generate(wr, N=300)
    times = bench.max_over_ranks([1.0 + rank, 10.0 - rank], dist, "cpu")
    q.put((rank, wr.seeds, int(g["K"][0, 0, 5, 3]), times))
    dist.barrier()
    dist.destroy_process_group()


def test_two_rank_replicas_and_timing_reduction():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    (r0, seeds0, k0, t0), (r1, seeds1, k1, t1) = res
    assert seeds0 != seeds1           # each rank decodes its own sequences
    assert t0 == t1 == [2.0, 10.0]    # max over ranks, seen by every rank


def test_gpus_flag_relaunches_under_torch_distributed_run(monkeypatch):
    # `bench.py --gpus 4` started as one process re-executes itself as four
    # ranks (rendezvous on 127.0.0.1) with the same arguments; a rank (with
    # WORLD_SIZE set) or --gpus 1 runs in place.
    import bench
    monkeypatch.delenv("WORLD_SIZE", raising=False)
    seen = []
    args = bench.parse(["--gpus", "4", "--steps", "7", "--warmup", "3"])
    rc = bench.maybe_relaunch(args, ["--gpus", "4", "--steps", "7", "--warmup", "3"],
                              run=lambda cmd: seen.append(cmd) or 0)
    assert rc == 0 and len(seen) == 1
    cmd = seen[0]
    i = cmd.index("-m")
    assert cmd[i + 1] == "torch.distributed.run"
    assert cmd[cmd.index("--nproc-per-node") + 1] == "4"
    assert cmd[cmd.index("--master-addr") + 1] == "127.0.0.1"
    assert int(cmd[cmd.index("--master-port") + 1]) > 0
    assert cmd[-7].endswith("bench.py") and cmd[-6:] == ["--gpus", "4", "--steps", "7", "--warmup", "3"]
    assert bench.maybe_relaunch(bench.parse(["--gpus", "1"]), [], run=seen.append) is None
    monkeypatch.setenv("WORLD_SIZE", "4")
    assert bench.maybe_relaunch(args, [], run=seen.append) is None
    assert len(seen) == 1
