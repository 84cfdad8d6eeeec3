"""Multi-process host logic of bench.py on CPU (gloo, world size 2).

The scan shards over independent channels / heads with no data exchange;
the only cross-rank steps are the barrier and the max-over-ranks timing.
These run here as two gloo processes on the CPU.
"""
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import bench


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    r, w, local = bench.dist_env()
    assert (r, w, local) == (rank, world, rank)
    # rank r "took" 10 + r ms for the timed region and 20 - r ms end to end
    ms, e2e = bench.max_over_ranks([10.0 + rank, 20.0 - rank], world, torch.device("cpu"))
    dist.barrier()
    out[rank] = (ms, e2e, bench.shard_seed(1, rank))
    dist.destroy_process_group()


def test_max_over_ranks_and_shards_with_gloo():
    world = 2
    port = _free_port()
    with mp.Manager() as m:
        out = m.dict()
        mp.spawn(_worker, args=(world, port, out), nprocs=world, join=True)
        res = dict(out)
    assert res[0][:2] == (11.0, 20.0) and res[1][:2] == (11.0, 20.0)
    assert res[0][2] != res[1][2]           # each rank draws its own batch


def test_single_rank_is_identity():
    assert bench.max_over_ranks([3.0, 4.0], 1, torch.device("cpu")) == [3.0, 4.0]


def test_reference_arm_runs_on_cpu(capsys, monkeypatch):
    # The reference arm is the fp64 oracle on host cores: it needs no GPU.
    import json
    monkeypatch.setattr("sys.argv", ["bench.py", "--impl", "reference", "--steps", "2",
                                     "--warmup", "1", "--workload", "diag_f32_Bs2_L64_ED64_N16"])
    bench.main()
    line = json.loads(capsys.readouterr().out.strip().splitlines()[-1])
    assert line["impl"] == "reference" and line["value"] > 0
    assert line["e2e"]["h2d_bytes_per_step"] == 0 and line["cpu_baseline"]["kind"] == "oracle"
