"""Multi-rank host logic of bench.py on CPU (gloo, world size 2).

Requests shard across ranks with no data-path collective: each rank resolves its own batch
(seed offset by rank) and only the step time is reduced (max over ranks). The reference arm
prints from rank 0 alone.
"""
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _worker(rank, ws, port, out):
    import sys
    sys.path[:0] = [ROOT]
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(ws))
    dist.init_process_group("gloo", rank=rank, world_size=ws)
    import bench
    import workloads as W
    local_time = 1.0 + rank  # rank 1 is the slower one
    t = bench.max_over_ranks(local_time, ws)
    wl = W.make("dsa", 0 + 1000 * rank, requests=2, steps=2)
    first = wl.top_k_tokens(1)[0, :8].tolist()
    gathered = [None] * ws
    dist.all_gather_object(gathered, first)
    out[rank] = (t, gathered[0] != gathered[1])
    bench.barrier(ws)
    dist.destroy_process_group()


def test_two_ranks_max_time_and_independent_shards():
    port = _free_port()
    manager = mp.Manager()
    out = manager.dict()
    mp.spawn(_worker, args=(2, port, out), nprocs=2, join=True)
    for rank in range(2):
        t, differ = out[rank]
        assert t == 2.0  # every rank reports the slowest rank's time
        assert differ  # ranks resolve different synthetic batches
    # whole-job throughput: all ranks' rows over the max time
    rows_per_rank = 65536 * 4
    assert 2 * rows_per_rank / 2.0 == rows_per_rank


def _ref_worker(rank, ws, port, out):
    import contextlib
    import io
    import sys
    sys.path[:0] = [ROOT]
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(ws))
    import bench
    args = type("A", (), dict(impl="reference", config="tiny", seed=0, steps=2, warmup=1, gpus=ws))()
    dist.init_process_group("gloo", rank=rank, world_size=ws)
    buf = io.StringIO()
    with contextlib.redirect_stdout(buf):
        bench.run_reference(args, ws, rank)
    out[rank] = buf.getvalue()
    dist.destroy_process_group()


def test_reference_arm_prints_from_rank0_only():
    port = _free_port()
    manager = mp.Manager()
    out = manager.dict()
    mp.spawn(_ref_worker, args=(2, port, out), nprocs=2, join=True)
    import json
    line = json.loads(out[0].strip().splitlines()[-1])
    assert line["impl"] == "reference" and line["value"] > 0 and line["cpu_baseline"]["kind"] == "oracle"
    assert out[1].strip() == ""
