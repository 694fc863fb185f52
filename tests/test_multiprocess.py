"""Multi-rank host logic of bench.py on CPU (gloo, world size 2).

Requests shard across ranks with no data-path collective: each rank resolves its own batch
(seed offset by rank) and only the step time is reduced (max over ranks); the job's value is
every rank's rows over that time. Each rank places its host pools on the memory node beside its
GPU (a fake GPU -> node map here) before their pages are touched. The reference arm prints from
rank 0 alone.
"""
import os
import socket

import numpy as np
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


FAKE_NODES = {0: 0, 1: 0}  # GPU -> host memory node, as a two-GPU rank pair on one CPU would have


def _worker(rank, ws, port, out):
    import sys
    sys.path[:0] = [ROOT]
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(ws))
    dist.init_process_group("gloo", rank=rank, world_size=ws)
    import bench
    import workloads as W
    # whole-job throughput as the bench reports it: every rank's rows over the slowest time
    rows = 4096  # the same batch shape on every rank
    value = bench.job_throughput(rows, 1.0 + rank, ws)  # rank 1 is the slower one
    # each rank's pools go to the node its GPU sits beside, before any page is touched
    node = bench.rank_numa_node(rank, query=FAKE_NODES.__getitem__)
    # a pool smaller than a huge page: an anonymous mapping on any host (no driver-pinned fallback)
    wl = W.make("tiny", 1000 * rank, requests=2, steps=2, seq0=(1000, 100))
    views, pools = bench.alloc_host_pools(wl, node)
    addr = "%x" % pools[0][0].ctypes.data
    policy = next((ln.split()[1] for ln in open("/proc/self/numa_maps") if ln.startswith(addr + " ")), None)
    filled = bool(np.array_equal(wl.host_row_bytes_of(views[0], int(wl.host_cache_locs[0, 5])),
                                 wl.rows(0, 0, [5])[0]))
    first = wl.top_k_tokens(1)[0, :8].tolist()
    gathered = [None] * ws
    dist.all_gather_object(gathered, first)
    out[rank] = (value, gathered[0] != gathered[1], node, policy, filled)
    bench.barrier(ws)
    dist.destroy_process_group()


def test_two_ranks_job_value_numa_placement_and_independent_shards():
    port = _free_port()
    manager = mp.Manager()
    out = manager.dict()
    mp.spawn(_worker, args=(2, port, out), nprocs=2, join=True)
    for rank in range(2):
        value, differ, node, policy, filled = out[rank]
        assert value == pytest.approx(2 * 4096 / 2.0)  # 2 ranks x 4096 rows in the slower rank's 2 s
        assert differ  # ranks resolve different synthetic batches
        assert node == FAKE_NODES[rank]
        assert policy == f"prefer:{node}", policy  # the pool's pages come from the rank's node
        assert filled


def test_rank_numa_node_without_an_answer():
    import sys
    sys.path[:0] = [ROOT]
    import bench

    def no_device(dev):
        raise RuntimeError("no CUDA device")
    assert bench.rank_numa_node(0, query=no_device) == -1
    assert bench.rank_numa_node(3, query={3: 7}.__getitem__) == 7


def _ref_worker(rank, ws, port, out):
    import contextlib
    import io
    import sys
    sys.path[:0] = [ROOT]
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(ws))
    import bench
    args = type("A", (), dict(impl="reference", config="tiny", seed=0, steps=2, warmup=1, gpus=ws,
                              host_layout="auto", rehearsal="disjoint"))()
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


def _rules_worker(rank, ws, port, out):
    import sys
    sys.path[:0] = [ROOT]
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(ws))
    dist.init_process_group("gloo", rank=rank, world_size=ws)
    import bench
    # rank 1 stalls in its first pass (one step at 10x), rank 0 never does
    first = [1.0, 1.0, 1.1, 10.0 if rank == 1 else 1.0]
    second = [1.2, 1.2, 1.3, 1.2] if rank == 0 else [0.9, 0.9, 1.0, 0.9]
    stalled_first = bench.stalled(first, ws)
    # a pass slow from end to end on rank 0 only, against the graph-replayed median 1.0 ms
    slow = bench.stalled([5.0, 5.0, 5.1] if rank == 0 else [1.0, 1.0, 1.1], ws, 1.0)
    # no pass was clean: the one with the lowest median over the ranks, the same on every rank
    picked = bench.pick_pass([first, second], False, ws)
    out[rank] = (stalled_first, slow, picked)
    bench.barrier(ws)
    dist.destroy_process_group()


def test_two_ranks_agree_on_stalled_passes_and_the_reported_one():
    port = _free_port()
    manager = mp.Manager()
    out = manager.dict()
    mp.spawn(_rules_worker, args=(2, port, out), nprocs=2, join=True)
    assert out[0] == out[1]  # every rank takes the same decision
    stalled_first, slow, picked = out[0]
    assert stalled_first  # rank 1's outlier stalls the pass for both
    assert slow  # rank 0's slow pass does too
    assert picked == 0  # medians over ranks: first max(1.0, 1.05) = 1.05, second max(1.2, 0.9) = 1.2
