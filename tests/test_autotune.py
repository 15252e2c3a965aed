"""The distributed autotuner's host logic on CPU: two gloo ranks that measured
different times must both pick the candidate whose slowest rank is fastest.
(The timing itself is exercised on the GPU in test_gpu_autotune.py.)"""
import os
import socket

import pytest
import torch.distributed as dist
import torch.multiprocessing as mp

from tile_centric_comm_gb300 import autotune


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _worker(rank, world, port, q):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        # rank 0 finds candidate 1 fastest, rank 1 finds candidate 2 fastest;
        # the max over ranks is [5, 6, 4.5, 9] -> candidate 2 everywhere
        times = {0: [5.0, 1.0, 4.5, 9.0], 1: [2.0, 6.0, 0.5, 3.0]}[rank]
        best, combined = autotune.choose(times)
        q.put((rank, best, combined))
        # the tuner caches the agreed choice under its key
        calls = []
        cfgs = [dict(x=i) for i in range(4)]
        autotune.clear_cache()
        autotune._cache[("k",)] = cfgs[best]
        got, table = autotune.tune(("k",), cfgs, lambda c: calls.append(c))
        assert got == cfgs[best] and table == [] and calls == []
    finally:
        dist.destroy_process_group()


def test_ranks_agree_on_min_of_max():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    ps = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in ps:
        p.start()
    res = [q.get(timeout=120) for _ in range(2)]
    for p in ps:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, best, combined in res:
        assert best == 2
        assert combined == [5.0, 6.0, 4.5, 9.0]


def test_single_process_ties_go_to_the_earlier_candidate():
    best, t = autotune.choose([3.0, 1.0, 1.0])
    assert best == 1 and t == [3.0, 1.0, 1.0]


def test_candidate_lists():
    ag = autotune.ag_candidates(8192)
    assert dict(mode="ce", producers=0, signal_rows=0, source_order=1) in ag
    assert sum(1 for c in ag if c["mode"] == "sm") == 6
    assert [c["owner_block"] for c in autotune.rs_candidates(8)] == [1, 2, 4, 8]
