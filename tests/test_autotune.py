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
        # over the real candidate list: each rank times every schedule
        # differently; both settle on the same one, the min over candidates of
        # the max over ranks
        cands = autotune.ag_candidates(8192, 1024)
        local = [float((hash(tuple(sorted(c.items()))) % 97) + 13 * rank * (i % 5))
                 for i, c in enumerate(cands)]
        b2, comb2 = autotune.choose(local)
        q.put((rank, "ag", b2, comb2))
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
    res = [q.get(timeout=120) for _ in range(4)]
    for p in ps:
        p.join(timeout=60)
        assert p.exitcode == 0
    plain = [r for r in res if len(r) == 3]
    for rank, best, combined in plain:
        assert best == 2
        assert combined == [5.0, 6.0, 4.5, 9.0]
    ag = [r for r in res if len(r) == 4]
    assert len(ag) == 2 and ag[0][2] == ag[1][2] and ag[0][3] == ag[1][3]
    comb = ag[0][3]
    assert comb[ag[0][2]] == min(comb)


def test_single_process_ties_go_to_the_earlier_candidate():
    best, t = autotune.choose([3.0, 1.0, 1.0])
    assert best == 1 and t == [3.0, 1.0, 1.0]


def test_candidate_lists():
    # the Qwen-32B up-projection shape: Ms = 1024 allows every cluster shape
    ag = autotune.ag_candidates(8192, 1024)
    assert dict(mode="ce", producers=0, signal_rows=0, source_order=1, push=1, cluster=2, stages=4) in ag
    # sm: 2 orders x 2 push x 2 clusters x 2 stage counts x 3 producer counts
    assert sum(1 for c in ag if c["mode"] == "sm") == 48
    assert sum(1 for c in ag if c["mode"] == "ce") == 16
    assert {c["cluster"] for c in ag} == {4, 2}
    # Ms = 256: no two-pair clusters; M = 128: one CTA per tile, at most 4 stages
    assert {c["cluster"] for c in autotune.ag_candidates(2048, 256)} == {2}
    small = autotune.ag_candidates(128, 64, stages=(0, 4, 6))
    assert {c["cluster"] for c in small} == {1} and {c["stages"] for c in small} == {0, 4}
    rs = autotune.rs_candidates(8, 1024)
    assert sorted({c["owner_block"] for c in rs}) == [1, 2, 4, 8]
    assert all(c["owner_block"] == 1 for c in rs if c["order"] == 1)
    assert dict(owner_block=2, order=0, cluster=4, stages=0) in rs
    assert {c["cluster"] for c in autotune.rs_candidates(8, 256)} == {2}
