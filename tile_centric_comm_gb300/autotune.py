"""Distributed autotuner for the tile-centric kernels.

The Triton-distributed paper summary (hyper.ai, arXiv 2504.19442, section 方法)
describes an autotuner made for distributed kernels: it accounts for the
synchronisation that launching them needs and synchronises the tuning results
across devices, so that every device settles on the same, globally best
configuration.  This module does that for the knobs of this library:

* every candidate configuration is run through the C ABI (``run(cfg)``),
  with warm-up, and timed with CUDA events on the launching stream;
* under ``torch.distributed`` the per-rank times are combined with a MAX
  all-reduce -- the job is as slow as its slowest rank -- and every rank picks
  the candidate with the lowest combined time (ties to the earlier
  candidate), so all ranks agree without any further message;
* the decision is cached per (operation, shape) key.

The host logic (``choose``) is separate from the timing so that it can be
tested without a GPU.
"""
from __future__ import annotations

import itertools
import statistics
from typing import Callable, Dict, List, Optional, Sequence, Tuple

_cache: Dict[tuple, dict] = {}


def choose(times: Sequence[float], group=None) -> Tuple[int, List[float]]:
    """Index of the best candidate after combining `times` over the ranks of
    `group` (max over ranks).  Without torch.distributed, the local times."""
    t = [float(x) for x in times]
    try:
        import torch
        import torch.distributed as dist
        if dist.is_available() and dist.is_initialized():
            ten = torch.tensor(t, dtype=torch.float64)
            if dist.get_backend(group) == "nccl":
                ten = ten.cuda()
            dist.all_reduce(ten, op=dist.ReduceOp.MAX, group=group)
            t = ten.cpu().tolist()
    except ImportError:  # pragma: no cover
        pass
    best = min(range(len(t)), key=lambda i: (t[i], i))
    return best, t


def time_candidate(run: Callable[[dict], None], cfg: dict, warmup: int = 2, iters: int = 5,
                   flush=None, pause: float = 0.0) -> float:
    """Median device time (ms) of `run(cfg)` over `iters` launches, queued
    back to back (the host waits once): the GPU stays busy as it does in use,
    so a schedule that saves DRAM traffic, and with it power and clock, is
    seen to; launches timed one at a time from an idle GPU start at full
    clock and hide that.  `pause` seconds of idle GPU before the timed
    launches give every candidate the same starting temperature and power
    state (a burst of work, as one serving step is)."""
    import time
    import torch
    stream = torch.cuda.current_stream()
    if pause > 0:
        torch.cuda.synchronize()
        time.sleep(pause)
    for _ in range(warmup):
        run(cfg)
    evs = []
    for _ in range(iters):
        if flush is not None:
            flush()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        run(cfg)
        b.record(stream)
        evs.append((a, b))
    torch.cuda.synchronize()
    return statistics.median(a.elapsed_time(b) for a, b in evs)


def tune(key: tuple, candidates: List[dict], run: Callable[[dict], None], group=None,
         warmup: int = 2, iters: int = 5, flush=None, use_cache: bool = True,
         rounds: int = 3, pause: float = 0.0) -> Tuple[dict, List[dict]]:
    """Time every candidate, agree on the best across ranks, cache it.
    The candidates are timed in `rounds` rounds, the order rotated every
    round, and each keeps the median of its rounds: a GPU's clock drifts over
    a long run (the power cap), which would otherwise favour whichever
    candidate runs first.  Returns (best config, table of {cfg, ms})."""
    if use_cache and key in _cache:
        return _cache[key], []
    per = [[] for _ in candidates]
    n = len(candidates)
    for r in range(max(1, rounds)):
        start = (r * n) // max(1, rounds)
        for j in range(n):
            i = (start + j) % n
            per[i].append(time_candidate(run, candidates[i], warmup if r == 0 else 1, iters, flush, pause))
    times = [statistics.median(t) for t in per]
    best, combined = choose(times, group)
    table = [dict(cfg=c, ms=t) for c, t in zip(candidates, combined)]
    _cache[key] = candidates[best]
    return candidates[best], table


def _clusters(allow2: bool, allow4: bool) -> List[int]:
    """GEMM cluster shapes a shape allows, the library's default first."""
    out = []
    if allow4:
        out.append(4)
    if allow2:
        out.append(2)
    return out or [1]


def ag_candidates(M: int, Ms: int = 0, modes=("ce", "sm"), producers=(0, 8, 16), signal_rows=(0,),
                  source_orders=(0, 1), pushes=(0, 1), clusters=None, stages=(0, 4)) -> List[dict]:
    """AllGather+GEMM schedules: mode x source order x push x GEMM cluster
    shape x ring stages (x producer CTAs in SM mode; 0 = the library's
    default count).  Ms = 0 leaves the cluster shape to the library."""
    if clusters is None:
        clusters = _clusters(M > 128, Ms > 0 and Ms % 512 == 0) if Ms else [0]
    out = []
    for mode, so, sr, push, cl, st in itertools.product(modes, source_orders, signal_rows, pushes, clusters,
                                                         stages):
        if cl == 1 and st > 4:
            continue
        base = dict(mode=mode, signal_rows=sr, source_order=so, push=push, cluster=cl, stages=st)
        if mode == "sm":
            for pr in producers:
                out.append(dict(base, producers=pr))
        else:
            out.append(dict(base, producers=0))
    return out


def rs_candidates(world: int, Mo: int = 0, clusters=None, stages=(0, 4), orders=(0, 1),
                  spares=(0,)) -> List[dict]:
    """GEMM+ReduceScatter schedules: owner block x tile order x GEMM cluster
    shape x ring stages (x, for order 0 on 4-CTA clusters, the tile groups
    given to CTA pairs on the SMs the clusters leave idle).  Mo (rows per
    owner) = 0 leaves the cluster shape to the library."""
    if clusters is None:
        clusters = _clusters(Mo % 256 == 0, Mo % 512 == 0) if Mo else [0]
    out = []
    for ob in (d for d in range(1, world + 1) if world % d == 0):
        for order, cl, st in itertools.product(orders, clusters, stages):
            if order == 1 and ob != 1:
                continue    # the rank-fastest order has no owner blocks
            if cl == 1 and st > 4:
                continue
            out.append(dict(owner_block=ob, order=order, cluster=cl, stages=st))
            if order == 0 and cl == 4:
                out += [dict(owner_block=ob, order=order, cluster=cl, stages=st, spare=sp)
                        for sp in spares if 0 < sp < world * world]
    return out


def clear_cache():
    _cache.clear()
