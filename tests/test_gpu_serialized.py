"""Copy-engine calls finish when the streams run one after the other.

In CE mode a call queues shard copies and stream-ordered flag writes on the
side stream and a GEMM on the main stream that waits (bounded) on those flags.
The copies are queued first, so the call completes whatever order the two
streams take -- also fully serialised, as under CUDA_LAUNCH_BLOCKING=1, a
profiler's replay, or a host thread that stalls between launches.  The child
process below runs the single-rank and the all-ranks AG-GEMM in CE mode, pull
and push, with every launch blocking and a 50 ms bound on each wait: a call that queued its
GEMM first would run out of time (TDG_ERR_TIMEOUT) instead of returning the
oracle's bits.
"""
import os
import subprocess
import sys

import pytest

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

CHILD = r"""
import sys
import numpy as np
import torch
sys.path.insert(0, {root!r}); sys.path.insert(0, {tests!r})
import oracle
from tile_centric_comm_gb300 import synth
from gpu_util import AGCase, to_bits
from test_gpu_ag_all import AGAllCase

T = 50_000_000
inp = synth.ag_inputs(4, 512, 128, 264, "int2", seed=31)
_, C16 = oracle.ag_gemm(inp.shards, inp.B)
case = AGCase(inp)
for rank in (0, 3):
    for push in (False, True):
        got, st = case.run(rank=rank, mode="ce", timeout_ns=T, check_status=False, push=push)
        assert st["code"] == 0, ("single rank", rank, push, st)
        assert np.array_equal(got, C16), ("single rank", rank, push)
aa = synth.ag_all_inputs(4, 512, 128, 264, "int2", seed=32)
case = AGAllCase(aa)
for rep, push in ((0, False), (1, True)):
    got, st = case.run(mode="ce", timeout_ns=T, check_status=False, push=push)
    assert st["code"] == 0, ("all ranks", rep, st)
    for r in range(4):
        assert np.array_equal(got[r], oracle.ag_gemm(aa.shards, aa.Bs[r])[1]), ("all ranks", r)
        assert np.array_equal(to_bits(case.gathered(r)), np.concatenate(aa.shards)), ("gathered", r)
print("serialized ok")
"""


def test_ce_calls_complete_with_blocking_launches():
    env = dict(os.environ, CUDA_LAUNCH_BLOCKING="1")
    code = CHILD.format(root=ROOT, tests=os.path.join(ROOT, "tests"))
    p = subprocess.run([sys.executable, "-c", code], cwd=ROOT, env=env, capture_output=True,
                       text=True, timeout=600)
    assert p.returncode == 0, p.stdout[-2000:] + p.stderr[-4000:]
    assert "serialized ok" in p.stdout
