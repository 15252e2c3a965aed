"""The autotuner on the GPU: it times real candidates through the C ABI and
its choice computes the same result as the oracle."""
import numpy as np
import pytest

import oracle
from tile_centric_comm_gb300 import autotune, synth, tdg
from gpu_util import AGCase, RSCase, assert_close

pytestmark = pytest.mark.gpu


def test_tune_ag_and_rs_small():
    inp = synth.ag_inputs(4, 256, 256, 512, "normal", seed=2)
    C64, _ = oracle.ag_gemm(inp.shards, inp.B)
    case = AGCase(inp)
    cands = autotune.ag_candidates(case.M, producers=(8,), source_orders=(0, 1))

    def run(cfg):
        tdg.ag_gemm(case.symm, 1, inp.Ms, inp.K, inp.N, case.a_off, case.g_off, case.B, case.C,
                    side_stream=_side, **cfg)

    import torch
    _side = torch.cuda.Stream()
    best, table = autotune.tune(("ag", 4, 256, 256, 512), cands, run, warmup=1, iters=3,
                                use_cache=False)
    assert best in cands and len(table) == len(cands) and all(r["ms"] > 0 for r in table)
    got, _ = case.run(rank=1, **best)
    assert_close(got, C64)

    rs = synth.rs_inputs(4, 1024, 128, 256, "normal", seed=3)
    out64, _ = oracle.gemm_rs(rs.As, rs.Bs)
    rcase = RSCase(rs)

    def run_rs(cfg):
        tdg.gemm_rs(rcase.symm, rs.M, rs.K, rs.N, rcase.a_off, rcase.b_off, rcase.stage_off,
                    rcase.out_off, **cfg)

    best, table = autotune.tune(("rs", 4, 1024, 128, 256), autotune.rs_candidates(4), run_rs,
                                warmup=1, iters=3, use_cache=False)
    got, _ = rcase.run(**best)
    assert_close(got, out64)
