"""The autotuner on the GPU: it times real candidates through the C ABI, and
every candidate schedule -- mode, source order, push or pull, GEMM cluster
shape, ring stages, producer count, owner block and tile order -- computes
the oracle's bits on integer inputs, the tuned one included."""
import numpy as np
import pytest

import oracle
from tile_centric_comm_gb300 import autotune, synth, tdg
from gpu_util import AGCase, RSCase, assert_close

pytestmark = pytest.mark.gpu


def test_tune_ag_and_rs_small():
    inp = synth.ag_inputs(4, 512, 256, 520, "normal", seed=2)
    C64, _ = oracle.ag_gemm(inp.shards, inp.B)
    case = AGCase(inp)
    cands = autotune.ag_candidates(case.M, inp.Ms, producers=(0, 8))
    assert {c["cluster"] for c in cands} == {4, 2}

    def run(cfg):
        tdg.ag_gemm(case.symm, 1, inp.Ms, inp.K, inp.N, case.a_off, case.g_off, case.B, case.C,
                    side_stream=_side, **cfg)

    import torch
    _side = torch.cuda.Stream()
    best, table = autotune.tune(("ag", 4, 512, 256, 520), cands, run, warmup=1, iters=3,
                                use_cache=False)
    assert best in cands and len(table) == len(cands) and all(r["ms"] > 0 for r in table)
    got, _ = case.run(rank=1, **best)
    assert_close(got, C64)

    rs = synth.rs_inputs(4, 2048, 128, 520, "normal", seed=3)
    out64, _ = oracle.gemm_rs(rs.As, rs.Bs)
    rcase = RSCase(rs)

    def run_rs(cfg):
        tdg.gemm_rs(rcase.symm, rs.M, rs.K, rs.N, rcase.a_off, rcase.b_off, rcase.stage_off,
                    rcase.out_off, **cfg)

    rc = autotune.rs_candidates(4, 512)
    assert {c["cluster"] for c in rc} == {4, 2}
    best, table = autotune.tune(("rs", 4, 2048, 128, 520), rc, run_rs, warmup=1, iters=3, use_cache=False)
    got, _ = rcase.run(**best)
    assert_close(got, out64)


def test_every_candidate_bit_exact_on_integers():
    inp = synth.ag_inputs(4, 512, 136, 264, "int2", seed=8)
    _, C16 = oracle.ag_gemm(inp.shards, inp.B)
    case = AGCase(inp)
    for cfg in autotune.ag_candidates(case.M, inp.Ms, producers=(0, 4)):
        got, _ = case.run(rank=2, **cfg)
        assert np.array_equal(got, C16), cfg
    rs = synth.rs_inputs(4, 2048, 64, 264, "int2", seed=9)
    _, out16 = oracle.gemm_rs(rs.As, rs.Bs)
    rcase = RSCase(rs)
    for cfg in autotune.rs_candidates(4, 512):
        got, _ = rcase.run(mode="sm", **cfg)
        assert np.array_equal(got, out16), cfg
