"""Host threads: different heaps used from different host threads at once
(the documented contract: a handle is thread-compatible, different handles
may be used concurrently).  Each thread runs its own operation on its own
stream many times; every result must still be the oracle's bits."""
import threading

import numpy as np
import pytest
import torch

import oracle
from tile_centric_comm_gb300 import synth, tdg
from gpu_util import AGCase, RSCase, to_bits

pytestmark = pytest.mark.gpu


def test_two_threads_two_heaps():
    ag_inp = synth.ag_inputs(4, 512, 128, 264, "int2", seed=51)
    rs_inp = synth.rs_inputs(4, 2048, 64, 264, "int2", seed=52)
    _, C16 = oracle.ag_gemm(ag_inp.shards, ag_inp.B)
    _, out16 = oracle.gemm_rs(rs_inp.As, rs_inp.Bs)
    ag, rs = AGCase(ag_inp), RSCase(rs_inp)
    errors = []

    def run_ag():
        try:
            s, side = torch.cuda.Stream(), torch.cuda.Stream()
            with torch.cuda.stream(s):
                for i in range(20):
                    mode = ("sm", "ce", "serial")[i % 3]
                    tdg.ag_gemm(ag.symm, i % 4, 512, 128, 264, ag.a_off, ag.g_off, ag.B, ag.C, mode=mode,
                                side_stream=side if mode == "ce" else None)
                s.synchronize()
        except Exception as e:  # pragma: no cover - reported below
            errors.append(e)

    def run_rs():
        try:
            s = torch.cuda.Stream()
            with torch.cuda.stream(s):
                for i in range(20):
                    tdg.gemm_rs(rs.symm, 2048, 64, 264, rs.a_off, rs.b_off, rs.stage_off, rs.out_off,
                                mode="sm" if i % 2 == 0 else "serial", partial_f32=False)
                s.synchronize()
        except Exception as e:  # pragma: no cover
            errors.append(e)

    threads = [threading.Thread(target=run_ag), threading.Thread(target=run_rs)]
    for t in threads:
        t.start()
    for t in threads:
        t.join()
    torch.cuda.synchronize()
    assert not errors, errors
    assert ag.symm.status()["code"] == 0 and rs.symm.status()["code"] == 0
    assert np.array_equal(to_bits(ag.C), C16)
    assert np.array_equal(np.stack([to_bits(rs.out(o)) for o in range(4)]), out16)
