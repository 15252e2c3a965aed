"""A tensor-parallel MLP forward (without the activation) for all W logical
ranks, composed through the C ABI: the all-ranks AllGather+GEMM writes each
rank's C_r into the heap, and the GEMM+ReduceScatter reads it there as its
A_r.  Checked against the oracle chain with the same bf16 rounding between
the two products."""
import numpy as np
import pytest
import torch

import oracle
from tile_centric_comm_gb300 import synth, tdg
from gpu_util import align, assert_close, to_bits, to_dev_bf16

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("W,Ms,H,F", [(4, 256, 128, 256), (2, 512, 192, 264), (8, 128, 64, 136)])
def test_tp_mlp_all_ranks_composed_in_the_heap(W, Ms, H, F):
    # x_r: Ms x H (rank r's rows); up: concat(x) @ Wu_r -> C_r (M x F);
    # down: out_o = rows o of sum_r C_r @ Wd_r (M x H)
    M = W * Ms
    up = synth.ag_all_inputs(W, Ms, H, F, "normal", seed=W + Ms)
    down = synth.rs_inputs(W, M, F, H, "normal", seed=W + Ms + 1)   # only the weights Wd_r are used
    a_off = 0
    g_off = align(Ms * H * 2)
    bu_off = align(g_off + M * H * 2)
    c_off = align(bu_off + H * F * 2)
    bd_off = align(c_off + M * F * 2)
    s_off = align(bd_off + F * H * 2)
    o_off = align(s_off + tdg.gemm_rs_stage_bytes(W, M, H))
    n_tiles = (H + 255) // 256
    symm = tdg.Symm(W, align(o_off + Ms * H * 2 + 1024), max(1024, M, (Ms // 128) * n_tiles * 4))
    for r in range(W):
        symm.view(r, a_off, (Ms, H), torch.bfloat16).copy_(to_dev_bf16(up.shards[r]))
        symm.view(r, bu_off, (H, F), torch.bfloat16).copy_(to_dev_bf16(up.Bs[r]))
        symm.view(r, bd_off, (F, H), torch.bfloat16).copy_(to_dev_bf16(down.Bs[r]))
    side = torch.cuda.Stream()
    for mode in ("overlapped", "serial"):
        for o in range(W):
            symm.view(o, o_off, (Ms, H), torch.int16).fill_(0x7FC1)
        tdg.ag_gemm_all_ranks(symm, Ms, H, F, a_off, g_off, bu_off, c_off,
                              mode="ce" if mode == "overlapped" else "serial",
                              side_stream=side if mode == "overlapped" else None)
        tdg.gemm_rs(symm, M, F, H, c_off, bd_off, s_off, o_off, mode="sm" if mode == "overlapped" else "serial")
        torch.cuda.synchronize()
        assert symm.status()["code"] == 0
        C16 = [oracle.ag_gemm(up.shards, up.Bs[r])[1] for r in range(W)]
        # each C_r is exactly the oracle's rounding of the first product ...
        for r in range(W):
            assert_close(to_bits(symm.view(r, c_off, (M, F), torch.bfloat16)),
                         oracle.ag_gemm(up.shards, up.Bs[r])[0])
        # ... and the output is the second product of the device's C_r
        C_dev = [to_bits(symm.view(r, c_off, (M, F), torch.bfloat16)) for r in range(W)]
        out64, _ = oracle.gemm_rs(C_dev, down.Bs)
        got = np.stack([to_bits(symm.view(o, o_off, (Ms, H), torch.bfloat16)) for o in range(W)])
        assert_close(got, out64)
        # and within tolerance of the chain through the oracle's own C_r
        chain64, _ = oracle.gemm_rs(C16, down.Bs)
        assert_close(got, chain64)
