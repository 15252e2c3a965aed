"""Sizes past 32-bit byte offsets, checked on sampled outputs against the
oracle: an AllGather+GEMM whose gathered buffer is 4.3 GB, a GEMM+ReduceScatter
whose staging area is 4.3 GB per region, and the MoE routing at the largest
expert count.  Integer inputs, so every sampled value is exact."""
import numpy as np
import pytest
import torch

import oracle
from tile_centric_comm_gb300 import synth, tdg
from gpu_util import align, to_bits

pytestmark = [pytest.mark.gpu, pytest.mark.slow]


def _sample(g, hi, n):
    return np.unique(np.concatenate([g.integers(0, hi, n), [0, hi - 1]]))


@pytest.mark.parametrize("mode", ["ce", "serial"])
def test_ag_gathered_buffer_past_4gb(mode):
    W, Ms, K, N = 8, 32768, 8192, 256          # gathered: 262144 x 8192 bf16 = 4.29 GB
    M = W * Ms
    g_off = align(Ms * K * 2)
    symm = tdg.Symm(W, align(g_off + M * K * 2 + 1024), 65536)
    for r in range(W):
        symm.view(r, 0, (Ms, K), torch.bfloat16).copy_(synth.device_int2((Ms, K), seed=100 + r))
    B = synth.device_int2((K, N), seed=99)
    C = torch.empty((M, N), dtype=torch.bfloat16, device="cuda")
    side = torch.cuda.Stream() if mode == "ce" else None
    rank = 5
    tdg.ag_gemm(symm, rank, Ms, K, N, 0, g_off, B, C, mode=mode, side_stream=side)
    torch.cuda.synchronize()
    assert symm.status()["code"] == 0
    rows = _sample(np.random.default_rng(3), M, 96)
    idx = torch.from_numpy(rows).cuda()
    gathered = symm.view(rank, g_off, (M, K), torch.bfloat16)
    a_rows = torch.cat([symm.view(int(r) // Ms, 0, (Ms, K), torch.bfloat16)[int(r) % Ms][None] for r in rows])
    assert torch.equal(gathered[idx], a_rows), "gathered rows differ from their shards"
    _, want = oracle.ag_gemm([to_bits(a_rows)], to_bits(B))   # the sampled rows times B
    assert np.array_equal(to_bits(C[idx]), want)
    del symm, C, gathered
    torch.cuda.empty_cache()


@pytest.mark.parametrize("f32", [False, True])
def test_rs_staging_past_4gb(f32):
    # staging per region: 8 x 16384 x 16640 partials = 4.36 GB in bf16, 8.72 GB in fp32
    W, M, K, N = 8, 131072, 64, 16640
    inp = synth.rs_inputs(W, M, K, N, "int2", seed=7)
    Mo = M // W
    a_off, b_off = 0, align(M * K * 2)
    s_off = align(b_off + K * N * 2)
    o_off = align(s_off + tdg.gemm_rs_stage_bytes(W, M, N) * (2 if f32 else 1))
    assert tdg.gemm_rs_stage_bytes(W, M, N) > (1 << 32)
    symm = tdg.Symm(W, align(o_off + Mo * N * 2 + 1024), (Mo // 128) * ((N + 255) // 256) * 4)
    for r in range(W):
        symm.view(r, a_off, (M, K), torch.bfloat16).copy_(
            torch.from_numpy(inp.As[r].view(np.int16)).view(torch.bfloat16).cuda())
        symm.view(r, b_off, (K, N), torch.bfloat16).copy_(
            torch.from_numpy(inp.Bs[r].view(np.int16)).view(torch.bfloat16).cuda())
    g = np.random.default_rng(4)
    rows, cols = g.integers(0, M, 1500), g.integers(0, N, 1500)
    rows = np.concatenate([rows, [M - 1, 0, Mo - 1, Mo]])
    cols = np.concatenate([cols, [N - 1, 0, 255, 256]])
    # every bf16 partial is exact (|partial| <= 4K = 256); the output is the
    # round-to-nearest-even bf16 of the exact sum
    want = oracle.f64_to_bf16(oracle.gemm_rs_sampled(inp.As, inp.Bs, rows, cols))
    for mode in ("sm", "serial"):
        tdg.gemm_rs(symm, M, K, N, a_off, b_off, s_off, o_off, mode=mode, partial_f32=f32)
        torch.cuda.synchronize()
        assert symm.status()["code"] == 0
        got = np.empty(len(rows), np.uint16)
        for o in range(W):
            sel = np.nonzero(rows // Mo == o)[0]
            if len(sel):
                out = symm.view(o, o_off, (Mo, N), torch.bfloat16)
                v = out[torch.from_numpy(rows[sel] % Mo).cuda(), torch.from_numpy(cols[sel]).cuda()]
                got[sel] = to_bits(v)
        assert np.array_equal(got, want), mode
    del symm
    torch.cuda.empty_cache()


def test_moe_route_at_the_largest_expert_count():
    from test_gpu_moe import MoECase, _check_route
    W, T, H, E, k = 8, 4096, 8, 4096, 8
    inp = synth.moe_inputs(W, T, H, E, k, seed=11)
    r = oracle.moe_route(inp.topk, E)
    case = MoECase(inp)
    case.run()
    _check_route(case, r)
    recv = oracle.moe_dispatch(inp.x, r["slot"], W * T * k)
    assert np.array_equal(to_bits(case.recv), recv)
