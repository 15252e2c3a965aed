"""AllGather+GEMM with float32 output (c_f32): C holds the fp32 accumulator
itself, with no rounding, against the oracle's exact sums."""
import numpy as np
import pytest
import torch

import oracle
from tile_centric_comm_gb300 import synth, tdg
from gpu_util import AGCase, bf16_f64

pytestmark = pytest.mark.gpu

# GEMM cluster shapes: two-pair clusters, CTA pairs, one CTA per tile
SHAPES = [4, 2, 1]


@pytest.mark.parametrize("cluster", SHAPES)
@pytest.mark.parametrize("b_layout", [tdg.B_KN, tdg.B_NK])
def test_integer_sums_exact_in_every_mode(cluster, b_layout):
    # integers in [-2, 2] and K = 1032: |sums| <= 4128, exact in fp32 but not
    # in bf16, so the fp32 output is the oracle's exact value and bf16 is not
    inp = synth.ag_inputs(2, 512, 1032, 264, "int2", seed=41)
    C64, C16 = oracle.ag_gemm(inp.shards, inp.B)
    assert not np.array_equal(bf16_f64(C16), C64)     # bf16 would have rounded
    case = AGCase(inp, b_layout=b_layout, ll=True, c_f32=True)
    for mode in ("sm", "serial", "ce", "ll"):
        got, _ = case.run(rank=1, mode=mode, ll_off=case.ll_off, cluster=cluster)
        assert got.dtype == np.float32
        assert np.array_equal(got.astype(np.float64), C64), mode


@pytest.mark.parametrize("W,Ms,K,N", [
    (3, 96, 136, 264),      # Ms not a multiple of 128, ragged m and n tails
    (4, 1024, 200, 712),    # two-pair clusters, ragged k block, last n tile 200 wide
])
def test_float_within_fp32_summation_bound(W, Ms, K, N):
    inp = synth.ag_inputs(W, Ms, K, N, "normal", seed=W + N)
    C64, _ = oracle.ag_gemm(inp.shards, inp.B)
    A = np.concatenate([bf16_f64(s) for s in inp.shards])
    mag = np.abs(A) @ np.abs(bf16_f64(inp.B))
    # bf16 products are exact in fp32; each of the K additions may lose up to
    # 2^-23 relative (the tensor core's rounding of its sums is not specified)
    bound = 2 * (K + 1) * 2.0 ** -24 * mag
    case = AGCase(inp, c_f32=True)
    for mode in ("sm", "ce"):
        got, _ = case.run(rank=W - 1, mode=mode)
        assert np.all(np.abs(got.astype(np.float64) - C64) <= bound), mode


def test_zero_k_writes_float_zeros_and_bf16_c_is_refused():
    inp = synth.ag_inputs(2, 64, 8, 16, "int2", seed=2)
    case = AGCase(inp, c_f32=True)
    case.C.fill_(7.0)
    tdg.ag_gemm(case.symm, 0, 64, 0, 16, case.a_off, case.g_off, case.B, case.C, c_f32=True)
    torch.cuda.synchronize()
    assert not case.C.cpu().numpy().any()             # K == 0: C = 0 over all M x N floats
    c16 = torch.empty((128, 16), dtype=torch.bfloat16, device="cuda")
    with pytest.raises(TypeError, match="float32"):
        tdg.ag_gemm(case.symm, 0, 64, 8, 16, case.a_off, case.g_off, case.B, c16, c_f32=True)
    assert case.symm.status()["code"] == 0
