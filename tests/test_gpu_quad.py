"""GPU parity of the GEMM on clusters of two CTA pairs (512-row tiles, each B
slice fetched by one pair and multicast to the other) against the CPU oracle
and against the same call on single pairs (cluster 2)."""
import numpy as np
import pytest

import oracle
from tile_centric_comm_gb300 import synth, tdg
from gpu_util import AGCase, RSCase, assert_close

pytestmark = pytest.mark.gpu


# Ms = 512: one 512-row tile per shard.  N = 3200: the last n tile is 128 wide
# (one 64-column slice per CTA, fetched by the first pair only); N = 520: last
# tile 8 wide; N = 456: last tile 200 wide (two slices, the second partial);
# N = 256: one full tile.
@pytest.mark.parametrize("b_layout", [tdg.B_KN, tdg.B_NK])
@pytest.mark.parametrize("N", [3200, 520, 456, 256])
def test_ag_integer_bit_exact_quad_and_pair(N, b_layout):
    inp = synth.ag_inputs(2, 512, 192, N, "int2", seed=N)
    _, C16 = oracle.ag_gemm(inp.shards, inp.B)
    case = AGCase(inp, b_layout=b_layout)
    for cluster in (4, 2):
        for mode in ("sm", "serial", "ce"):
            got, _ = case.run(rank=1, mode=mode, cluster=cluster)
            assert np.array_equal(got, C16), (cluster, mode)


@pytest.mark.parametrize("b_layout", [tdg.B_KN, tdg.B_NK])
def test_ag_float_parity_and_same_bits_as_pairs(b_layout):
    # W=4, Ms=1024 (two 512-row tiles per shard), K=200 (ragged k block),
    # N=712 (last n tile 200 wide).  The quad and pair kernels run the same
    # MMA sequence per output tile, so their outputs agree bit for bit.
    inp = synth.ag_inputs(4, 1024, 200, 712, "normal", seed=11)
    C64, _ = oracle.ag_gemm(inp.shards, inp.B)
    case = AGCase(inp, b_layout=b_layout)
    outs = {}
    for cluster in (4, 2):
        for rank in (0, 3):
            got, _ = case.run(rank=rank, mode="sm", cluster=cluster)
            assert_close(got, C64)
            outs[(cluster, rank)] = got
    for rank in (0, 3):
        assert np.array_equal(outs[(4, rank)], outs[(2, rank)]), rank


# Mo = M / W a multiple of 512: one or more 512-row tiles per owner.  K = 64
# keeps every bf16 partial exact, so the reduced output is exact too.
@pytest.mark.parametrize("b_layout", [tdg.B_KN, tdg.B_NK])
@pytest.mark.parametrize("W,M,N", [(2, 1024, 520), (4, 2048, 3200), (2, 2048, 456)])
def test_rs_integer_bit_exact_quad_and_pair(W, M, N, b_layout):
    inp = synth.rs_inputs(W, M, 64, N, "int2", seed=W + N)
    _, out16 = oracle.gemm_rs(inp.As, inp.Bs)
    case = RSCase(inp, b_layout=b_layout)
    for cluster in (4, 2):
        for mode in ("sm", "serial"):
            got, _ = case.run(mode=mode, cluster=cluster)
            assert np.array_equal(got, out16), (cluster, mode)


@pytest.mark.parametrize("b_layout", [tdg.B_KN, tdg.B_NK])
def test_rs_float_parity_and_same_bits_as_pairs(b_layout):
    inp = synth.rs_inputs(2, 1024, 328, 776, "normal", seed=13)
    out64, _ = oracle.gemm_rs(inp.As, inp.Bs)
    case = RSCase(inp, b_layout=b_layout)
    outs = {}
    for cluster in (4, 2):
        got, _ = case.run(mode="sm", cluster=cluster)
        assert_close(got, out64)
        outs[cluster] = got
    assert np.array_equal(outs[4], outs[2])


@pytest.mark.parametrize("mode", ["sm", "ce"])
def test_ag_missing_signal_times_out_then_next_call_succeeds(mode):
    # two-pair clusters (Ms = 512): one signal group of shard 1 is never set
    # (host-side injection), so the bounded wait of the CTAs that read those
    # rows runs out; the call reports TIMEOUT with the group index and the
    # next call (new epoch) gives the exact result
    inp = synth.ag_inputs(2, 512, 128, 512, "int2", seed=5)
    _, C16 = oracle.ag_gemm(inp.shards, inp.B)
    case = AGCase(inp)
    sig = 32 if mode == "sm" else 512
    g = 512 // sig + 1 if mode == "sm" else 1   # a group of shard 1 (remote for rank 0)
    _, st = case.run(rank=0, mode=mode, signal_rows=sig, test_skip_notify=1 << g,
                     timeout_ns=20_000_000, check_status=False)
    assert st["code"] == tdg.TDG_ERR_TIMEOUT and st["where"] == "ag_flag" and st["index"] == g
    got, st = case.run(rank=0, mode=mode, signal_rows=sig)
    assert st["code"] == 0 and np.array_equal(got, C16)
