"""GPU parity of the AllGather+GEMM of every rank in one call (through the C
ABI) against the CPU oracle, one rank's product at a time."""
import numpy as np
import pytest
import torch

import oracle
from tile_centric_comm_gb300 import synth, tdg
from gpu_util import AGCase, POISON, align, assert_close, bf16_f64, to_bits, to_dev_bf16

pytestmark = pytest.mark.gpu


class AGAllCase:
    def __init__(self, inp, b_layout=tdg.B_KN, c_f32=False):
        self.inp = inp
        self.c_f32 = c_f32
        W, Ms, K, N = inp.W, inp.Ms, inp.K, inp.N
        self.M = M = W * Ms
        self.a_off = 0
        self.g_off = align(Ms * K * 2)
        self.b_off = align(self.g_off + M * K * 2)
        self.c_off = align(self.b_off + K * N * 2)
        self.symm = tdg.Symm(W, align(self.c_off + M * N * (4 if c_f32 else 2) + 1024), max(1024, M))
        self.b_layout = b_layout
        for r in range(W):
            self.symm.view(r, self.a_off, (Ms, K), torch.bfloat16).copy_(to_dev_bf16(inp.shards[r]))
            b = inp.Bs[r] if b_layout == tdg.B_KN else np.ascontiguousarray(inp.Bs[r].T)
            self.symm.view(r, self.b_off, b.shape, torch.bfloat16).copy_(to_dev_bf16(b))

    def C(self, r):
        return self.symm.view(r, self.c_off, (self.M, self.inp.N),
                              torch.float32 if self.c_f32 else torch.bfloat16)

    def gathered(self, r):
        return self.symm.view(r, self.g_off, (self.M, self.inp.K), torch.bfloat16)

    def run(self, mode="ce", check_status=True, **kw):
        inp = self.inp
        for r in range(inp.W):
            if self.c_f32:
                self.C(r).view(torch.int32).fill_(0x7FC00001)     # a NaN float32 pattern
            else:
                self.C(r).view(torch.int16).fill_(POISON)
            self.gathered(r).view(torch.int16).fill_(POISON)
        side = torch.cuda.Stream() if mode == "ce" else None
        tdg.ag_gemm_all_ranks(self.symm, inp.Ms, inp.K, inp.N, self.a_off, self.g_off, self.b_off,
                              self.c_off, mode=mode, b_layout=self.b_layout, side_stream=side,
                              c_f32=self.c_f32, **kw)
        torch.cuda.synchronize()
        st = self.symm.status()
        if check_status:
            assert st["code"] == 0, st
        if self.c_f32:
            return [self.C(r).cpu().numpy() for r in range(inp.W)], st
        return [to_bits(self.C(r)) for r in range(inp.W)], st


@pytest.mark.parametrize("b_layout", [tdg.B_KN, tdg.B_NK])
@pytest.mark.parametrize("W,Ms,K,N", [
    (2, 512, 128, 264),    # two-pair clusters, own shard read in place, ragged n tile
    (4, 256, 200, 136),    # CTA pairs, ragged k block
    (3, 384, 64, 256),     # 384 rows: not a whole number of 256-row tiles, own shard copied and waited on
    (3, 96, 136, 520),     # shards smaller than a tile
])
def test_integer_bit_exact_every_rank(W, Ms, K, N, b_layout):
    inp = synth.ag_all_inputs(W, Ms, K, N, "int2", seed=W * 100 + Ms)
    case = AGAllCase(inp, b_layout=b_layout)
    want = [oracle.ag_gemm(inp.shards, inp.Bs[r])[1] for r in range(W)]
    for mode in ("ce", "serial"):
        got, _ = case.run(mode=mode)
        for r in range(W):
            assert np.array_equal(got[r], want[r]), (mode, r)
            assert np.array_equal(to_bits(case.gathered(r)), np.concatenate(inp.shards)), (mode, r)


def test_float_parity_and_same_bits_as_single_rank_calls():
    W, Ms, K, N = 4, 512, 320, 264
    inp = synth.ag_all_inputs(W, Ms, K, N, "normal", seed=5)
    case = AGAllCase(inp)
    got, _ = case.run(mode="ce")
    for r in range(W):
        C64, _ = oracle.ag_gemm(inp.shards, inp.Bs[r])
        assert_close(got[r], C64)
        # the single-rank call of rank r with B_r: same kernel arithmetic, same bits
        one = AGCase(synth.AGInputs(inp.shards, inp.Bs[r], W, Ms, K, N))
        single, _ = one.run(rank=r, mode="ce")
        assert np.array_equal(got[r], single), r


def test_missing_signal_times_out_then_next_call_succeeds():
    # host-side injection: rank 0's flag for its group 1 (shard 1, remote) is
    # never written; the bounded wait runs out and reports it; the next call
    # (a new epoch) succeeds
    W, Ms, K, N = 2, 512, 64, 256
    inp = synth.ag_all_inputs(W, Ms, K, N, "int2", seed=9)
    case = AGAllCase(inp)
    _, st = case.run(mode="ce", check_status=False, test_skip_notify=1 << 1, timeout_ns=20_000_000)
    assert st["code"] == tdg.TDG_ERR_TIMEOUT and st["where"] == "ag_flag" and st["index"] == 1
    got, _ = case.run(mode="ce")
    for r in range(W):
        assert np.array_equal(got[r], oracle.ag_gemm(inp.shards, inp.Bs[r])[1]), r


def test_degenerate_shapes():
    inp = synth.ag_all_inputs(2, 128, 8, 16, "int2", seed=2)
    case = AGAllCase(inp)
    tdg.ag_gemm_all_ranks(case.symm, 128, 0, 16, case.a_off, case.g_off, case.b_off, case.c_off,
                          mode="serial")                         # K == 0: C_r = 0
    torch.cuda.synchronize()
    for r in range(2):
        assert int(case.C(r).view(torch.int16).abs().sum()) == 0
    tdg.ag_gemm_all_ranks(case.symm, 0, 8, 16, case.a_off, case.g_off, case.b_off, case.c_off,
                          mode="serial")                         # M == 0: no-op
    torch.cuda.synchronize()
    assert case.symm.status()["code"] == 0


@pytest.mark.parametrize("W,Ms,N", [(2, 512, 264), (4, 256, 136)])   # two-pair clusters; pairs
def test_f32_output_exact_where_bf16_rounds(W, Ms, N):
    # integers in [-2, 2] and K = 1032: every C_r value (up to 4128) is exact in
    # the fp32 accumulator but not in bf16
    inp = synth.ag_all_inputs(W, Ms, 1032, N, "int2", seed=W + N)
    case = AGAllCase(inp, c_f32=True)
    want = [oracle.ag_gemm(inp.shards, inp.Bs[r])[0] for r in range(W)]
    assert any(not np.array_equal(bf16_f64(oracle.ag_gemm(inp.shards, inp.Bs[r])[1]), want[r])
               for r in range(W))
    for mode in ("ce", "serial"):
        got, _ = case.run(mode=mode)
        for r in range(W):
            assert got[r].dtype == np.float32
            assert np.array_equal(got[r].astype(np.float64), want[r]), (mode, r)
