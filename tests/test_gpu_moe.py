"""GPU parity of MoE routing / dispatch / combine (through the C ABI) against the
CPU oracle: integer outputs bit-exact, combine within the float tolerance."""
import numpy as np
import pytest
import torch

import oracle
from tile_centric_comm_gb300 import synth, tdg
from gpu_util import POISON, align, assert_close, to_bits, to_dev_bf16

pytestmark = pytest.mark.gpu


class MoECase:
    def __init__(self, inp, device="cuda"):
        self.inp = inp
        W, T, H, k, E = inp.W, inp.T, inp.H, inp.k, inp.E
        self.x_off = 0
        self.topk_off = align(T * H * 2)
        self.gate_off = align(self.topk_off + T * k * 4)
        self.out_off = align(self.gate_off + T * k * 4)
        region = align(self.out_off + T * H * 2 + 1024)
        self.symm = tdg.Symm(W, region, 1024, device=device)
        for s in range(W):
            self.symm.view(s, self.x_off, (T, H), torch.bfloat16).copy_(to_dev_bf16(inp.x[s]))
            self.symm.view(s, self.topk_off, (T, k), torch.int32).copy_(
                torch.from_numpy(np.ascontiguousarray(inp.topk[s])))
            self.symm.view(s, self.gate_off, (T, k), torch.float32).copy_(
                torch.from_numpy(np.ascontiguousarray(inp.gate[s])))
        total = W * T * k
        d = device
        self.recv = torch.empty((total, H), dtype=torch.bfloat16, device=d)
        self.counts = torch.empty((W, E), dtype=torch.int64, device=d)
        self.base = torch.empty(E + 1, dtype=torch.int64, device=d)
        self.slot = torch.empty((W, T, k), dtype=torch.int64, device=d)
        self.row_src = torch.empty(total, dtype=torch.int32, device=d)
        self.row_tok = torch.empty(total, dtype=torch.int32, device=d)
        self.row_k = torch.empty(total, dtype=torch.int32, device=d)
        self.ws = torch.empty(tdg.moe_workspace_bytes(W, T, E), dtype=torch.uint8, device=d)

    def out(self, s):
        return self.symm.view(s, self.out_off, (self.inp.T, self.inp.H), torch.bfloat16)

    def run(self, phases=tdg.MOE_ALL, y=None, check_status=True):
        inp = self.inp
        self.recv.view(torch.int16).fill_(POISON)
        for s in range(inp.W):
            self.out(s).view(torch.int16).fill_(POISON)
        tdg.moe_dispatch_combine(self.symm, inp.T, inp.H, inp.E, inp.k, self.x_off, self.topk_off,
                                 self.gate_off, self.out_off, self.recv, self.counts, self.base,
                                 self.slot, self.ws, y=y, row_src=self.row_src,
                                 row_tok=self.row_tok, row_k=self.row_k, phases=phases)
        torch.cuda.synchronize()
        st = self.symm.status()
        if check_status:
            assert st["code"] == 0, st
        return st


def _check_route(case, r):
    assert np.array_equal(case.counts.cpu().numpy(), r["counts"])
    assert np.array_equal(case.base.cpu().numpy(), r["base"])
    assert np.array_equal(case.slot.cpu().numpy(), r["slot"])
    assert np.array_equal(case.row_src.cpu().numpy(), r["row_src"])
    assert np.array_equal(case.row_tok.cpu().numpy(), r["row_tok"])
    assert np.array_equal(case.row_k.cpu().numpy(), r["row_k"])


@pytest.mark.parametrize("W,T,H,E,k", [(2, 100, 72, 8, 3), (4, 257, 512, 64, 8), (8, 64, 7168, 256, 8)])
def test_route_dispatch_combine_parity(W, T, H, E, k):
    inp = synth.moe_inputs(W, T, H, E, k, seed=T + E)
    r = oracle.moe_route(inp.topk, E)
    case = MoECase(inp)
    case.run()
    _check_route(case, r)
    recv = oracle.moe_dispatch(inp.x, r["slot"], W * T * k)
    assert np.array_equal(to_bits(case.recv), recv)
    _, out64 = oracle.moe_combine(recv, r["slot"], inp.gate)
    got = np.stack([to_bits(case.out(s)) for s in range(W)])
    assert_close(got, out64)


def test_top1_unit_weight_round_trip_is_identity():
    inp = synth.moe_inputs(4, 128, 256, 16, 8, seed=11, top1_unit=True)
    case = MoECase(inp)
    case.run()
    got = np.stack([to_bits(case.out(s)) for s in range(4)])
    assert np.array_equal(got, inp.x)


def test_unit_weights_integer_x_gives_k_times_x_exactly():
    inp = synth.moe_inputs(2, 64, 128, 16, 8, seed=4, x_dist="int2")
    inp.gate[:] = 1.0
    case = MoECase(inp)
    case.run()
    got = np.stack([to_bits(case.out(s)) for s in range(2)])
    want = oracle.f64_to_bf16(8.0 * oracle.bf16_to_f64(inp.x))
    assert np.array_equal(got, want)


def test_phases_separately_and_external_y():
    inp = synth.moe_inputs(2, 96, 64, 8, 2, seed=2)
    r = oracle.moe_route(inp.topk, inp.E)
    case = MoECase(inp)
    case.run(phases=tdg.MOE_ROUTE)
    _check_route(case, r)
    case.run(phases=tdg.MOE_ROUTE | tdg.MOE_DISPATCH)
    y = torch.flip(case.recv, dims=[1]).contiguous()    # any expert output in recv layout
    case.run(phases=tdg.MOE_COMBINE, y=y)
    _, out64 = oracle.moe_combine(to_bits(y), r["slot"], inp.gate)
    got = np.stack([to_bits(case.out(s)) for s in range(2)])
    assert_close(got, out64)


def test_bad_expert_id_reported():
    inp = synth.moe_inputs(2, 64, 32, 8, 2, seed=3)
    inp.topk[1, 5, 1] = 8     # out of range
    case = MoECase(inp)
    st = case.run(phases=tdg.MOE_ROUTE, check_status=False)
    assert st["code"] == tdg.TDG_ERR_DEVICE and st["where"] == "moe_expert"
    assert st["index"] == (1 * 64 + 5) * 2 + 1
    assert int(case.slot[1, 5, 1]) == -1


@pytest.mark.slow
def test_full_size():
    inp = synth.make("moe_8x4096_h7168_e256_top8")
    r = oracle.moe_route(inp.topk, inp.E)
    case = MoECase(inp)
    case.run()
    _check_route(case, r)
    # dispatch: every receive row equals its source row (bit-exact), checked on
    # a sample of rows plus the per-rank boundaries
    g = np.random.default_rng(0)
    rows = np.unique(np.concatenate([g.integers(0, inp.W * inp.T * 8, 4000),
                                     r["base"][::32][:-1], r["base"][1:] - 1]))
    got = to_bits(case.recv[torch.from_numpy(rows).cuda()])
    assert np.array_equal(got, inp.x[r["row_src"][rows], r["row_tok"][rows]])
    # combine on sampled tokens: the oracle's combine over just those rows
    toks = g.integers(0, inp.W * inp.T, 300)
    src, t = toks // inp.T, toks % inp.T
    sub_slot = r["slot"][src, t]                               # (n, k)
    y_sub = to_bits(case.recv[torch.from_numpy(sub_slot.reshape(-1)).cuda()])
    n = len(toks)
    _, ref = oracle.moe_combine(y_sub, np.arange(n * 8).reshape(1, n, 8),
                                inp.gate[src, t].reshape(1, n, 8))
    out = np.stack([to_bits(case.out(int(s))[int(tt)]) for s, tt in zip(src, t)])
    assert_close(out, ref[0])
