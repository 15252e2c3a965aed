"""GPU parity of the tile-centric ring AllReduce (through the C ABI) against the
oracle's element-wise sum: bit-exact on integer-valued data, within a float32
rounding bound on normal data."""
import numpy as np
import pytest
import torch

import oracle
from tile_centric_comm_gb300 import tdg
from gpu_util import align

pytestmark = pytest.mark.gpu


class RingCase:
    def __init__(self, W, count, seed, integer):
        g = np.random.default_rng(seed)
        if integer:
            self.xs = [g.integers(-1000, 1001, count).astype(np.float32) for _ in range(W)]
        else:
            self.xs = [g.standard_normal(count).astype(np.float32) for _ in range(W)]
        self.W, self.count = W, count
        self.x_off = 0
        self.recv_off = align(count * 4)
        region = align(self.recv_off + tdg.allreduce_recv_bytes(W, count) + 1024)
        self.symm = tdg.Symm(W, region, 65536)

    def run(self, check_status=True, **kw):
        for r in range(self.W):
            self.symm.view(r, self.x_off, (self.count,), torch.float32).copy_(torch.from_numpy(self.xs[r]))
        tdg.allreduce(self.symm, self.count, self.x_off, self.recv_off, **kw)
        torch.cuda.synchronize()
        st = self.symm.status()
        if check_status:
            assert st["code"] == 0, st
        return [self.symm.view(r, self.x_off, (self.count,), torch.float32).cpu().numpy()
                for r in range(self.W)], st


@pytest.mark.parametrize("W,count,tile,G", [
    (2, 1024, 0, 0), (4, 4096, 128, 3), (8, 8192 * 8, 1000 - 1000 % 4, 5), (3, 12 * 1000, 200, 0),
    (8, 1 << 22, 0, 0)])
def test_integer_bit_exact(W, count, tile, G):
    case = RingCase(W, count, seed=W + count, integer=True)
    want = oracle.allreduce(case.xs)
    outs, _ = case.run(tile_elems=tile, ctas_per_rank=G)
    for r in range(W):
        assert np.array_equal(outs[r].astype(np.float64), want), r


@pytest.mark.parametrize("W,count", [(8, 1 << 20), (5, 5 * 4 * 777)])
def test_float_within_rounding_bound(W, count):
    case = RingCase(W, count, seed=7, integer=False)
    want = oracle.allreduce(case.xs)
    outs, _ = case.run()
    # W-1 float32 additions: |error| <= (W-1) * 2^-24 * sum_r |x_r| (plus slack)
    bound = (W - 1) * 2.0 ** -24 * np.sum(np.abs(np.stack(case.xs)).astype(np.float64), axis=0) + 1e-30
    for r in range(W):
        assert np.all(np.abs(outs[r] - want) <= bound * 1.01), r
        assert np.array_equal(outs[r], outs[0])     # every rank holds the same bits


def test_degenerate_and_invalid():
    case = RingCase(4, 64, seed=1, integer=True)
    tdg.allreduce(case.symm, 0, case.x_off, case.recv_off)        # no-op
    with pytest.raises(tdg.TdgError):
        tdg.allreduce(case.symm, 66, case.x_off, case.recv_off)   # count % (4W) != 0
    one = tdg.Symm(1, 4096, 64)
    tdg.allreduce(one, 16, 0, 2048)                                # single rank: no-op
    torch.cuda.synchronize()


def test_missing_signal_times_out_then_next_call_succeeds():
    # host-side injection: rank 0's signal for (step 2, tile 1) is never
    # notified; rank 0's bounded wait must run out and report it, the launch
    # must still end, and the next call (a new epoch) must give the sum
    W, count, tile = 4, 4 * 4096, 1024
    tiles = (count // W) // tile
    case = RingCase(W, count, seed=3, integer=True)
    want = oracle.allreduce(case.xs)
    sig = 2 * tiles + 1
    _, st = case.run(check_status=False, tile_elems=tile, timeout_ns=20_000_000, test_skip_signal=sig + 1)
    assert st["code"] == tdg.TDG_ERR_TIMEOUT and st["where"] == "ring" and st["index"] == sig
    outs, st = case.run(tile_elems=tile)
    for r in range(W):
        assert np.array_equal(outs[r].astype(np.float64), want), r
