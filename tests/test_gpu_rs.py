"""GPU parity of GEMM+ReduceScatter (through the C ABI) against the CPU oracle."""
import numpy as np
import pytest
import torch

import oracle
from tile_centric_comm_gb300 import synth, tdg
from gpu_util import RSCase, assert_close

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("W,M", [(4, 512), (2, 1024)])   # (2, 1024): CTA pairs
def test_integer_small_k_bit_exact_both_modes(W, M):
    # integer inputs with small K: every partial |.| <= 2*2*K <= 256 is exact in
    # bf16, and the fp32 sum of W of them is exact too
    inp = synth.rs_inputs(W, M, 64, 520, "int2", seed=5)
    _, out16 = oracle.gemm_rs(inp.As, inp.Bs)
    case = RSCase(inp)
    for mode in ("sm", "serial", "sm"):
        got, _ = case.run(mode=mode)
        assert np.array_equal(got, out16), mode


@pytest.mark.parametrize("order", [1, 0])
@pytest.mark.parametrize("W,M", [(4, 2048), (8, 4096)])
def test_rank_fastest_tile_order_gives_the_same_bits(W, M, order):
    # order 1 walks the tiles rank-fastest instead of in owner blocks; the
    # reduction still sums in rank order, so the bits do not change
    inp = synth.rs_inputs(W, M, 64, 264, "int2", seed=W + M)
    _, out16 = oracle.gemm_rs(inp.As, inp.Bs)
    case = RSCase(inp)
    for mode in ("sm", "serial"):
        got, _ = case.run(mode=mode, order=order)
        assert np.array_equal(got, out16), mode
    f = synth.rs_inputs(W, M, 200, 264, "normal", seed=W * M)
    ref = RSCase(f).run(mode="sm", order=order)[0]
    assert np.array_equal(RSCase(f).run(mode="sm", order=1 - order)[0], ref)


@pytest.mark.parametrize("cluster", [0, 1])
@pytest.mark.parametrize("b_layout", [tdg.B_KN, tdg.B_NK])
@pytest.mark.parametrize("W,M,K,N", [
    (2, 256, 200, 264),    # ragged k block and n tile
    (4, 1024, 320, 512),   # 2 m tiles per owner (one pair tile)
    (8, 1024, 128, 256),
    (2, 1024, 136, 136),   # pairs with a narrow n tile
])
def test_float_parity_small(W, M, K, N, b_layout, cluster):
    inp = synth.rs_inputs(W, M, K, N, "normal", seed=M + K)
    out64, _ = oracle.gemm_rs(inp.As, inp.Bs)
    case = RSCase(inp, b_layout=b_layout)
    for mode in ("sm", "serial"):
        got, _ = case.run(mode=mode, cluster=cluster)
        assert_close(got, out64)


def test_counters_reset_between_calls():
    inp = synth.rs_inputs(2, 256, 64, 256, "int2", seed=9)
    _, out16 = oracle.gemm_rs(inp.As, inp.Bs)
    case = RSCase(inp)
    for _ in range(3):
        got, _ = case.run(mode="sm")
        assert np.array_equal(got, out16)
    for o in range(2):
        assert int(case.symm.counters(o, 8).abs().sum()) == 0


def test_degenerate_and_invalid():
    inp = synth.rs_inputs(2, 256, 8, 16, "int2", seed=1)
    case = RSCase(inp)
    tdg.gemm_rs(case.symm, 256, 0, 16, case.a_off, case.b_off, case.stage_off, case.out_off)
    torch.cuda.synchronize()
    assert int(case.out(0).view(torch.int16).abs().sum()) == 0
    with pytest.raises(tdg.TdgError):   # M/W not a multiple of 128
        tdg.gemm_rs(case.symm, 192, 8, 16, case.a_off, case.b_off, case.stage_off, case.out_off)


@pytest.mark.slow
def test_full_size_sampled():
    inp = synth.make("rs_qwen32b_down")
    case = RSCase(inp)
    g = np.random.default_rng(1)
    M, N = inp.M, inp.N
    rows = np.concatenate([g.integers(0, M, 1000), [0, M - 1]])
    cols = np.concatenate([g.integers(0, N, 1000), [N - 1, 0]])
    ref = oracle.gemm_rs_sampled(inp.As, inp.Bs, rows, cols)
    base = None
    for mode in ("sm", "serial"):
        got, _ = case.run(mode=mode)
        flat = got.reshape(M, N)
        assert_close(flat[rows, cols], ref)
        if base is None:
            base = got
    # other schedules at the full size: the same partials summed in the same
    # rank order, so the same bits (blocks of 2 owners, no L2 hints on the
    # pushes; CTA pairs on the spare SMs; pairs-only clusters)
    for kw in (dict(owner_block=2), dict(spare=2), dict(cluster=2)):
        got, _ = case.run(mode="sm", **kw)
        assert np.array_equal(got, base), kw
    del case
    torch.cuda.empty_cache()


def _bf16_ulp(x):
    e = np.floor(np.log2(np.maximum(np.abs(x), 2.0 ** -126)))
    return 2.0 ** (e - 7)


@pytest.mark.parametrize("M", [256, 512, 1024])   # W = 2: 128-row tiles, CTA pairs, two pairs
def test_f32_partials_integer_bit_exact_where_bf16_partials_round(M):
    # K = 1024: a partial reaches |.| = 4096, beyond the integers bf16 holds
    # exactly (256), but fp32 holds every partial and the sum exactly, so the
    # fp32-partial path must give the oracle's bits in both modes
    inp = synth.rs_inputs(2, M, 1024, 264, "int2", seed=M + 3)
    _, out16 = oracle.gemm_rs(inp.As, inp.Bs)
    case = RSCase(inp, f32=True)
    for mode in ("sm", "serial"):
        got, _ = case.run(mode=mode)
        assert np.array_equal(got, out16), mode


@pytest.mark.parametrize("b_layout", [tdg.B_KN, tdg.B_NK])
def test_f32_partials_float_within_one_ulp(b_layout):
    # one rounding (the fp32 sum to bf16): every output within one bf16 ulp of
    # the exact sum plus the fp32 accumulation bound 2 (K + W) 2^-24 sum|a b|
    # (which matters only where the sum cancels), and no worse than the
    # bf16-partial path
    W, M, K, N = 4, 2048, 320, 520
    inp = synth.rs_inputs(W, M, K, N, "normal", seed=31)
    out64, _ = oracle.gemm_rs(inp.As, inp.Bs)
    absdot, _ = oracle.gemm_rs([a & 0x7FFF for a in inp.As], [b & 0x7FFF for b in inp.Bs])
    f32 = RSCase(inp, b_layout=b_layout, f32=True)
    got, _ = f32.run(mode="sm")
    got64 = (got.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    bound = _bf16_ulp(out64) + 2 * (K + W) * 2.0 ** -24 * absdot
    assert np.all(np.abs(got64 - out64) <= bound)
    assert_close(got, out64)
    bf16, _ = RSCase(inp, b_layout=b_layout).run(mode="sm")
    b64 = (bf16.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    assert np.max(np.abs(got64 - out64)) <= np.max(np.abs(b64 - out64))


@pytest.mark.parametrize("W,M,N", [(8, 8192, 2048), (2, 8192, 4096)])
@pytest.mark.parametrize("red_rows", [4, 8, 32])
def test_owed_reductions_worked_off_in_slices(red_rows, W, M, N):
    # many tiles per epilogue warp, fp32 partials: the last arriver queues its
    # reduction and works it off a few rows per tile.  With W = 2 and 128
    # quad tiles per owner, about 7 last-rank tiles come to each cluster in a
    # row, so a warp's queue fills (a fourth owed reduction finishes the
    # oldest at once) and the pass after the last tile finishes up to four.
    # Every output must match the oracle and the separate reduction launch
    # bit for bit (integer inputs: exact), and every counter ends at zero.
    K = 64
    inp = synth.rs_inputs(W, M, K, N, "int2", seed=41)
    case = RSCase(inp, f32=True)
    fused, _ = case.run(mode="sm", red_rows=red_rows)
    serial, _ = case.run(mode="serial")
    assert np.array_equal(fused, serial)
    g = np.random.default_rng(5)
    rows = np.concatenate([g.integers(0, M, 3000), [0, M - 1]])
    cols = np.concatenate([g.integers(0, N, 3000), [0, N - 1]])
    want = oracle.f64_to_bf16(oracle.gemm_rs_sampled(inp.As, inp.Bs, rows, cols))
    assert np.array_equal(fused.reshape(M, N)[rows, cols], want)
    for o in range(W):
        assert int(case.symm.counters(o, case.symm.nsig).abs().sum()) == 0


@pytest.mark.parametrize("f32", [False, True])
def test_counts_left_by_an_earlier_call_are_ignored(f32):
    # an earlier call that ended early (on a fault, say) can leave arrival
    # counts behind; emulate that on the host by writing counter words tagged
    # with the last epoch used (the one before tdg_symm_epoch, which names the
    # next call's) and counts 1..W-1: the next call must ignore them and give
    # the oracle's bits
    W = 4
    inp = synth.rs_inputs(W, 2048, 64, 520, "int2", seed=43)
    _, out16 = oracle.gemm_rs(inp.As, inp.Bs)
    case = RSCase(inp, f32=f32)
    g = np.random.default_rng(7)
    for _ in range(2):
        tag = ((case.symm.epoch() - 1) & 0x01FFFFFF) << 7
        stage = tdg.gemm_rs_stage_bytes(W, inp.M, inp.N) * (2 if f32 else 1)
        for o in range(W):
            n = case.symm.nsig
            stale = (tag | g.integers(1, W, n)).astype(np.uint32).view(np.int32)
            case.symm.counters(o, n).copy_(torch.from_numpy(stale))
            # NaN in the staging area: a reduction that started before all W
            # pushes landed would read it
            case.symm.view(o, case.stage_off, (stage // 2,), torch.int16).fill_(0x7FC1)
        got, _ = case.run(mode="sm")
        assert np.array_equal(got, out16)
