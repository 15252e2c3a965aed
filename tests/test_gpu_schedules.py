"""Schedules of the same computation, chosen per call, against the CPU oracle:
push-mode AllGather (the senders order the transfers), the GEMM's ring stage
count and cluster shape, and the producers' copy-ring shape.  Integer inputs,
so every schedule must give the oracle's bits and the bit-exact gathered
buffer; out-of-range schedule values are rejected before any launch."""
import numpy as np
import pytest
import torch

import oracle
from tile_centric_comm_gb300 import synth, tdg
from gpu_util import AGCase, RSCase, to_bits
from test_gpu_ag_all import AGAllCase

pytestmark = pytest.mark.gpu


def _gathered_ok(case, rank):
    assert np.array_equal(to_bits(case.gathered(rank)), np.concatenate(case.inp.shards)), rank


@pytest.mark.parametrize("source_order", [0, 1])
@pytest.mark.parametrize("W,Ms,K,N", [
    (4, 512, 128, 264),     # two-pair clusters, the local shard read in place
    (3, 96, 136, 136),      # shards smaller than a tile: the local shard copied and waited on
    (8, 256, 64, 520),      # CTA pairs, one shard per tile
])
def test_push_mode_bit_exact_every_mode(W, Ms, K, N, source_order):
    inp = synth.ag_inputs(W, Ms, K, N, "int2", seed=W * 31 + Ms)
    _, C16 = oracle.ag_gemm(inp.shards, inp.B)
    case = AGCase(inp, ll=True)
    for mode in ("sm", "ce", "ll", "serial"):
        for rank in (0, W - 1):
            got, _ = case.run(rank=rank, mode=mode, push=True, source_order=source_order,
                              ll_off=case.ll_off, signal_rows=32 if Ms % 32 == 0 else 0)
            assert np.array_equal(got, C16), (mode, rank)
            _gathered_ok(case, rank)


def test_push_mode_without_swizzle_and_with_producer_items():
    inp = synth.ag_inputs(4, 1536, 128, 520, "int2", seed=77)
    _, C16 = oracle.ag_gemm(inp.shards, inp.B)
    case = AGCase(inp)
    for swizzle in (True, False):
        for items in (0, 3):
            got, _ = case.run(rank=2, mode="sm", push=True, swizzle=swizzle, producers=16,
                              producer_items=items)
            assert np.array_equal(got, C16), (swizzle, items)
            _gathered_ok(case, 2)


@pytest.mark.parametrize("W,Ms,K,N", [(4, 512, 128, 264), (3, 384, 64, 256), (2, 96, 136, 520)])
def test_all_ranks_push_mode_bit_exact(W, Ms, K, N):
    # (4, 512): every shard is whole tiles, so the GEMM follows the push steps;
    # (3, 384) and (2, 96): it keeps the rank-by-rank order while the copies go
    # step by step
    inp = synth.ag_all_inputs(W, Ms, K, N, "int2", seed=W * 7 + Ms)
    case = AGAllCase(inp)
    want = [oracle.ag_gemm(inp.shards, inp.Bs[r])[1] for r in range(W)]
    for mode in ("ce", "serial"):
        for rep in range(2):
            got, _ = case.run(mode=mode, push=True)
            for r in range(W):
                assert np.array_equal(got[r], want[r]), (mode, rep, r)
                assert np.array_equal(to_bits(case.gathered(r)), np.concatenate(inp.shards)), (mode, r)


@pytest.mark.parametrize("cluster,stages", [(4, 2), (4, 3), (4, 5), (2, 2), (2, 4), (1, 2), (1, 3)])
def test_ring_stages_bit_exact(cluster, stages):
    inp = synth.ag_inputs(2, 1024, 520, 264, "int2", seed=cluster * 10 + stages)
    _, C16 = oracle.ag_gemm(inp.shards, inp.B)
    case = AGCase(inp)
    for mode in ("ce", "sm"):
        got, _ = case.run(rank=1, mode=mode, cluster=cluster, stages=stages)
        assert np.array_equal(got, C16), mode
    rs = synth.rs_inputs(2, 2048, 64, 520, "int2", seed=stages)
    _, out16 = oracle.gemm_rs(rs.As, rs.Bs)
    got, _ = RSCase(rs).run(mode="sm", cluster=cluster, stages=stages)
    assert np.array_equal(got, out16)
    aa = synth.ag_all_inputs(2, 512, 64, 264, "int2", seed=stages + 1)
    got, _ = AGAllCase(aa).run(mode="ce", cluster=cluster, stages=stages)
    for r in range(2):
        assert np.array_equal(got[r], oracle.ag_gemm(aa.shards, aa.Bs[r])[1]), r


@pytest.mark.parametrize("kb,cluster", [(1, 4), (5, 4), (6, 4), (7, 4), (13, 4), (7, 2), (5, 1), (13, 1)])
def test_unrolled_ring_rounds_bit_exact(kb, cluster):
    # With every ring slot in use and every tile full width, the MMA issuer
    # runs whole rounds of its ring unrolled.  k-block counts below, at and
    # past the ring's depth (6 slots for pairs and clusters, 4 for one CTA),
    # with several tiles per cluster so that tiles start at every slot: the
    # integer AG-GEMM equals the oracle bit for bit on sampled entries, and a
    # ring one slot shorter (the per-stage loop) gives the same bits
    # everywhere; the GEMM-RS likewise against its one-slot-shorter ring.
    K = 64 * kb
    depth = 4 if cluster == 1 else 6
    inp = synth.ag_inputs(8, 2048, K, 2048, "int2", seed=100 + kb)
    case = AGCase(inp)
    g = np.random.default_rng(kb)
    rows = np.concatenate([g.integers(0, case.M, 2000), [0, case.M - 1]])
    cols = np.concatenate([g.integers(0, inp.N, 2000), [inp.N - 1, 0]])
    want = oracle.f64_to_bf16(oracle.ag_gemm_sampled(inp.shards, inp.B, rows, cols))
    for mode in ("serial", "ce"):
        got, _ = case.run(rank=0, mode=mode, cluster=cluster)
        assert np.array_equal(got[rows, cols], want), mode
        short, _ = case.run(rank=0, mode=mode, cluster=cluster, stages=depth - 1)
        assert np.array_equal(got, short), mode
    del case
    rs = synth.rs_inputs(8, 8192, K, 1024, "int2", seed=200 + kb)
    rcase = RSCase(rs)
    got, _ = rcase.run(mode="sm", cluster=cluster)
    short, _ = rcase.run(mode="sm", cluster=cluster, stages=depth - 1)
    assert np.array_equal(got, short)
    if kb == 1:   # |partial| <= 4K = 256: every bf16 partial is exact
        M, N = rs.M, rs.N
        r_s = np.concatenate([g.integers(0, M, 2000), [0, M - 1]])
        c_s = np.concatenate([g.integers(0, N, 2000), [N - 1, 0]])
        ref = oracle.f64_to_bf16(oracle.gemm_rs_sampled(rs.As, rs.Bs, r_s, c_s))
        assert np.array_equal(got.reshape(M, N)[r_s, c_s], ref)
    del rcase
    torch.cuda.empty_cache()


@pytest.mark.parametrize("W,Mo,N,spare", [(2, 512, 520, 1), (2, 1024, 264, 3), (4, 512, 520, 5),
                                           (8, 512, 264, 63), (8, 1024, 8, 2)])
def test_spare_sm_pairs_bit_exact(W, Mo, N, spare):
    # CTA pairs on the SMs the 4-CTA clusters leave idle take the last `spare`
    # (owner block, rank, owner) tile groups in a second launch: the same
    # partials and reductions, so the oracle's bits in both modes and with
    # fp32 partials, and bits equal to the clusters alone on float data
    inp = synth.rs_inputs(W, W * Mo, 64, N, "int2", seed=W * 1000 + spare)
    _, out16 = oracle.gemm_rs(inp.As, inp.Bs)
    for f32 in (False, True):
        case = RSCase(inp, f32=f32)
        for mode in ("sm", "serial"):
            got, _ = case.run(mode=mode, cluster=4, spare=spare)
            assert np.array_equal(got, out16), (f32, mode)
    fl = synth.rs_inputs(W, W * Mo, 520, N, "normal", seed=W + spare)
    case = RSCase(fl)
    base, _ = case.run(mode="sm", cluster=4)
    for mode in ("sm", "serial"):
        got, _ = case.run(mode=mode, cluster=4, spare=spare)
        assert np.array_equal(got, base), mode


@pytest.mark.parametrize("W", [3, 5, 6, 8])
def test_rs_default_owner_blocks_bit_exact(W):
    # the default owner block: all W owners with bf16 partials, the largest
    # divisor of W up to 4 with fp32 partials (3, 1, 3 and 4 here); also the
    # order that keeps the pushes' L2 hint off (rank fastest)
    inp = synth.rs_inputs(W, W * 256, 64, 264, "int2", seed=W * 77)
    _, out16 = oracle.gemm_rs(inp.As, inp.Bs)
    for f32 in (False, True):
        case = RSCase(inp, f32=f32)
        for mode in ("sm", "serial"):
            for order in (0, 1):
                got, _ = case.run(mode=mode, order=order)
                assert np.array_equal(got, out16), (f32, mode, order)


@pytest.mark.parametrize("warps,chunk", [(1, 4096), (1, 65536), (2, 16384), (3, 8192), (4, 16384), (4, 4096)])
def test_producer_ring_shapes_bit_exact(warps, chunk):
    # unit sizes that are not a multiple of the chunk (K = 520: 1040-byte rows),
    # units of one chunk or less (signal_rows 8), and the serial copy launch
    inp = synth.ag_inputs(4, 512, 520, 264, "int2", seed=warps * 100 + chunk // 1024)
    _, C16 = oracle.ag_gemm(inp.shards, inp.B)
    case = AGCase(inp)
    for mode, sig in (("sm", 0), ("sm", 8), ("serial", 0)):
        for order in (0, 1):
            got, _ = case.run(rank=3, mode=mode, signal_rows=sig, source_order=order,
                              producer_warps=warps, producer_chunk=chunk, producers=8)
            assert np.array_equal(got, C16), (mode, sig, order)
            _gathered_ok(case, 3)


def test_out_of_range_schedules_are_rejected():
    inp = synth.ag_inputs(2, 256, 64, 264, "int2", seed=3)
    case = AGCase(inp)
    bad = [dict(cluster=4),                # Ms = 256 is not a whole number of 512-row tiles
           dict(cluster=3), dict(stages=1), dict(stages=7), dict(cluster=1, stages=5),
           dict(producer_items=-2), dict(producer_warps=5), dict(producer_chunk=3000),
           dict(producer_chunk=2048), dict(producer_chunk=131072),
           dict(producer_warps=4, producer_chunk=65536)]
    for kw in bad:
        with pytest.raises(tdg.TdgError) as ei:
            case.run(rank=0, mode="sm", **kw)
        assert ei.value.code == tdg.TDG_ERR_INVALID, kw
    # flags other than 0 / 1, through the struct (the binding passes booleans)
    import ctypes
    for field in ("push", "split_tail"):
        a = tdg.AgGemmArgs(world=2, rank=0, Ms=256, K=64, N=264, a_off=case.a_off, g_off=case.g_off,
                           B=case.B.data_ptr(), C=case.C.data_ptr(), mode=tdg.MODE_SM, swizzle=1)
        setattr(a, field, 2)
        rc = tdg.lib().tdg_ag_gemm(case.symm.h, ctypes.byref(a), tdg._stream(None), None)
        assert rc == tdg.TDG_ERR_INVALID, field
    rs = RSCase(synth.rs_inputs(2, 512, 64, 264, "int2", seed=4))   # 256 rows per owner
    for kw in (dict(cluster=4), dict(order=2), dict(red_rows=3), dict(red_rows=64), dict(stages=9),
               dict(spare=-1), dict(spare=4)):
        with pytest.raises(tdg.TdgError) as ei:
            rs.run(mode="sm", **kw)
        assert ei.value.code == tdg.TDG_ERR_INVALID, kw
    torch.cuda.synchronize()
    assert case.symm.status()["code"] == 0 and rs.symm.status()["code"] == 0
    # nothing was launched: the next calls are exact
    _, C16 = oracle.ag_gemm(inp.shards, inp.B)
    assert np.array_equal(case.run(rank=0, mode="sm")[0], C16)


@pytest.mark.parametrize("push", [False, True])
def test_allgather_alone_when_n_is_zero(push):
    # N == 0: no GEMM (B and C may be None); the gathered buffer is the exact
    # concatenation, and in the signalled modes every group's flag holds the
    # call's epoch; SERIAL's copy launch may use a few CTAs only
    inp = synth.ag_inputs(4, 512, 264, 8, "int2", seed=5)
    case = AGCase(inp, ll=True)
    M, K = case.M, inp.K
    for mode, kw in (("sm", dict(producers=4)), ("sm", {}), ("ce", {}), ("ll", dict(ll_off=case.ll_off)),
                     ("serial", dict(producers=3)), ("serial", {})):
        for rank in (0, 3):
            case.gathered(rank).view(torch.int16).fill_(0x7FC1)
            case.symm.flags(rank, M // 32).zero_()
            epoch = case.symm.epoch()
            side = torch.cuda.Stream() if mode == "ce" else None
            tdg.ag_gemm(case.symm, rank, inp.Ms, K, 0, case.a_off, case.g_off, None, None, mode=mode,
                        signal_rows=32, side_stream=side, push=push, **kw)
            torch.cuda.synchronize()
            assert case.symm.status()["code"] == 0, (mode, rank)
            _gathered_ok(case, rank)
            fl = case.symm.flags(rank, M // 32).cpu().numpy()
            if mode != "serial":
                assert np.all(fl == epoch), (mode, rank)
