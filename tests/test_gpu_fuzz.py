"""Seeded random shapes through the C ABI, bit-exact against the oracle on
integer inputs: W from 1 to 8, shards and owners that select every GEMM shape
(one CTA, CTA pairs, two-pair clusters), ragged K and N tails, both B layouts,
every mode."""
import numpy as np
import pytest

import oracle
from tile_centric_comm_gb300 import synth, tdg
from gpu_util import AGCase, RSCase, to_bits

pytestmark = pytest.mark.gpu


def _ag_cases(n=16, seed=2024):
    g = np.random.default_rng(seed)
    out = []
    for i in range(n):
        W = int(g.choice([1, 2, 3, 4, 8]))
        Ms = int(g.choice([64, 128, 192, 256, 512, 1024]))
        if W * Ms > 4096:
            Ms = 512
        K = int(g.choice([8, 64, 136, 256]))
        N = int(g.choice([8, 72, 264, 520, 776]))
        lay = int(g.integers(0, 2))
        out.append((W, Ms, K, N, lay, 1000 + i))
    return out


def _ag_all_cases(n=8, seed=2028):
    g = np.random.default_rng(seed)
    out = []
    for i in range(n):
        W = int(g.choice([1, 2, 3, 4, 8]))
        Ms = int(g.choice([64, 128, 192, 256, 512]))
        while W * Ms > 2048:
            Ms //= 2
        K = int(g.choice([8, 64, 136, 256]))
        N = int(g.choice([8, 72, 264, 520]))
        lay = int(g.integers(0, 2))
        out.append((W, Ms, K, N, lay, 4000 + i))
    return out


@pytest.mark.parametrize("W,Ms,K,N,lay,seed", _ag_all_cases())
def test_ag_all_ranks_random_shapes_bit_exact(W, Ms, K, N, lay, seed):
    from test_gpu_ag_all import AGAllCase
    inp = synth.ag_all_inputs(W, Ms, K, N, "int2", seed=seed)
    case = AGAllCase(inp, b_layout=tdg.B_KN if lay == 0 else tdg.B_NK)
    want = [oracle.ag_gemm(inp.shards, inp.Bs[r])[1] for r in range(W)]
    for mode in ("ce", "serial"):
        got, _ = case.run(mode=mode)
        for r in range(W):
            assert np.array_equal(got[r], want[r]), (mode, r)
            assert np.array_equal(to_bits(case.gathered(r)), np.concatenate(inp.shards)), (mode, r)


def _rs_cases(n=12, seed=2025):
    g = np.random.default_rng(seed)
    out = []
    for i in range(n):
        W = int(g.choice([1, 2, 4, 8]))
        Mo = int(g.choice([128, 256, 512, 1024]))
        if W * Mo > 4096:
            Mo = 512
        K = int(g.choice([8, 32, 64]))   # |partial| <= 4K <= 256: exact in bf16
        N = int(g.choice([8, 264, 520, 1032]))
        lay = int(g.integers(0, 2))
        out.append((W, W * Mo, K, N, lay, 2000 + i))
    return out


@pytest.mark.parametrize("W,Ms,K,N,lay,seed", _ag_cases())
def test_ag_sm_mode_producers_take_items_random_shapes(W, Ms, K, N, lay, seed):
    # producer clusters take the last 3 GEMM items once their copies are done
    # (all of them when there are fewer)
    inp = synth.ag_inputs(W, Ms, K, N, "int2", seed=seed)
    _, C16 = oracle.ag_gemm(inp.shards, inp.B)
    case = AGCase(inp, b_layout=tdg.B_KN if lay == 0 else tdg.B_NK)
    for producers in (4, 16):
        got, _ = case.run(rank=seed % W, mode="sm", producers=producers, producer_items=3)
        assert np.array_equal(got, C16), producers
        assert np.array_equal(to_bits(case.gathered(seed % W)), np.concatenate(inp.shards)), producers


@pytest.mark.parametrize("W,Ms,K,N,lay,seed", _ag_cases())
def test_ag_random_shapes_bit_exact(W, Ms, K, N, lay, seed):
    inp = synth.ag_inputs(W, Ms, K, N, "int2", seed=seed)
    _, C16 = oracle.ag_gemm(inp.shards, inp.B)
    b_layout = tdg.B_KN if lay == 0 else tdg.B_NK
    case = AGCase(inp, b_layout=b_layout, ll=(W * Ms * K <= 1 << 20))
    rank = seed % W
    modes = ["sm", "ce", "serial"] + (["ll"] if W * Ms * K <= 1 << 20 else [])
    for mode in modes:
        kw = {"ll_off": case.ll_off} if mode == "ll" else {}
        got, _ = case.run(rank=rank, mode=mode, **kw)
        assert np.array_equal(got, C16), (mode, rank)
        assert np.array_equal(to_bits(case.gathered(rank)), np.concatenate(inp.shards)), (mode, "gathered")


@pytest.mark.parametrize("W,M,K,N,lay,seed", _rs_cases())
def test_rs_random_shapes_bit_exact(W, M, K, N, lay, seed):
    inp = synth.rs_inputs(W, M, K, N, "int2", seed=seed)
    _, out16 = oracle.gemm_rs(inp.As, inp.Bs)
    b_layout = tdg.B_KN if lay == 0 else tdg.B_NK
    case = RSCase(inp, b_layout=b_layout)
    for mode in ("sm", "serial", "sm"):
        got, _ = case.run(mode=mode)
        assert np.array_equal(got, out16), mode


def _rs_f32_cases(n=8, seed=2027):
    # fp32 partials hold integer partials up to 2^24 exactly, so K can reach
    # the thousands (ragged k blocks included) and the result stays bit-exact
    g = np.random.default_rng(seed)
    out = []
    for i in range(n):
        W = int(g.choice([1, 2, 4]))
        Mo = int(g.choice([128, 256, 512]))
        K = int(g.choice([200, 1032, 2056]))
        N = int(g.choice([136, 264, 520]))
        while W * W * Mo * K * N > 2_000_000_000 and Mo > 128:
            Mo //= 2
        lay = int(g.integers(0, 2))
        out.append((W, W * Mo, K, N, lay, 3000 + i))
    return out


@pytest.mark.parametrize("W,M,K,N,lay,seed", _rs_f32_cases())
def test_rs_f32_partials_random_shapes_bit_exact(W, M, K, N, lay, seed):
    inp = synth.rs_inputs(W, M, K, N, "int2", seed=seed)
    _, out16 = oracle.gemm_rs(inp.As, inp.Bs)
    b_layout = tdg.B_KN if lay == 0 else tdg.B_NK
    case = RSCase(inp, b_layout=b_layout, f32=True)
    for mode in ("sm", "serial"):
        got, _ = case.run(mode=mode)
        assert np.array_equal(got, out16), mode



def _moe_cases(n=12, seed=2026):
    g = np.random.default_rng(seed)
    out = []
    for i in range(n):
        W = int(g.choice([1, 2, 4, 8]))
        E = W * int(g.choice([1, 2, 4, 16, 32]))
        k = int(min(E, g.choice([1, 2, 3, 8])))
        T = int(g.choice([1, 5, 63, 64, 65, 200]))
        H = int(g.choice([8, 16, 72, 264, 1032]))
        out.append((W, T, H, E, k, 3000 + i))
    return out


@pytest.mark.parametrize("W,T,H,E,k,seed", _moe_cases())
def test_moe_random_shapes(W, T, H, E, k, seed):
    from test_gpu_moe import MoECase, _check_route
    from gpu_util import assert_close
    inp = synth.moe_inputs(W, T, H, E, k, seed=seed)
    r = oracle.moe_route(inp.topk, E)
    case = MoECase(inp)
    recv = oracle.moe_dispatch(inp.x, r["slot"], W * T * k)
    _, out64 = oracle.moe_combine(recv, r["slot"], inp.gate)
    for _ in range(2):   # the workspace and outputs are reused by the second call
        case.run()
        _check_route(case, r)
        assert np.array_equal(to_bits(case.recv), recv)
        assert_close(np.stack([to_bits(case.out(s)) for s in range(W)]), out64)


def _ring_cases(n=8, seed=2027):
    g = np.random.default_rng(seed)
    out = []
    for i in range(n):
        W = int(g.choice([2, 3, 4, 5, 8]))
        count = 4 * W * int(g.choice([1, 3, 250, 1000, 4099]))
        tile = 4 * int(g.choice([0, 1, 16, 257]))
        G = int(g.choice([0, 1, 3]))
        out.append((W, count, tile, G, 4000 + i))
    return out


@pytest.mark.parametrize("W,count,tile,G,seed", _ring_cases())
def test_ring_allreduce_random_shapes_bit_exact(W, count, tile, G, seed):
    from test_gpu_allreduce import RingCase
    case = RingCase(W, count, seed=seed, integer=True)
    want = oracle.allreduce(case.xs)
    for _ in range(2):
        outs, _ = case.run(tile_elems=tile, ctas_per_rank=G)
        for r in range(W):
            assert np.array_equal(outs[r].astype(np.float64), want), r


def _flash_cases(n=8, seed=2028):
    g = np.random.default_rng(seed)
    out = []
    for i in range(n):
        W = int(g.choice([1, 2, 3, 4, 8]))
        Hkv = int(g.choice([1, 2, 4]))
        Hq = Hkv * int(g.choice([1, 2, 8, 16]))
        B = int(g.choice([1, 2, 3]))
        S = W * int(g.choice([1, 63, 64, 65, 300]))
        chunk = int(g.choice([0, 64, 128]))
        out.append((W, B, Hq, Hkv, S, chunk, 5000 + i))
    return out


@pytest.mark.parametrize("W,B,Hq,Hkv,S,chunk,seed", _flash_cases())
def test_flash_decode_random_shapes(W, B, Hq, Hkv, S, chunk, seed):
    from test_gpu_flash import FlashCase
    from gpu_util import assert_close
    case = FlashCase(W, B, Hq, Hkv, S, chunk=chunk, seed=seed, root=seed % W)
    ref = oracle.attention_decode(case.q, case.full(case.k), case.full(case.v))
    for _ in range(2):
        assert_close(case.run(), ref)


def _schedule_cases(n=16, seed=2031):
    """Random shapes with a random schedule drawn from what each shape allows:
    push or pull, one source at a time or all at once, GEMM cluster shape,
    ring stages, producer count and copy-ring shape."""
    g = np.random.default_rng(seed)
    out = []
    for i in range(n):
        W = int(g.choice([1, 2, 3, 4, 8]))
        Ms = int(g.choice([64, 96, 256, 512, 1024]))
        while W * Ms > 4096:
            Ms //= 2
        K = int(g.choice([8, 72, 136, 520]))
        N = int(g.choice([8, 136, 264, 520]))
        M = W * Ms
        clusters = [1] + ([2] if M > 128 else []) + ([4] if Ms % 512 == 0 else [])
        cl = int(g.choice(clusters))
        st = int(g.integers(2, (4 if cl == 1 else 6) + 1))
        warps = int(g.integers(1, 5))
        chunk = int(g.choice([4096, 8192, 16384, 32768]))
        while (196608 // warps) // chunk < 3:
            chunk //= 2
        sched = dict(push=bool(g.integers(0, 2)), source_order=int(g.integers(0, 2)), cluster=cl, stages=st,
                     producers=int(g.choice([0, 4, 8])), producer_warps=warps, producer_chunk=chunk,
                     producer_items=int(g.choice([0, -1, 2])))
        out.append((W, Ms, K, N, int(g.integers(0, 2)), 6000 + i, sched))
    return out


@pytest.mark.parametrize("W,Ms,K,N,lay,seed,sched", _schedule_cases())
def test_ag_random_schedules_bit_exact(W, Ms, K, N, lay, seed, sched):
    inp = synth.ag_inputs(W, Ms, K, N, "int2", seed=seed)
    _, C16 = oracle.ag_gemm(inp.shards, inp.B)
    case = AGCase(inp, b_layout=tdg.B_KN if lay == 0 else tdg.B_NK)
    rank = seed % W
    for mode in ("sm", "ce", "serial"):
        kw = dict(sched)
        if mode != "sm":
            kw.pop("producer_items")
        got, _ = case.run(rank=rank, mode=mode, **kw)
        assert np.array_equal(got, C16), (mode, sched)
        assert np.array_equal(to_bits(case.gathered(rank)), np.concatenate(inp.shards)), (mode, "gathered")


def _rs_schedule_cases(n=10, seed=2032):
    g = np.random.default_rng(seed)
    out = []
    for i in range(n):
        W = int(g.choice([1, 2, 4, 8]))
        Mo = int(g.choice([128, 256, 512, 1024]))
        while W * Mo > 4096:
            Mo //= 2
        K = int(g.choice([8, 64]))
        N = int(g.choice([8, 264, 520]))
        clusters = [1] + ([2] if Mo % 256 == 0 else []) + ([4] if Mo % 512 == 0 else [])
        cl = int(g.choice(clusters))
        obs = [d for d in range(1, W + 1) if W % d == 0]
        sched = dict(cluster=cl, stages=int(g.integers(2, (4 if cl == 1 else 6) + 1)),
                     order=int(g.integers(0, 2)), owner_block=int(g.choice(obs)),
                     red_rows=int(g.choice([4, 8, 16, 32])), partial_f32=bool(g.integers(0, 2)))
        out.append((W, W * Mo, K, N, 7000 + i, sched))
    return out


@pytest.mark.parametrize("W,M,K,N,seed,sched", _rs_schedule_cases())
def test_rs_random_schedules_bit_exact(W, M, K, N, seed, sched):
    inp = synth.rs_inputs(W, M, K, N, "int2", seed=seed)
    _, out16 = oracle.gemm_rs(inp.As, inp.Bs)
    case = RSCase(inp, f32=sched["partial_f32"])
    for mode in ("sm", "serial"):
        got, _ = case.run(mode=mode, **sched)
        assert np.array_equal(got, out16), (mode, sched)
