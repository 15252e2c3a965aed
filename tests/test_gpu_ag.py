"""GPU parity of AllGather+GEMM (through the C ABI) against the CPU oracle."""
import numpy as np
import pytest
import torch

import oracle
from tile_centric_comm_gb300 import synth, tdg
from gpu_util import AGCase, assert_close, to_bits

pytestmark = pytest.mark.gpu


def _gathered_ok(case, rank):
    g = to_bits(case.gathered(rank))
    assert np.array_equal(g, np.concatenate(case.inp.shards)), "gathered buffer differs"


def test_tiny_integer_bit_exact_all_modes_and_ranks():
    # W=2, A_r 64x256, B 256x128, integers in [-2, 2]: bit-exact
    inp = synth.make("ag_tiny")
    C64, C16 = oracle.ag_gemm(inp.shards, inp.B)
    case = AGCase(inp)
    for mode in ("sm", "serial", "ce"):
        for rank in range(inp.W):
            got, _ = case.run(rank=rank, mode=mode)
            assert np.array_equal(got, C16), (mode, rank)
            _gathered_ok(case, rank)


@pytest.mark.parametrize("cluster", [0, 1])
@pytest.mark.parametrize("b_layout", [tdg.B_KN, tdg.B_NK])
@pytest.mark.parametrize("W,Ms,K,N", [
    (4, 256, 320, 520),     # 8 m tiles, 3 n tiles (last one 8 columns), 5 k blocks
    (3, 96, 136, 264),      # Ms not a multiple of 128: gathered read, ragged m tail
    (2, 128, 64, 256),      # exactly one k block, full n tile
    (2, 384, 128, 136),     # pairs: 3 tiles of 256 rows, the last half empty
])
def test_float_parity_small(W, Ms, K, N, b_layout, cluster):
    # cluster 0: the default shape (CTA pairs, cta_group::2, 256-row tiles,
    # where the shape allows); cluster 1: one CTA per 128-row tile
    inp = synth.ag_inputs(W, Ms, K, N, "normal", seed=W * 7 + K)
    C64, C16 = oracle.ag_gemm(inp.shards, inp.B)
    case = AGCase(inp, b_layout=b_layout)
    for mode in ("sm", "serial", "ce"):
        got, _ = case.run(rank=W - 1, mode=mode, cluster=cluster)
        assert_close(got, C64)
        _gathered_ok(case, W - 1)


@pytest.mark.parametrize("cluster", [0, 1])
def test_integer_exact_larger_and_swizzle_invariance(cluster):
    # integer inputs, |sums| <= 4K: exact in fp32; output identical for every
    # rank, swizzle on/off, signal granularity and producer count
    inp = synth.ag_inputs(4, 256, 512, 384, "int2", seed=3)
    _, C16 = oracle.ag_gemm(inp.shards, inp.B)
    case = AGCase(inp)
    outs = []
    for rank in range(4):
        for swz in (True, False):
            for sig in (0, 64, 256):
                got, _ = case.run(rank=rank, mode="sm", swizzle=swz, signal_rows=sig,
                                  producers=4 + rank, cluster=cluster)
                outs.append(got)
    for o in outs:
        assert np.array_equal(o, C16)


@pytest.mark.parametrize("cluster", [2, 1])
@pytest.mark.parametrize("N", [2440, 2432])
def test_split_tail_wave_bit_exact(N, cluster):
    # 2048 x N: 80 pair tiles (160 single tiles) over 76 pairs (152 CTAs), so
    # the last wave's few tiles are cut into 128-column halves; with N = 2440
    # the last n tile is 136 wide (halves of 128 and 8), with N = 2432 it is
    # 128 wide (its second half is empty and skipped by every role)
    inp = synth.ag_inputs(8, 256, 64, N, "int2", seed=N)
    _, C16 = oracle.ag_gemm(inp.shards, inp.B)
    case = AGCase(inp)
    for mode in ("ce", "sm", "serial"):
        got, _ = case.run(rank=5, mode=mode, cluster=cluster, split_tail=True, producer_items=-1)
        assert np.array_equal(got, C16), mode


def test_timeout_reported_then_next_call_succeeds():
    # fault injection on the host side: producers skip one notify; the consumer's
    # bounded wait must run out, report TIMEOUT with the signal index, and the
    # next call (new epoch) must succeed.
    inp = synth.ag_inputs(2, 128, 64, 256, "int2", seed=1)
    _, C16 = oracle.ag_gemm(inp.shards, inp.B)
    case = AGCase(inp)
    # group 4 = rows 128..159 = the first rows of shard 1, remote for rank 0
    _, st = case.run(rank=0, mode="sm", signal_rows=32, test_skip_notify=1 << 4,
                     timeout_ns=20_000_000, check_status=False)
    assert st["code"] == tdg.TDG_ERR_TIMEOUT and st["where"] == "ag_flag" and st["index"] == 4
    got, st = case.run(rank=0, mode="sm", signal_rows=32)
    assert st["code"] == 0 and np.array_equal(got, C16)


def test_ll_mode_bit_exact_and_words_match_the_codec():
    # LL path: 8-byte {payload, flag=epoch} words; the GEMM result, the gathered
    # buffer and every LL word are bit-exact (words against the oracle's codec)
    inp = synth.make("ag_tiny")
    _, C16 = oracle.ag_gemm(inp.shards, inp.B)
    case = AGCase(inp, ll=True)
    payload = np.concatenate(inp.shards).view(np.uint32).reshape(-1)
    for rank in range(inp.W):
        epoch = case.symm.epoch()
        got, _ = case.run(rank=rank, mode="ll", ll_off=case.ll_off)
        assert np.array_equal(got, C16)
        _gathered_ok(case, rank)
        assert np.array_equal(case.ll_words(rank), oracle.ll_pack(payload, epoch))


@pytest.mark.parametrize("mode", ["sm", "ce", "ll", "serial"])
def test_all_sources_at_once_order_bit_exact(mode):
    # the full-mesh source order (round robin over sources) gives the same bits
    inp = synth.ag_inputs(4, 96, 200, 136, "int2", seed=21)
    _, C16 = oracle.ag_gemm(inp.shards, inp.B)
    case = AGCase(inp, ll=True)
    for rank in (0, 3):
        got, _ = case.run(rank=rank, mode=mode, source_order=1, ll_off=case.ll_off,
                          signal_rows=32)
        assert np.array_equal(got, C16), (mode, rank)
        _gathered_ok(case, rank)


def test_ll_mode_float_parity():
    inp = synth.ag_inputs(4, 128, 256, 264, "normal", seed=12)
    C64, _ = oracle.ag_gemm(inp.shards, inp.B)
    case = AGCase(inp, ll=True)
    got, _ = case.run(rank=2, mode="ll", ll_off=case.ll_off, signal_rows=32)
    assert_close(got, C64)
    _gathered_ok(case, 2)


def test_ll_missing_words_time_out_then_recover():
    # the senders skip the words of group 1 (host-side injection): the
    # receiver's bounded spin runs out and reports it; the next call succeeds
    inp = synth.make("ag_tiny")
    _, C16 = oracle.ag_gemm(inp.shards, inp.B)
    case = AGCase(inp, ll=True)
    _, st = case.run(rank=0, mode="ll", ll_off=case.ll_off, test_skip_notify=1 << 1,
                     timeout_ns=20_000_000, check_status=False)
    assert st["code"] == tdg.TDG_ERR_TIMEOUT and st["where"] == "ll" and st["index"] == 1
    got, st = case.run(rank=0, mode="ll", ll_off=case.ll_off)
    assert st["code"] == 0 and np.array_equal(got, C16)


def test_degenerate_shapes():
    # K == 0 gives C = 0; N == 0 and Ms == 0 are no-ops
    inp = synth.ag_inputs(2, 64, 8, 16, "int2", seed=2)
    case = AGCase(inp)
    tdg.ag_gemm(case.symm, 0, 64, 0, 16, case.a_off, case.g_off, case.B, case.C)
    torch.cuda.synchronize()
    assert np.all(to_bits(case.C) == 0)
    case.C.view(torch.int16).fill_(7)
    tdg.ag_gemm(case.symm, 0, 64, 8, 0, case.a_off, case.g_off, case.B, case.C)
    tdg.ag_gemm(case.symm, 0, 0, 8, 16, case.a_off, case.g_off, case.B, case.C)
    torch.cuda.synchronize()
    assert np.all(to_bits(case.C) == 7)
    B12 = torch.zeros(12, 16, dtype=torch.bfloat16, device="cuda")
    with pytest.raises(tdg.TdgError):     # K not a multiple of 8
        tdg.ag_gemm(case.symm, 0, 64, 12, 16, case.a_off, case.g_off, B12, case.C)
    with pytest.raises(tdg.TdgError):     # bad rank
        tdg.ag_gemm(case.symm, 2, 64, 8, 16, case.a_off, case.g_off, case.B, case.C)


@pytest.mark.slow
@pytest.mark.parametrize("name", ["ag_qwen32b_up", "ag_llama70b_gateup"])
def test_full_size_sampled(name):
    inp = synth.make(name)
    case = AGCase(inp)
    g = np.random.default_rng(0)
    M, N = case.M, inp.N
    rows = np.concatenate([g.integers(0, M, 1500), [0, M - 1]])
    cols = np.concatenate([g.integers(0, N, 1500), [N - 1, 0]])
    ref = oracle.ag_gemm_sampled(inp.shards, inp.B, rows, cols)
    # ce is the mode the benchmark times; every mode must reproduce the oracle
    # at the full size and leave the bit-exact gathered buffer
    for mode in ("ce", "sm", "serial"):
        got, _ = case.run(rank=3, mode=mode)
        assert_close(got[rows, cols], ref)
        _gathered_ok(case, 3)
    del case
    torch.cuda.empty_cache()


def test_ll_second_heap_on_the_same_memory():
    # a heap laid over memory that an earlier heap's LL call filled with words:
    # the new call's epoch differs from every earlier call's, so no stale word
    # counts as delivered and the result is exact for the new inputs
    first = synth.ag_inputs(2, 256, 64, 128, "int2", seed=21)
    second = synth.ag_inputs(2, 256, 64, 128, "int2", seed=22)
    case = AGCase(first, ll=True)
    _, C1 = oracle.ag_gemm(first.shards, first.B)
    for _ in range(3):
        got, _ = case.run(rank=1, mode="ll", ll_off=case.ll_off)
        assert np.array_equal(got, C1)
    buf, region, nsig = case.symm.buf, case.symm.region_bytes, case.symm.nsig
    case.symm.close()
    again = AGCase.__new__(AGCase)
    again.__dict__.update(case.__dict__)
    again.inp = second
    again.symm = tdg.Symm(2, region, nsig, buffer=buf)   # same memory, new handle
    for s in range(2):
        again.symm.view(s, again.a_off, (second.Ms, second.K), torch.bfloat16).copy_(
            torch.from_numpy(second.shards[s].view(np.int16)).view(torch.bfloat16).cuda())
    again.B = torch.from_numpy(second.B.view(np.int16)).view(torch.bfloat16).cuda()
    _, C2 = oracle.ag_gemm(second.shards, second.B)
    # two calls of another mode first: with epochs counted per handle, the LL
    # call below would take the epoch of the stale words (the third call)
    for _ in range(2):
        got, _ = again.run(rank=1, mode="sm")
        assert np.array_equal(got, C2)
    got, _ = again.run(rank=1, mode="ll", ll_off=again.ll_off)
    assert np.array_equal(got, C2)


@pytest.mark.parametrize("items", [4, 1, 0, -1, 40])
def test_sm_mode_producers_take_the_last_items(items):
    # 36 two-pair-cluster tiles (M 6144, 3 n tiles); 16 producer CTAs are 4
    # clusters.  producer_items n > 0: the producer clusters take the last n
    # items after their copies (40 > 36: all of them, the GEMM clusters none);
    # 0: the split balanced on the host; -1: none.  Every split gives the
    # oracle's bits.
    inp = synth.ag_inputs(4, 1536, 128, 520, "int2", seed=17)
    _, C16 = oracle.ag_gemm(inp.shards, inp.B)
    case = AGCase(inp)
    for rank in (0, 3):
        got, _ = case.run(rank=rank, mode="sm", producers=16, producer_items=items)
        assert np.array_equal(got, C16), rank
        _gathered_ok(case, rank)
