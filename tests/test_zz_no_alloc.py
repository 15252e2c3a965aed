"""The allocation-free MoE entry point (tdg_moe_dispatch_combine_noalloc).

Some callers cannot allocate device memory at the moment they call -- a
runtime that hands out all memory from a fixed budget at start-up, or code
without an allocator of its own -- so they cannot pass the routing workspace
that tdg_moe_dispatch_combine needs.  The allocation-free variant keeps that
scratch in a fixed 2 MiB device array inside the library instead.

These tests call it through the C ABI, two calls in a row (the second reuses
the array the first left behind), and check its routing tables and receive
rows bit for bit against the oracle, its combined output against the oracle
within the float tolerance of the other tests, and every output bit for bit
against the regular entry point's (both run the same kernels on the same
inputs).  Bad arguments get the regular entry point's codes, whatever scratch
they would need.  The file is named so that pytest collects it last.
"""
import numpy as np
import pytest
import torch

import oracle
from tile_centric_comm_gb300 import synth, tdg
from gpu_util import POISON, align, assert_close, bf16_f64, to_bits, to_dev_bf16

pytestmark = pytest.mark.gpu


def _setup(W, T, H, E, k, seed):
    inp = synth.moe_inputs(W, T, H, E, k, seed=seed)
    x_off = 0
    topk_off = align(T * H * 2)
    gate_off = align(topk_off + T * k * 4)
    out_off = align(gate_off + T * k * 4)
    symm = tdg.Symm(W, align(out_off + T * H * 2 + 1024), 1024)
    for s in range(W):
        symm.view(s, x_off, (T, H), torch.bfloat16).copy_(to_dev_bf16(inp.x[s]))
        symm.view(s, topk_off, (T, k), torch.int32).copy_(torch.from_numpy(np.ascontiguousarray(inp.topk[s])))
        symm.view(s, gate_off, (T, k), torch.float32).copy_(torch.from_numpy(np.ascontiguousarray(inp.gate[s])))
    return inp, symm, (x_off, topk_off, gate_off, out_off)


def _outputs(W, T, H, E, k):
    total = W * T * k
    return dict(recv=torch.empty((total, H), dtype=torch.bfloat16, device="cuda"),
                counts=torch.empty((W, E), dtype=torch.int64, device="cuda"),
                base=torch.empty(E + 1, dtype=torch.int64, device="cuda"),
                slot=torch.empty((W, T, k), dtype=torch.int64, device="cuda"),
                row_src=torch.empty(total, dtype=torch.int32, device="cuda"),
                row_tok=torch.empty(total, dtype=torch.int32, device="cuda"),
                row_k=torch.empty(total, dtype=torch.int32, device="cuda"))


def _poison(o, symm, out_off, W, T, H):
    o["recv"].view(torch.int16).fill_(POISON)
    for key in ("counts", "base", "slot"):
        o[key].fill_(-7)
    for key in ("row_src", "row_tok", "row_k"):
        o[key].fill_(-7)
    for s in range(W):
        symm.view(s, out_off, (T, H), torch.bfloat16).view(torch.int16).fill_(POISON)


def _snapshot(o, symm, out_off, W, T, H):
    snap = {k: v.cpu().numpy().copy() if v.dtype != torch.bfloat16 else to_bits(v) for k, v in o.items()}
    snap["out"] = np.stack([to_bits(symm.view(s, out_off, (T, H), torch.bfloat16)) for s in range(W)])
    return snap


@pytest.mark.parametrize("W,T,H,E,k", [(4, 257, 512, 64, 8), (8, 512, 7168, 256, 8)])
def test_noalloc_matches_oracle_and_regular_entry_point_twice(W, T, H, E, k):
    inp, symm, (x_off, topk_off, gate_off, out_off) = _setup(W, T, H, E, k, seed=T + 1)
    r = oracle.moe_route(inp.topk, E)
    recv_ref = oracle.moe_dispatch(inp.x, r["slot"], W * T * k)
    _, out64 = oracle.moe_combine(recv_ref, r["slot"], inp.gate)
    o = _outputs(W, T, H, E, k)
    ws = torch.empty(tdg.moe_workspace_bytes(W, T, E), dtype=torch.uint8, device="cuda")

    _poison(o, symm, out_off, W, T, H)
    tdg.moe_dispatch_combine(symm, T, H, E, k, x_off, topk_off, gate_off, out_off, o["recv"],
                             o["counts"], o["base"], o["slot"], ws, row_src=o["row_src"],
                             row_tok=o["row_tok"], row_k=o["row_k"])
    torch.cuda.synchronize()
    assert symm.status()["code"] == 0
    regular = _snapshot(o, symm, out_off, W, T, H)

    for _ in range(2):  # two calls in a row share (and reuse) the fixed array
        _poison(o, symm, out_off, W, T, H)
        tdg.moe_dispatch_combine_noalloc(symm, T, H, E, k, x_off, topk_off, gate_off, out_off,
                                         o["recv"], o["counts"], o["base"], o["slot"],
                                         row_src=o["row_src"], row_tok=o["row_tok"], row_k=o["row_k"])
        torch.cuda.synchronize()
        assert symm.status()["code"] == 0
        got = _snapshot(o, symm, out_off, W, T, H)
        # against the oracle: routing and receive rows bit-exact, combine within tolerance
        for key in ("counts", "base", "slot", "row_src", "row_tok", "row_k"):
            assert np.array_equal(got[key], r[key]), key
        assert np.array_equal(got["recv"], recv_ref)
        assert_close(got["out"], out64)
        # against the regular entry point: the same kernels, so the same bits everywhere
        for key in regular:
            assert np.array_equal(got[key], regular[key]), key


def test_noalloc_rejects_routing_beyond_the_fixed_array():
    # W * ceil(T/64) * E = 8 * 129 * 256 > 262144 entries: rejected before any launch
    inp, symm, (x_off, topk_off, gate_off, out_off) = _setup(8, 8256, 8, 256, 2, seed=1)
    o = _outputs(8, 8256, 8, 256, 2)
    with pytest.raises(tdg.TdgError) as ei:
        tdg.moe_dispatch_combine_noalloc(symm, 8256, 8, 256, 2, x_off, topk_off, gate_off, out_off,
                                         o["recv"], o["counts"], o["base"], o["slot"])
    assert ei.value.code == tdg.TDG_ERR_NOMEM


def test_noalloc_bad_arguments_get_the_regular_codes():
    # an expert count above the limit (4096) or a world that is not the heap's
    # is an invalid argument for both entry points, although its routing
    # scratch would also exceed the fixed array; nothing is launched
    W, T, H, k = 8, 8256, 8, 2
    inp, symm, (x_off, topk_off, gate_off, out_off) = _setup(W, T, H, 256, k, seed=2)
    o = _outputs(W, T, H, 8192, k)
    ws = torch.empty(16, dtype=torch.uint8, device="cuda")
    for fn, extra in ((tdg.moe_dispatch_combine_noalloc, ()), (tdg.moe_dispatch_combine, (ws,))):
        with pytest.raises(tdg.TdgError) as ei:
            fn(symm, T, H, 8192, k, x_off, topk_off, gate_off, out_off, o["recv"], o["counts"],
               o["base"], o["slot"], *extra)
        assert ei.value.code == tdg.TDG_ERR_INVALID, fn.__name__
    a = tdg._moe_args(symm, T, H, 256, k, x_off, topk_off, gate_off, out_off, o["recv"], o["counts"],
                      o["base"], o["slot"], None, None, None, None, tdg.MOE_ALL)
    a.world = 4                                    # the heap has 8 ranks
    import ctypes
    rc = tdg.lib().tdg_moe_dispatch_combine_noalloc(symm.h, ctypes.byref(a), tdg._stream(None))
    assert rc == tdg.TDG_ERR_INVALID
    torch.cuda.synchronize()
    assert symm.status()["code"] == 0
