"""Argument validation through the C ABI: every rejected call returns the
documented error code, launches nothing and leaves the device status clean;
degenerate sizes are no-ops."""
import numpy as np
import pytest
import torch

from tile_centric_comm_gb300 import synth, tdg
from gpu_util import AGCase, RSCase, align

pytestmark = pytest.mark.gpu


def _code(fn):
    with pytest.raises(tdg.TdgError) as ei:
        fn()
    return ei.value.code


def test_ag_gemm_rejections():
    inp = synth.ag_inputs(2, 128, 64, 256, "int2", seed=1)
    c = AGCase(inp, ll=True)
    call = lambda **kw: tdg.ag_gemm(c.symm, kw.pop("rank", 0), kw.pop("Ms", 128), kw.pop("K", 64),
                                    kw.pop("N", 256), kw.pop("a_off", c.a_off), kw.pop("g_off", c.g_off),
                                    c.B, c.C, **kw)
    assert _code(lambda: call(N=250)) == tdg.TDG_ERR_INVALID             # N not a multiple of 8
    assert _code(lambda: call(a_off=8)) == tdg.TDG_ERR_INVALID           # misaligned shard
    assert _code(lambda: call(g_off=c.a_off)) == tdg.TDG_ERR_INVALID     # gathered overlaps the shard
    assert _code(lambda: call(rank=2)) == tdg.TDG_ERR_INVALID            # rank out of range
    assert _code(lambda: call(signal_rows=48)) == tdg.TDG_ERR_INVALID    # does not divide Ms
    assert _code(lambda: call(Ms=1 << 20)) == tdg.TDG_ERR_NOMEM          # regions too small
    assert _code(lambda: call(mode="ce")) == tdg.TDG_ERR_INVALID         # CE needs a side stream
    assert _code(lambda: call(mode="ll", ll_off=c.g_off)) == tdg.TDG_ERR_INVALID  # LL overlaps gathered
    assert _code(lambda: call(source_order=2)) == tdg.TDG_ERR_INVALID
    torch.cuda.synchronize()
    assert c.symm.status()["code"] == 0
    got, _ = c.run(rank=1, mode="sm")                                   # still usable
    import oracle
    assert np.array_equal(got, oracle.ag_gemm(inp.shards, inp.B)[1])


def test_gemm_rs_rejections():
    inp = synth.rs_inputs(2, 512, 64, 256, "int2", seed=2)
    c = RSCase(inp)
    call = lambda **kw: tdg.gemm_rs(c.symm, kw.pop("M", 512), kw.pop("K", 64), kw.pop("N", 256),
                                    kw.pop("a_off", c.a_off), c.b_off, c.stage_off, c.out_off, **kw)
    assert _code(lambda: call(M=384)) == tdg.TDG_ERR_INVALID             # M/W not a multiple of 128
    assert _code(lambda: call(N=252)) == tdg.TDG_ERR_INVALID
    assert _code(lambda: call(a_off=4)) == tdg.TDG_ERR_INVALID
    assert _code(lambda: call(owner_block=3)) == tdg.TDG_ERR_INVALID     # does not divide W
    assert _code(lambda: call(M=1 << 20)) == tdg.TDG_ERR_NOMEM
    torch.cuda.synchronize()
    assert c.symm.status()["code"] == 0


def test_moe_rejections_and_empty():
    from test_gpu_moe import MoECase
    inp = synth.moe_inputs(2, 64, 128, 16, 4, seed=3)
    c = MoECase(inp)
    def call(T=64, H=128, E=16, k=4, phases=tdg.MOE_ALL, ws=None):
        tdg.moe_dispatch_combine(c.symm, T, H, E, k, c.x_off, c.topk_off, c.gate_off, c.out_off,
                                 c.recv, c.counts, c.base, c.slot, c.ws if ws is None else ws,
                                 phases=phases)
    assert _code(lambda: call(E=15)) == tdg.TDG_ERR_INVALID              # E not a multiple of W
    assert _code(lambda: call(k=17)) == tdg.TDG_ERR_INVALID              # k > E
    assert _code(lambda: call(H=100)) == tdg.TDG_ERR_INVALID             # H not a multiple of 8
    assert _code(lambda: call(phases=0)) == tdg.TDG_ERR_INVALID
    small = torch.empty(16, dtype=torch.uint8, device="cuda")
    assert _code(lambda: call(ws=small)) == tdg.TDG_ERR_NOMEM            # workspace too small
    call(T=0)                                                            # no tokens: a no-op
    torch.cuda.synchronize()
    assert c.symm.status()["code"] == 0


def test_flash_decode_rejections():
    from test_gpu_flash import FlashCase
    c = FlashCase(2, 1, 8, 1, 256, 64, seed=4)
    def call(**kw):
        a = dict(B=1, Hq=8, Hkv=1, D=128, S=256, chunk=64)
        a.update(kw)
        tdg.flash_decode(c.symm, a["B"], a["Hq"], a["Hkv"], a["D"], a["S"], c.k_off, c.v_off, c.part_off,
                         c.qd, c.out, chunk=a["chunk"], root=kw.get("root", 0))
    assert _code(lambda: call(S=255)) == tdg.TDG_ERR_INVALID             # S not a multiple of W
    assert _code(lambda: call(D=64)) == tdg.TDG_ERR_INVALID              # head dim other than 128
    assert _code(lambda: call(Hq=6, Hkv=4)) == tdg.TDG_ERR_INVALID       # Hq not a multiple of Hkv
    assert _code(lambda: call(Hq=32, Hkv=1)) == tdg.TDG_ERR_INVALID      # more than 16 heads per kv head
    assert _code(lambda: call(chunk=96)) == tdg.TDG_ERR_INVALID          # chunk not a multiple of 64
    assert _code(lambda: call(root=2)) == tdg.TDG_ERR_INVALID
    assert _code(lambda: call(S=1 << 24)) == tdg.TDG_ERR_NOMEM
    torch.cuda.synchronize()
    assert c.symm.status()["code"] == 0
