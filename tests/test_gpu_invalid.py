"""Argument validation.  Through the C ABI (the argument structs passed to
libtdg as they are): every rejected call returns the documented error code,
launches nothing and leaves the device status clean; degenerate sizes are
no-ops.  Through the Python binding: tensors whose layout the library cannot
see (dtype, contiguity, size) are refused before any call."""
import ctypes

import numpy as np
import pytest
import torch

from tile_centric_comm_gb300 import synth, tdg
from gpu_util import AGCase, RSCase

pytestmark = pytest.mark.gpu


def _ag_rc(c, **kw):
    a = tdg.AgGemmArgs(world=c.symm.world, rank=0, Ms=128, K=64, N=256, a_off=c.a_off,
                       g_off=c.g_off, B=c.B.data_ptr(), C=c.C.data_ptr(), b_layout=tdg.B_KN,
                       mode=tdg.MODE_SM, swizzle=1)
    side = kw.pop("side", None)
    for key, v in kw.items():
        setattr(a, key, v)
    cur = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    return tdg.lib().tdg_ag_gemm(c.symm.h, ctypes.byref(a), cur, ctypes.c_void_p(side))


def test_ag_gemm_rejections():
    inp = synth.ag_inputs(2, 128, 64, 256, "int2", seed=1)
    c = AGCase(inp, ll=True)
    assert _ag_rc(c, N=250) == tdg.TDG_ERR_INVALID                    # N not a multiple of 8
    assert _ag_rc(c, a_off=8) == tdg.TDG_ERR_INVALID                  # misaligned shard
    assert _ag_rc(c, g_off=c.a_off) == tdg.TDG_ERR_INVALID            # gathered overlaps the shard
    assert _ag_rc(c, rank=2) == tdg.TDG_ERR_INVALID                   # rank out of range
    assert _ag_rc(c, signal_rows=48) == tdg.TDG_ERR_INVALID           # does not divide Ms
    assert _ag_rc(c, Ms=1 << 20) == tdg.TDG_ERR_NOMEM                 # regions too small
    assert _ag_rc(c, mode=tdg.MODE_CE) == tdg.TDG_ERR_INVALID         # CE needs a side stream
    assert _ag_rc(c, mode=tdg.MODE_LL, ll_off=c.g_off) == tdg.TDG_ERR_INVALID  # LL overlaps gathered
    assert _ag_rc(c, source_order=2) == tdg.TDG_ERR_INVALID
    assert _ag_rc(c, mode=7) == tdg.TDG_ERR_INVALID
    assert _ag_rc(c, b_layout=2) == tdg.TDG_ERR_INVALID
    assert _ag_rc(c, c_f32=2) == tdg.TDG_ERR_INVALID
    torch.cuda.synchronize()
    assert c.symm.status()["code"] == 0
    got, _ = c.run(rank=1, mode="sm")                                  # still usable
    import oracle
    assert np.array_equal(got, oracle.ag_gemm(inp.shards, inp.B)[1])


def test_gemm_rs_rejections():
    inp = synth.rs_inputs(2, 512, 64, 256, "int2", seed=2)
    c = RSCase(inp)

    def rc(**kw):
        a = tdg.GemmRsArgs(world=2, M=512, K=64, N=256, a_off=c.a_off, b_off=c.b_off,
                           stage_off=c.stage_off, out_off=c.out_off, b_layout=tdg.B_KN,
                           mode=tdg.MODE_SM)
        for key, v in kw.items():
            setattr(a, key, v)
        cur = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
        return tdg.lib().tdg_gemm_rs(c.symm.h, ctypes.byref(a), cur)
    assert rc(M=384) == tdg.TDG_ERR_INVALID                           # M/W not a multiple of 128
    assert rc(N=252) == tdg.TDG_ERR_INVALID
    assert rc(a_off=4) == tdg.TDG_ERR_INVALID
    assert rc(owner_block=3) == tdg.TDG_ERR_INVALID                   # does not divide W
    assert rc(world=3) == tdg.TDG_ERR_INVALID                         # not the heap's world
    assert rc(mode=tdg.MODE_CE) == tdg.TDG_ERR_INVALID                # SM or SERIAL only
    assert rc(partial_f32=2) == tdg.TDG_ERR_INVALID
    assert rc(partial_f32=1) == tdg.TDG_ERR_NOMEM                     # fp32 staging runs past the region
    assert rc(out_off=c.stage_off) == tdg.TDG_ERR_INVALID             # out overlaps the staging
    assert rc(stage_off=c.b_off) == tdg.TDG_ERR_INVALID               # staging overlaps B
    assert rc(out_off=c.a_off) == tdg.TDG_ERR_INVALID                 # out overlaps A
    assert rc(M=1 << 20) == tdg.TDG_ERR_NOMEM
    torch.cuda.synchronize()
    assert c.symm.status()["code"] == 0


def test_moe_rejections_and_empty():
    from test_gpu_moe import MoECase
    inp = synth.moe_inputs(2, 64, 128, 16, 4, seed=3)
    c = MoECase(inp)

    def rc(T=64, H=128, E=16, k=4, phases=tdg.MOE_ALL, ws=None, out_off=None):
        ws = c.ws if ws is None else ws
        a = tdg.MoeArgs(world=2, T=T, H=H, E=E, k=k, x_off=c.x_off, topk_off=c.topk_off,
                        gate_off=c.gate_off, out_off=c.out_off if out_off is None else out_off,
                        recv=c.recv.data_ptr(),
                        counts=c.counts.data_ptr(), base=c.base.data_ptr(), slot=c.slot.data_ptr(),
                        workspace=ws.data_ptr(), workspace_bytes=ws.numel(), phases=phases)
        cur = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
        return tdg.lib().tdg_moe_dispatch_combine(c.symm.h, ctypes.byref(a), cur)
    assert rc(E=15) == tdg.TDG_ERR_INVALID                            # E not a multiple of W
    assert rc(k=17) == tdg.TDG_ERR_INVALID                            # k > E
    assert rc(H=100) == tdg.TDG_ERR_INVALID                           # H not a multiple of 8
    assert rc(phases=0) == tdg.TDG_ERR_INVALID
    assert rc(out_off=c.gate_off) == tdg.TDG_ERR_INVALID                  # out over the gates, combining
    small = torch.empty(16, dtype=torch.uint8, device="cuda")
    assert rc(ws=small) == tdg.TDG_ERR_NOMEM                          # workspace too small
    assert rc(T=0) == tdg.TDG_OK                                      # no tokens: a no-op
    torch.cuda.synchronize()
    assert c.symm.status()["code"] == 0


def test_flash_decode_rejections():
    from test_gpu_flash import FlashCase
    c = FlashCase(2, 1, 8, 1, 256, 64, seed=4)

    def rc(**kw):
        a = tdg.FlashDecodeArgs(world=2, root=0, B=1, Hq=8, Hkv=1, D=128, S=256, k_off=c.k_off,
                                v_off=c.v_off, part_off=c.part_off, q=c.qd.data_ptr(),
                                out=c.out.data_ptr(), chunk=64)
        for key, v in kw.items():
            setattr(a, key, v)
        cur = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
        return tdg.lib().tdg_flash_decode(c.symm.h, ctypes.byref(a), cur)
    assert rc(S=255) == tdg.TDG_ERR_INVALID                           # S not a multiple of W
    assert rc(D=64) == tdg.TDG_ERR_INVALID                            # head dim other than 128
    assert rc(Hq=6, Hkv=4) == tdg.TDG_ERR_INVALID                     # Hq not a multiple of Hkv
    assert rc(Hq=32, Hkv=1) == tdg.TDG_ERR_INVALID                    # more than 16 heads per kv head
    assert rc(chunk=96) == tdg.TDG_ERR_INVALID                        # chunk not a multiple of 64
    assert rc(root=2) == tdg.TDG_ERR_INVALID
    assert rc(part_off=c.v_off) == tdg.TDG_ERR_INVALID                # partials overlap V
    assert rc(S=1 << 24) == tdg.TDG_ERR_NOMEM
    torch.cuda.synchronize()
    assert c.symm.status()["code"] == 0


def test_binding_refuses_tensors_it_cannot_describe():
    inp = synth.ag_inputs(2, 128, 64, 256, "int2", seed=5)
    c = AGCase(inp)
    call = lambda B, C: tdg.ag_gemm(c.symm, 0, 128, 64, 256, c.a_off, c.g_off, B, C)
    with pytest.raises(ValueError, match="contiguous"):
        call(c.B.t().contiguous().t(), c.C)                           # K x N values, N x K memory
    with pytest.raises(TypeError, match="bfloat16"):
        call(c.B.float(), c.C)
    with pytest.raises(ValueError, match="needs"):
        call(c.B, c.C[:100])                                          # C too small for M x N
    with pytest.raises(ValueError, match="CUDA"):
        call(c.B.cpu(), c.C)
    from test_gpu_flash import FlashCase
    f = FlashCase(2, 1, 8, 1, 256, 64, seed=6)
    with pytest.raises(ValueError, match="needs"):
        tdg.flash_decode(f.symm, 1, 32, 1, 128, 256, f.k_off, f.v_off, f.part_off, f.qd, f.out)
    with pytest.raises(ValueError, match="rank"):
        c.symm.view(2, 0, (4,), torch.int32)
    torch.cuda.synchronize()
    assert c.symm.status()["code"] == 0
    got, _ = c.run(rank=0, mode="sm")                                  # nothing was launched
    import oracle
    assert np.array_equal(got, oracle.ag_gemm(inp.shards, inp.B)[1])


def test_ag_gemm_all_ranks_rejections():
    from test_gpu_ag_all import AGAllCase
    inp = synth.ag_all_inputs(2, 128, 64, 256, "int2", seed=7)
    c = AGAllCase(inp)

    def rc(side=None, **kw):
        a = tdg.AgGemmAllArgs(world=2, Ms=128, K=64, N=256, a_off=c.a_off, g_off=c.g_off,
                              b_off=c.b_off, c_off=c.c_off, b_layout=tdg.B_KN, mode=tdg.MODE_SERIAL)
        for key, v in kw.items():
            setattr(a, key, v)
        cur = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
        return tdg.lib().tdg_ag_gemm_all_ranks(c.symm.h, ctypes.byref(a), cur, ctypes.c_void_p(side))
    assert rc(mode=tdg.MODE_SM) == tdg.TDG_ERR_INVALID                # CE or SERIAL only
    assert rc(mode=tdg.MODE_CE) == tdg.TDG_ERR_INVALID                # CE needs a side stream
    assert rc(N=250) == tdg.TDG_ERR_INVALID
    assert rc(b_off=8) == tdg.TDG_ERR_INVALID                         # misaligned
    assert rc(c_off=c.b_off) == tdg.TDG_ERR_INVALID                   # C overlaps B
    assert rc(g_off=c.a_off) == tdg.TDG_ERR_INVALID                   # gathered overlaps the shard
    assert rc(signal_rows=48) == tdg.TDG_ERR_INVALID                  # does not divide Ms
    assert rc(world=3) == tdg.TDG_ERR_INVALID
    assert rc(c_f32=2) == tdg.TDG_ERR_INVALID
    assert rc(c_f32=1) == tdg.TDG_ERR_NOMEM                         # fp32 C_r runs past the region
    assert rc(Ms=1 << 20) == tdg.TDG_ERR_NOMEM
    torch.cuda.synchronize()
    assert c.symm.status()["code"] == 0
