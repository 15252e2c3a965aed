"""Helpers for the GPU parity tests: place seeded inputs into a symmetric heap,
run the CUDA path through the C ABI, and bring results back as bf16 bit
patterns.  (Test infrastructure; imports the oracle only in the tests.)"""
from __future__ import annotations

import numpy as np
import torch

from tile_centric_comm_gb300 import tdg

POISON = 0x7FC1  # a NaN bf16 pattern written into outputs before each call


def to_dev_bf16(bits: np.ndarray, device="cuda") -> torch.Tensor:
    t = torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16)
    return t.to(device)


def to_bits(t: torch.Tensor) -> np.ndarray:
    return t.contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


def align(x, a=1024):
    return (x + a - 1) // a * a


def bf16_f64(bits):
    return (np.ascontiguousarray(bits, np.uint16).astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def assert_close(got_bits, ref64, tol=1e-2):
    """max|got - ref| <= tol * max|ref| (the float tolerance of the path)."""
    got = bf16_f64(got_bits)
    assert np.all(np.isfinite(got)), "non-finite output (poison left or overflow)"
    err = np.max(np.abs(got - ref64))
    scale = np.max(np.abs(ref64))
    assert err <= tol * scale, f"max|diff| {err:.4g} > {tol} * max|ref| {scale:.4g}"
    return err / max(scale, 1e-30)


class AGCase:
    """Inputs of one AllGather+GEMM call laid out in a symmetric heap."""

    def __init__(self, inp, b_layout=tdg.B_KN, device="cuda", ll=False, c_f32=False):
        self.inp = inp
        self.c_f32 = c_f32
        W, Ms, K, N = inp.W, inp.Ms, inp.K, inp.N
        self.M = W * Ms
        self.a_off = 0
        self.g_off = align(Ms * K * 2)
        self.ll_off = align(self.g_off + self.M * K * 2)     # LL words (M*K*4 bytes)
        region = align(self.ll_off + (self.M * K * 4 if ll else 0) + 1024)
        nsig = max(1024, self.M)
        self.symm = tdg.Symm(W, region, nsig, device=device)
        for s in range(W):
            self.symm.view(s, self.a_off, (Ms, K), torch.bfloat16).copy_(to_dev_bf16(inp.shards[s]))
        self.b_layout = b_layout
        if b_layout == tdg.B_KN:
            self.B = to_dev_bf16(inp.B)
        else:
            self.B = to_dev_bf16(np.ascontiguousarray(inp.B.T))
        self.C = torch.empty((self.M, N), dtype=torch.float32 if c_f32 else torch.bfloat16, device=device)

    def gathered(self, rank):
        return self.symm.view(rank, self.g_off, (self.M, self.inp.K), torch.bfloat16)

    def ll_words(self, rank):
        n = self.M * self.inp.K // 2
        return self.symm.view(rank, self.ll_off, (n,), torch.int64).cpu().numpy().view(np.uint64)

    def run(self, rank=0, mode="sm", check_status=True, **kw):
        inp = self.inp
        if self.c_f32:
            self.C.view(torch.int32).fill_(0x7FC00001)   # a NaN float32 pattern
        else:
            self.C.view(torch.int16).fill_(POISON)
        self.gathered(rank).view(torch.int16).fill_(POISON)
        side = torch.cuda.Stream() if mode == "ce" else None
        tdg.ag_gemm(self.symm, rank, inp.Ms, inp.K, inp.N, self.a_off, self.g_off, self.B, self.C,
                    mode=mode, b_layout=self.b_layout, side_stream=side, c_f32=self.c_f32, **kw)
        torch.cuda.synchronize()
        st = self.symm.status()
        if check_status:
            assert st["code"] == 0, st
        if self.c_f32:
            return self.C.cpu().numpy(), st      # float32 values
        return to_bits(self.C), st


class RSCase:
    """Inputs of one GEMM+ReduceScatter call laid out in a symmetric heap."""

    def __init__(self, inp, b_layout=tdg.B_KN, device="cuda", f32=False):
        self.inp = inp
        self.f32 = f32           # fp32 partials: the staging area is twice as large
        W, M, K, N = inp.W, inp.M, inp.K, inp.N
        self.Mo = M // W
        self.a_off = 0
        self.b_off = align(M * K * 2)
        self.stage_off = align(self.b_off + K * N * 2)
        self.out_off = align(self.stage_off + tdg.gemm_rs_stage_bytes(W, M, N) * (2 if f32 else 1))
        region = align(self.out_off + self.Mo * N * 2 + 1024)
        n_tiles = (N + 255) // 256
        nsig = max(1024, (self.Mo // 128) * n_tiles * 4)
        self.symm = tdg.Symm(W, region, nsig, device=device)
        self.b_layout = b_layout
        for r in range(W):
            self.symm.view(r, self.a_off, (M, K), torch.bfloat16).copy_(to_dev_bf16(inp.As[r]))
            b = inp.Bs[r] if b_layout == tdg.B_KN else np.ascontiguousarray(inp.Bs[r].T)
            self.symm.view(r, self.b_off, b.shape, torch.bfloat16).copy_(to_dev_bf16(b))

    def out(self, o):
        return self.symm.view(o, self.out_off, (self.Mo, self.inp.N), torch.bfloat16)

    def run(self, mode="sm", check_status=True, **kw):
        inp = self.inp
        for o in range(inp.W):
            self.out(o).view(torch.int16).fill_(POISON)
        kw.setdefault("partial_f32", self.f32)
        tdg.gemm_rs(self.symm, inp.M, inp.K, inp.N, self.a_off, self.b_off, self.stage_off,
                    self.out_off, mode=mode, b_layout=self.b_layout, **kw)
        torch.cuda.synchronize()
        st = self.symm.status()
        if check_status:
            assert st["code"] == 0, st
        return np.stack([to_bits(self.out(o)) for o in range(inp.W)]), st
