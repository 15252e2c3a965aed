"""GPU parity of distributed flash decoding (through the C ABI) against the
oracle's softmax attention over the whole, unsplit KV cache."""
import numpy as np
import pytest
import torch

import oracle
from tile_centric_comm_gb300 import synth, tdg
from gpu_util import align, assert_close, to_bits, to_dev_bf16

pytestmark = pytest.mark.gpu


class FlashCase:
    def __init__(self, W, B, Hq, Hkv, S, chunk=0, seed=0, root=0):
        g = np.random.default_rng(seed)
        D = 128
        self.W, self.B, self.Hq, self.Hkv, self.S, self.D = W, B, Hq, Hkv, S, D
        self.chunk, self.root = chunk, root
        Sr = S // W
        self.q = synth.f32_to_bf16_bits(g.standard_normal((B, Hq, D)).astype(np.float32))
        self.k = synth.f32_to_bf16_bits(g.standard_normal((W, B, Hkv, Sr, D)).astype(np.float32))
        self.v = synth.f32_to_bf16_bits(g.standard_normal((W, B, Hkv, Sr, D)).astype(np.float32))
        kv_bytes = B * Hkv * Sr * D * 2
        self.k_off = 0
        self.v_off = align(kv_bytes)
        self.part_off = align(self.v_off + kv_bytes)
        region = align(self.part_off + tdg.flash_decode_part_bytes(W, B, Hq, D, S, chunk) + 1024)
        self.symm = tdg.Symm(W, region, 4096)
        for r in range(W):
            self.symm.view(r, self.k_off, self.k[r].shape, torch.bfloat16).copy_(to_dev_bf16(self.k[r]))
            self.symm.view(r, self.v_off, self.v[r].shape, torch.bfloat16).copy_(to_dev_bf16(self.v[r]))
        self.qd = to_dev_bf16(self.q)
        self.out = torch.empty((B, Hq, D), dtype=torch.bfloat16, device="cuda")

    def full(self, x):
        # (W, B, Hkv, Sr, D) -> (B, Hkv, S, D): rank r holds tokens [r*Sr, (r+1)*Sr)
        return np.ascontiguousarray(x.transpose(1, 2, 0, 3, 4).reshape(self.B, self.Hkv, self.S, self.D))

    def run(self):
        self.out.view(torch.int16).fill_(0x7FC1)
        tdg.flash_decode(self.symm, self.B, self.Hq, self.Hkv, self.D, self.S, self.k_off, self.v_off,
                         self.part_off, self.qd, self.out, root=self.root, chunk=self.chunk)
        torch.cuda.synchronize()
        assert self.symm.status()["code"] == 0
        return to_bits(self.out)


@pytest.mark.parametrize("W,B,Hq,Hkv,S,chunk", [
    (2, 1, 8, 1, 256, 64),       # G = 8, 2 splits per rank
    (4, 1, 16, 1, 400, 64),      # G = 16, ragged last chunk of every rank (100 = 64 + 36)
    (4, 2, 4, 4, 512, 128),      # G = 1
    (8, 2, 64, 8, 8 * 2048, 0),  # Llama-3-70B head layout, default chunk
])
def test_parity(W, B, Hq, Hkv, S, chunk):
    c = FlashCase(W, B, Hq, Hkv, S, chunk, seed=S + Hq, root=W - 1)
    want = oracle.attention_decode(c.q, c.full(c.k), c.full(c.v))
    for _ in range(2):          # counters reset: a second call gives the same result
        assert_close(c.run(), want)


@pytest.mark.slow
def test_full_size_sampled():
    # 4 sequences x 64 heads (8 kv heads) x 128 Ki cached tokens over 8 ranks
    c = FlashCase(8, 4, 64, 8, 131072, 0, seed=1)
    got = c.run()
    kf, vf = c.full(c.k), c.full(c.v)
    for b in (0, 3):
        want = oracle.attention_decode(c.q[b:b + 1, :16], kf[b:b + 1, :2], vf[b:b + 1, :2])
        assert_close(got[b:b + 1, :16], want)
