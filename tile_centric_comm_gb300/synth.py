"""Seeded synthetic inputs shared by the CUDA path's tests, the oracle's tests
and the benchmark.

This module draws random numbers and converts them to bf16; it holds none of
the method's arithmetic (no GEMM, no gather, no scan, no reduction).  Both the
oracle and the CUDA library receive the bytes it produces.

Recipe (numpy ``Generator(PCG64(seed))``, seed 0 unless stated):
  * "normal"  : ``standard_normal(float32) * std`` in float32, then bf16 by
                round-to-nearest-even (torch's float32 -> bfloat16 cast).
  * "int2"    : integers uniform in {-2, -1, 0, 1, 2} (each 1/5), exact in bf16.
                (`device_int2` draws the same distribution on the device with
                torch's generator, for inputs too large for the host.)
  * Tensors are drawn in the order the workload lists them: AG-GEMM draws
    A_0 .. A_{W-1} then B; GEMM-RS draws A_0, B_0, A_1, B_1, ...; MoE draws x,
    then the routing noise, then the gate logits.
  * MoE routing: expert popularity p_e proportional to (e+1)^-s (Zipf, s=1.2,
    expert 0 most popular); each token picks top-k distinct experts by
    Gumbel-top-k (key = log p_e + Gumbel noise, k largest keys in descending
    key order).  Gate weights are the float32 softmax of k N(0,1) logits.

bf16 arrays are returned as numpy ``uint16`` bit patterns.
"""
from __future__ import annotations

from dataclasses import dataclass

import numpy as np
import torch


def rng(seed: int = 0) -> np.random.Generator:
    return np.random.Generator(np.random.PCG64(seed))


def f32_to_bf16_bits(a: np.ndarray) -> np.ndarray:
    """float32 -> bf16 bit patterns, round to nearest even (torch's cast)."""
    t = torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32))
    return t.to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


def bf16_bits_to_f32(h: np.ndarray) -> np.ndarray:
    return (np.ascontiguousarray(h, np.uint16).astype(np.uint32) << 16).view(np.float32)


def draw(g: np.random.Generator, shape, dist: str, std: float = 1.0) -> np.ndarray:
    if dist == "int2":
        return f32_to_bf16_bits(g.integers(-2, 3, size=shape).astype(np.float32))
    if dist == "normal":
        x = g.standard_normal(size=shape, dtype=np.float32)
        if std != 1.0:
            x *= np.float32(std)
        return f32_to_bf16_bits(x)
    raise ValueError(f"unknown distribution {dist!r}")


def device_int2(shape, seed: int, device="cuda") -> torch.Tensor:
    """bf16 integers uniform in {-2..2} drawn on the device by torch's seeded
    generator (for inputs too large to draw and hold on the host)."""
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    return torch.randint(-2, 3, shape, generator=g, device=device, dtype=torch.int8).to(torch.bfloat16)


# ------------------------------------------------------------------ AG ----
@dataclass
class AGInputs:
    shards: list          # W arrays (Ms, K) bf16 bits
    B: np.ndarray         # (K, N) bf16 bits
    W: int
    Ms: int
    K: int
    N: int


def ag_inputs(W: int, Ms: int, K: int, N: int, dist: str = "normal",
              seed: int = 0, b_std: float = 0.02) -> AGInputs:
    g = rng(seed)
    shards = [draw(g, (Ms, K), dist) for _ in range(W)]
    B = draw(g, (K, N), dist, 1.0 if dist == "int2" else b_std)
    return AGInputs(shards, B, W, Ms, K, N)


@dataclass
class AGAllInputs:
    shards: list          # W arrays (Ms, K)
    Bs: list              # W arrays (K, N): rank r's weight shard
    W: int
    Ms: int
    K: int
    N: int


def ag_all_inputs(W: int, Ms: int, K: int, N: int, dist: str = "normal",
                  seed: int = 0, b_std: float = 0.02) -> AGAllInputs:
    """Inputs of the AllGather+GEMM of every rank: the W shards, then W weight
    shards B_r, drawn in that order."""
    g = rng(seed)
    shards = [draw(g, (Ms, K), dist) for _ in range(W)]
    Bs = [draw(g, (K, N), dist, 1.0 if dist == "int2" else b_std) for _ in range(W)]
    return AGAllInputs(shards, Bs, W, Ms, K, N)


# ------------------------------------------------------------------ RS ----
@dataclass
class RSInputs:
    As: list              # W arrays (M, K)
    Bs: list              # W arrays (K, N)
    W: int
    M: int
    K: int
    N: int


def rs_inputs(W: int, M: int, K: int, N: int, dist: str = "normal",
              seed: int = 0, b_std: float = 0.02) -> RSInputs:
    g = rng(seed)
    As, Bs = [], []
    for _ in range(W):
        As.append(draw(g, (M, K), dist))
        Bs.append(draw(g, (K, N), dist, 1.0 if dist == "int2" else b_std))
    return RSInputs(As, Bs, W, M, K, N)


# ----------------------------------------------------------------- MoE ----
@dataclass
class MoEInputs:
    x: np.ndarray         # (W, T, H) bf16 bits
    topk: np.ndarray      # (W, T, k) int32 expert ids
    gate: np.ndarray      # (W, T, k) float32, rows sum to ~1
    W: int
    T: int
    H: int
    E: int
    k: int


def zipf_popularity(E: int, s: float = 1.2) -> np.ndarray:
    p = (np.arange(1, E + 1, dtype=np.float64)) ** (-s)
    return p / p.sum()


def moe_inputs(W: int, T: int, H: int, E: int = 256, k: int = 8,
               zipf_s: float = 1.2, seed: int = 0, x_dist: str = "normal",
               top1_unit: bool = False) -> MoEInputs:
    """top1_unit=True keeps only the first routed expert with gate 1.0 (the
    degenerate top-1 case used to check that dispatch+combine is the identity)."""
    g = rng(seed)
    x = draw(g, (W, T, H), x_dist)
    logp = np.log(zipf_popularity(E, zipf_s))
    topk = np.empty((W, T, k), np.int32)
    chunk = 4096
    for src in range(W):
        for t0 in range(0, T, chunk):
            t1 = min(T, t0 + chunk)
            keys = logp[None, :] + g.gumbel(size=(t1 - t0, E))
            order = np.argsort(-keys, axis=1, kind="stable")[:, :k]
            topk[src, t0:t1] = order.astype(np.int32)
    logits = g.standard_normal(size=(W, T, k), dtype=np.float32)
    ex = np.exp(logits - logits.max(axis=-1, keepdims=True))
    gate = (ex / ex.sum(axis=-1, keepdims=True)).astype(np.float32)
    if top1_unit:
        topk = np.ascontiguousarray(topk[:, :, :1])
        gate = np.ones((W, T, 1), np.float32)
        k = 1
    return MoEInputs(x, topk, gate, W, T, H, E, k)


# ------------------------------------------------------- named workloads ----
WORKLOADS = {
    # AllGather+GEMM, W=2, A_r 64x256, B 256x128, integers in [-2, 2]
    "ag_tiny": dict(kind="ag", W=2, Ms=64, K=256, N=128, dist="int2"),
    # AllGather+GEMM at the Qwen-32B MLP up-projection shape
    "ag_qwen32b_up": dict(kind="ag", W=8, Ms=1024, K=5120, N=3200, dist="normal"),
    # GEMM+ReduceScatter at the Qwen-32B MLP down-projection shape
    "rs_qwen32b_down": dict(kind="rs", W=8, M=8192, K=3200, N=5120, dist="normal"),
    # AllGather+GEMM at the Llama-3-70B fused gate+up shape
    "ag_llama70b_gateup": dict(kind="ag", W=8, Ms=2048, K=8192, N=7168, dist="normal"),
    # MoE dispatch+combine, 8 ranks x 4096 tokens, hidden 7168, 256 experts, top-8
    "moe_8x4096_h7168_e256_top8": dict(kind="moe", W=8, T=4096, H=7168, E=256, k=8),
}


def make(name: str, seed: int = 0):
    w = dict(WORKLOADS[name])
    kind = w.pop("kind")
    if kind == "ag":
        return ag_inputs(w["W"], w["Ms"], w["K"], w["N"], w["dist"], seed)
    if kind == "rs":
        return rs_inputs(w["W"], w["M"], w["K"], w["N"], w["dist"], seed)
    return moe_inputs(w["W"], w["T"], w["H"], w["E"], w["k"], seed=seed)
