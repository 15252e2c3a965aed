"""Pins for the CPU oracle, checked against things other than the oracle itself:
hand-derived golden values (tests/golden/), closed forms, brute force in pure
Python on tiny inputs, library special cases and invariants.  CPU only.

Each pin is chosen so that a plausible slip in the oracle -- a dropped term, a
wrong sign, a shard taken in the wrong order, a transposed operand, an
off-by-one in the scan -- makes at least one of these fail.
"""
import json
import os

import numpy as np
import pytest
import torch

import oracle
from tile_centric_comm_gb300 import synth

GOLD = os.path.join(os.path.dirname(__file__), "golden")


def _gold(name):
    with open(os.path.join(GOLD, name)) as f:
        return json.load(f)


def _bf(x):
    """float values exactly representable in bf16 -> bit patterns."""
    return synth.f32_to_bf16_bits(np.asarray(x, np.float32))


# ------------------------------------------------------------------ bf16 ----
def test_bf16_rounding_golden():
    for c in _gold("bf16_rne.json")["cases"]:
        x = float(c["m"]) * 2.0 ** c["e"]
        assert oracle.f64_to_bf16(np.array([x]))[0] == int(c["bits"], 16), c["note"]
        # sign symmetry
        if x != 0:
            assert oracle.f64_to_bf16(np.array([-x]))[0] == int(c["bits"], 16) ^ 0x8000


def test_bf16_rounding_matches_torch_on_float32_values():
    # special case: for float32 inputs the one-step rounding equals torch's
    # float32 -> bfloat16 cast (round to nearest even)
    g = np.random.default_rng(1)
    x = np.concatenate([
        g.standard_normal(20000).astype(np.float32) * np.float32(1e3),
        g.standard_normal(20000).astype(np.float32) * np.float32(1e-3),
        (g.integers(-2 ** 20, 2 ** 20, 20000) / 64.0).astype(np.float32),
        np.float32(2.0) ** g.integers(-140, 127, 2000).astype(np.float32),
    ])
    want = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    got = oracle.f64_to_bf16(x.astype(np.float64))
    assert np.array_equal(got, want)


def test_bf16_widening_exact():
    h = np.arange(0, 65536, dtype=np.uint32).astype(np.uint16)
    f = oracle.bf16_to_f64(h)
    fin = np.isfinite(f)
    back = oracle.f64_to_bf16(f[fin])
    assert np.array_equal(back, h[fin])


# -------------------------------------------------------------- AG-GEMM ----
def _py_ag_gemm(shards, B):
    """Brute force in pure Python (independent of the C loops)."""
    rows = []
    for a in shards:
        rows.extend(oracle.bf16_to_f64(a).tolist())
    b = oracle.bf16_to_f64(B).tolist()
    K, N = len(b), len(b[0])
    return [[sum(r[k] * b[k][j] for k in range(K)) for j in range(N)] for r in rows]


@pytest.mark.parametrize("dist", ["int2", "normal"])
@pytest.mark.parametrize("W,Ms,K,N", [(2, 3, 5, 4), (3, 2, 7, 5), (1, 4, 3, 6)])
def test_ag_gemm_brute_force(dist, W, Ms, K, N):
    inp = synth.ag_inputs(W, Ms, K, N, dist, seed=W * 100 + K)
    C64, C16 = oracle.ag_gemm(inp.shards, inp.B)
    ref = np.array(_py_ag_gemm(inp.shards, inp.B))
    assert C64.shape == (W * Ms, N)
    assert np.array_equal(C64, ref)
    assert np.array_equal(C16, oracle.f64_to_bf16(ref))


def test_ag_gemm_closed_form_selector_rows():
    # A_s rows are unit vectors: row i of shard s selects row sel[s][i] of B,
    # so C must be those rows of B in shard order (catches shard order and
    # operand transposition; K != N != Ms)
    W, Ms, K, N = 3, 4, 6, 5
    g = np.random.default_rng(7)
    B = _bf(g.integers(-50, 50, (K, N)))
    sel = g.integers(0, K, (W, Ms))
    shards = []
    for s in range(W):
        a = np.zeros((Ms, K), np.float32)
        a[np.arange(Ms), sel[s]] = 1.0
        shards.append(_bf(a))
    C64, C16 = oracle.ag_gemm(shards, B)
    Bf = oracle.bf16_to_f64(B)
    want = np.concatenate([Bf[sel[s]] for s in range(W)])
    assert np.array_equal(C64, want)
    assert np.array_equal(C16, B[sel.reshape(-1)])


def test_ag_gemm_identity_B_gives_gather():
    W, Ms, K = 4, 3, 8
    inp = synth.ag_inputs(W, Ms, K, K, "normal", seed=3)
    I = _bf(np.eye(K))
    _, C16 = oracle.ag_gemm(inp.shards, I)
    assert np.array_equal(C16, np.concatenate(inp.shards))


def test_ag_gemm_sign_and_scaling():
    # negating one shard negates exactly its rows; nothing else moves
    inp = synth.ag_inputs(2, 4, 16, 8, "normal", seed=11)
    C64, _ = oracle.ag_gemm(inp.shards, inp.B)
    neg = [inp.shards[0], inp.shards[1] ^ np.uint16(0x8000)]
    D64, _ = oracle.ag_gemm(neg, inp.B)
    assert np.array_equal(D64[:4], C64[:4])
    assert np.array_equal(D64[4:], -C64[4:])


def test_ag_gemm_sampled_equals_full():
    inp = synth.ag_inputs(2, 16, 32, 24, "normal", seed=5)
    C64, _ = oracle.ag_gemm(inp.shards, inp.B)
    g = np.random.default_rng(0)
    r = g.integers(0, 32, 50)
    c = g.integers(0, 24, 50)
    assert np.array_equal(oracle.ag_gemm_sampled(inp.shards, inp.B, r, c), C64[r, c])


def test_ag_gemm_integer_tiny_workload_is_exact():
    # the integer workload: |partial sums| <= 4 * 256, exact in any float
    inp = synth.make("ag_tiny")
    C64, C16 = oracle.ag_gemm(inp.shards, inp.B)
    assert np.all(C64 == np.round(C64)) and np.abs(C64).max() <= 1024
    assert C64.shape == (128, 128)
    small = np.abs(C64) <= 256          # integers up to 256 are exact in bf16
    assert np.array_equal(oracle.bf16_to_f64(C16)[small], C64[small])


# -------------------------------------------------------------- GEMM-RS ----
def _py_gemm_rs(As, Bs):
    W = len(As)
    M = As[0].shape[0]
    a = [oracle.bf16_to_f64(x).tolist() for x in As]
    b = [oracle.bf16_to_f64(x).tolist() for x in Bs]
    K, N = len(b[0]), len(b[0][0])
    full = [[sum(sum(a[r][i][k] * b[r][k][j] for k in range(K)) for r in range(W))
             for j in range(N)] for i in range(M)]
    return np.array(full).reshape(W, M // W, N)


@pytest.mark.parametrize("dist", ["int2", "normal"])
@pytest.mark.parametrize("W,M,K,N", [(2, 4, 3, 5), (4, 8, 5, 3)])
def test_gemm_rs_brute_force(dist, W, M, K, N):
    inp = synth.rs_inputs(W, M, K, N, dist, seed=M + K)
    out64, out16 = oracle.gemm_rs(inp.As, inp.Bs)
    ref = _py_gemm_rs(inp.As, inp.Bs)
    assert out64.shape == (W, M // W, N)
    np.testing.assert_allclose(out64, ref, rtol=1e-13, atol=1e-13)
    if dist == "int2":
        assert np.array_equal(out64, ref)


def test_gemm_rs_equals_full_k_gemm_row_scattered():
    # invariant: sum_r A_r B_r = [A_0 | ... | A_{W-1}] @ [B_0; ...; B_{W-1}]
    W, M, K, N = 4, 8, 6, 5
    inp = synth.rs_inputs(W, M, K, N, "int2", seed=2)
    out64, out16 = oracle.gemm_rs(inp.As, inp.Bs)
    Acat = np.concatenate(inp.As, axis=1)         # M x W*K
    Bcat = np.concatenate(inp.Bs, axis=0)         # W*K x N
    C64, C16 = oracle.ag_gemm([Acat], Bcat)       # one shard: plain GEMM
    assert np.array_equal(out64.reshape(M, N), C64)
    assert np.array_equal(out16.reshape(M, N), C16)


def test_gemm_rs_is_sum_of_partials_and_owner_rows():
    W, M, K, N = 2, 6, 4, 3
    inp = synth.rs_inputs(W, M, K, N, "normal", seed=9)
    out64, _ = oracle.gemm_rs(inp.As, inp.Bs)
    P = [oracle.gemm_partial(a, b) for a, b in zip(inp.As, inp.Bs)]
    full = P[0] + P[1]
    np.testing.assert_allclose(out64[0], full[:3], rtol=1e-14, atol=1e-15)
    np.testing.assert_allclose(out64[1], full[3:], rtol=1e-14, atol=1e-15)


def test_gemm_rs_closed_form_scaled_identity():
    # A_r = c_r * I  =>  out = sum_r c_r * B_r, split by rows
    W, M = 4, 8
    c = [1.0, -2.0, 0.5, 3.0]
    g = np.random.default_rng(4)
    As = [_bf(np.eye(M) * c[r]) for r in range(W)]
    Bs = [_bf(g.integers(-8, 9, (M, 5))) for _ in range(W)]
    out64, _ = oracle.gemm_rs(As, Bs)
    want = sum(c[r] * oracle.bf16_to_f64(Bs[r]) for r in range(W))
    assert np.array_equal(out64.reshape(M, 5), want)


def test_gemm_rs_sampled_equals_full():
    inp = synth.rs_inputs(2, 8, 5, 7, "normal", seed=1)
    out64, _ = oracle.gemm_rs(inp.As, inp.Bs)
    r = np.array([0, 3, 4, 7, 5])
    cc = np.array([6, 0, 2, 3, 1])
    got = oracle.gemm_rs_sampled(inp.As, inp.Bs, r, cc)
    np.testing.assert_array_equal(got, out64.reshape(8, 7)[r, cc])
