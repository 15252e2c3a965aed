"""CPU oracle for the tile-centric AG-GEMM / GEMM-RS / MoE path.

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and
``bench.py``'s CPU-baseline leg (and its ``--impl reference`` arm) import this
package.  The product library under ``tile_centric_comm_gb300/`` never imports
it and shares no code with it.

The arithmetic lives in ``tdg_oracle.c`` (plain C, double precision, explicit
loops, each function citing the published passage it writes out).  This
module only compiles it with gcc and marshals numpy arrays through ctypes.

bf16 values travel as numpy ``uint16`` bit patterns.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "tdg_oracle.c")
_BUILD = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD, "libtdg_oracle.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile the oracle with gcc (OpenMP when available); returns the path."""
    os.makedirs(_BUILD, exist_ok=True)
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    base = ["gcc", "-O2", "-std=c11", "-shared", "-fPIC", "-o", tmp, _SRC, "-lm"]
    try:
        subprocess.run(base[:1] + ["-fopenmp"] + base[1:], check=True,
                       capture_output=True)
    except subprocess.CalledProcessError:
        subprocess.run(base, check=True, capture_output=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _L():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            i64, i32, vp = ctypes.c_int64, ctypes.c_int, ctypes.c_void_p
            lib.orc_bf16_to_f64.restype = ctypes.c_double
            lib.orc_bf16_to_f64.argtypes = [ctypes.c_uint16]
            lib.orc_f64_to_bf16.restype = ctypes.c_uint16
            lib.orc_f64_to_bf16.argtypes = [ctypes.c_double]
            lib.orc_f64_to_bf16_array.argtypes = [vp, vp, i64]
            lib.orc_ag_gemm.argtypes = [i32, i64, i64, i64, vp, vp, vp, vp]
            lib.orc_ag_gemm_sampled.argtypes = [i32, i64, i64, i64, vp, vp, i64,
                                                vp, vp, vp]
            lib.orc_gemm_rs.argtypes = [i32, i64, i64, i64, vp, vp, vp, vp]
            lib.orc_gemm_rs_sampled.argtypes = [i32, i64, i64, i64, vp, vp, i64,
                                                vp, vp, vp]
            lib.orc_gemm_partial.argtypes = [i64, i64, i64, vp, vp, vp]
            lib.orc_moe_route.restype = ctypes.c_int
            lib.orc_moe_route.argtypes = [i32, i64, i32, i32, vp, vp, vp, vp, vp,
                                          vp, vp, vp]
            lib.orc_moe_dispatch.argtypes = [i32, i64, i32, i64, vp, vp, vp]
            lib.orc_moe_combine.argtypes = [i32, i64, i32, i64, vp, vp, vp, vp,
                                            vp]
            lib.orc_ll_pack.argtypes = [vp, i64, ctypes.c_uint32, vp]
            lib.orc_ll_unpack.restype = ctypes.c_int64
            lib.orc_ll_unpack.argtypes = [vp, i64, ctypes.c_uint32, vp]
            lib.orc_swizzle_order.argtypes = [i32, i64, i64, i64, vp, vp]
            lib.orc_allreduce.argtypes = [i32, i64, vp, vp]
            lib.orc_attention_decode.argtypes = [i64, i64, i64, i64, i64, vp, vp, vp,
                                                 ctypes.c_double, vp]
            _lib = lib
    return _lib


def _p(a: np.ndarray):
    assert a.flags["C_CONTIGUOUS"], "oracle arrays must be C-contiguous"
    return ctypes.c_void_p(a.ctypes.data)


def _ptr_array(arrs):
    return (ctypes.c_void_p * len(arrs))(*[a.ctypes.data for a in arrs])


def _u16(a):
    a = np.ascontiguousarray(a)
    assert a.dtype == np.uint16, "bf16 arrays travel as uint16 bit patterns"
    return a


# ----------------------------------------------------------------- bf16 ----
def bf16_to_f64(h: np.ndarray) -> np.ndarray:
    """Exact widening of bf16 bit patterns (uint16) to float64."""
    h = np.ascontiguousarray(h, dtype=np.uint16)
    with np.errstate(invalid="ignore"):
        return (h.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def f64_to_bf16(x) -> np.ndarray:
    """Round float64 values once to bf16 (nearest, ties to even)."""
    x = np.ascontiguousarray(x, dtype=np.float64)
    out = np.empty(x.shape, dtype=np.uint16)
    _L().orc_f64_to_bf16_array(_p(x), _p(out), x.size)
    return out


# -------------------------------------------------------------- AG-GEMM ----
def ag_gemm(shards, B):
    """C = concat_rows(shards) @ B; returns (C64 float64, C16 bf16 bits)."""
    shards = [_u16(a) for a in shards]
    B = _u16(B)
    W = len(shards)
    Ms, K = shards[0].shape
    K2, N = B.shape
    assert K == K2 and all(a.shape == (Ms, K) for a in shards)
    C64 = np.empty((W * Ms, N), np.float64)
    C16 = np.empty((W * Ms, N), np.uint16)
    _L().orc_ag_gemm(W, Ms, K, N, _ptr_array(shards), _p(B), _p(C64), _p(C16))
    return C64, C16


def ag_gemm_sampled(shards, B, rows, cols):
    """C64 at the given (row, col) positions only."""
    shards = [_u16(a) for a in shards]
    B = _u16(B)
    Ms, K = shards[0].shape
    N = B.shape[1]
    rows = np.ascontiguousarray(rows, np.int64)
    cols = np.ascontiguousarray(cols, np.int64)
    out = np.empty(rows.shape, np.float64)
    _L().orc_ag_gemm_sampled(len(shards), Ms, K, N, _ptr_array(shards), _p(B),
                             rows.size, _p(rows), _p(cols), _p(out))
    return out


# -------------------------------------------------------------- GEMM-RS ----
def gemm_rs(As, Bs):
    """Owner-major (W, M/W, N) result of rows-scatter(sum_r As[r] @ Bs[r])."""
    As = [_u16(a) for a in As]
    Bs = [_u16(b) for b in Bs]
    W = len(As)
    M, K = As[0].shape
    N = Bs[0].shape[1]
    assert M % W == 0
    out64 = np.empty((W, M // W, N), np.float64)
    out16 = np.empty((W, M // W, N), np.uint16)
    _L().orc_gemm_rs(W, M, K, N, _ptr_array(As), _ptr_array(Bs), _p(out64),
                     _p(out16))
    return out64, out16


def gemm_rs_sampled(As, Bs, rows, cols):
    As = [_u16(a) for a in As]
    Bs = [_u16(b) for b in Bs]
    M, K = As[0].shape
    N = Bs[0].shape[1]
    rows = np.ascontiguousarray(rows, np.int64)
    cols = np.ascontiguousarray(cols, np.int64)
    out = np.empty(rows.shape, np.float64)
    _L().orc_gemm_rs_sampled(len(As), M, K, N, _ptr_array(As), _ptr_array(Bs),
                             rows.size, _p(rows), _p(cols), _p(out))
    return out


def gemm_partial(A, B):
    A, B = _u16(A), _u16(B)
    M, K = A.shape
    N = B.shape[1]
    P = np.empty((M, N), np.float64)
    _L().orc_gemm_partial(M, K, N, _p(A), _p(B), _p(P))
    return P


# ------------------------------------------------------------------ MoE ----
def moe_route(topk: np.ndarray, n_experts: int):
    """Routing metadata.  topk: (W, T, k) int32.  Returns a dict of arrays."""
    topk = np.ascontiguousarray(topk, np.int32)
    W, T, KK = topk.shape
    E = int(n_experts)
    counts = np.zeros((W, E), np.int64)
    base = np.zeros(E + 1, np.int64)
    off = np.zeros((W, E), np.int64)
    slot = np.zeros((W, T, KK), np.int64)
    total = W * T * KK
    row_src = np.full(total, -1, np.int32)
    row_tok = np.full(total, -1, np.int32)
    row_k = np.full(total, -1, np.int32)
    rc = _L().orc_moe_route(W, T, KK, E, _p(topk), _p(counts), _p(base), _p(off),
                            _p(slot), _p(row_src), _p(row_tok), _p(row_k))
    if rc != 0:
        raise ValueError(f"orc_moe_route failed ({rc}): expert id out of range")
    return dict(counts=counts, base=base, off=off, slot=slot, row_src=row_src,
                row_tok=row_tok, row_k=row_k)


def moe_dispatch(x: np.ndarray, slot: np.ndarray, total_rows: int):
    """recv[slot(src,t,k)] = x[src][t]; x: (W, T, H) bf16 bits."""
    x = _u16(x)
    slot = np.ascontiguousarray(slot, np.int64)
    W, T, H = x.shape
    KK = slot.shape[2]
    recv = np.zeros((total_rows, H), np.uint16)
    _L().orc_moe_dispatch(W, T, KK, H, _p(x), _p(slot), _p(recv))
    return recv


def moe_combine(y: np.ndarray, slot: np.ndarray, gate: np.ndarray):
    """out[src][t] = bf16(sum_k gate*y[slot]); returns (out16, out64)."""
    y = _u16(y)
    slot = np.ascontiguousarray(slot, np.int64)
    gate = np.ascontiguousarray(gate, np.float32)
    W, T, KK = slot.shape
    H = y.shape[1]
    out16 = np.empty((W, T, H), np.uint16)
    out64 = np.empty((W, T, H), np.float64)
    _L().orc_moe_combine(W, T, KK, H, _p(y), _p(slot), _p(gate), _p(out16),
                         _p(out64))
    return out16, out64


# ------------------------------------------------------------ LL / order ----
def ll_pack(payload: np.ndarray, flag: int) -> np.ndarray:
    payload = np.ascontiguousarray(payload, np.uint32)
    words = np.empty(payload.shape, np.uint64)
    _L().orc_ll_pack(_p(payload), payload.size, flag, _p(words))
    return words


def ll_unpack(words: np.ndarray, flag: int):
    """Returns (payload, number of words whose flag did not match)."""
    words = np.ascontiguousarray(words, np.uint64)
    payload = np.zeros(words.shape, np.uint32)
    missing = _L().orc_ll_unpack(_p(words), words.size, flag, _p(payload))
    return payload, int(missing)


def swizzle_order(rank: int, tiles_per_pe: int, total_m: int, n_tiles: int):
    pm = np.empty(total_m * n_tiles, np.int64)
    pn = np.empty(total_m * n_tiles, np.int64)
    _L().orc_swizzle_order(rank, tiles_per_pe, total_m, n_tiles, _p(pm), _p(pn))
    return pm, pn


# ------------------------------------------------------------- AllReduce ----
def allreduce(xs):
    """Element-wise sum (float64) of W float32 buffers of equal length."""
    xs = [np.ascontiguousarray(x, np.float32).reshape(-1) for x in xs]
    n = xs[0].size
    assert all(x.size == n for x in xs)
    out = np.empty(n, np.float64)
    _L().orc_allreduce(len(xs), n, _ptr_array(xs), _p(out))
    return out


# ------------------------------------------------------ decode attention ----
def attention_decode(q, k, v, scale=None):
    """Softmax attention of one query token per (batch, head) over the whole
    KV cache.  q: (B, Hq, D); k, v: (B, Hkv, S, D) bf16 bits.  Returns float64
    (B, Hq, D)."""
    q, k, v = _u16(q), _u16(k), _u16(v)
    B, Hq, D = q.shape
    _, Hkv, S, _ = k.shape
    assert Hq % Hkv == 0 and k.shape == v.shape == (B, Hkv, S, D)
    if scale is None:
        scale = 1.0 / np.sqrt(D)
    out = np.empty((B, Hq, D), np.float64)
    _L().orc_attention_decode(B, Hq, Hkv, D, S, _p(q), _p(k), _p(v), float(scale), _p(out))
    return out
