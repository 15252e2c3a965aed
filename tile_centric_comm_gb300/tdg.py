"""Thin ctypes binding of libtdg (include/tdg.h).  Argument marshalling only:
every step of the path runs in the library's CUDA kernels.  PyTorch supplies
device memory and streams.

The library must have been built (``python -m tile_centric_comm_gb300.build``
or ``__graft_entry__.build()``); when it is missing every call raises -- there
is no fallback.
"""
from __future__ import annotations

import ctypes
import os
import threading

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "_build", "libtdg.so")

TDG_OK = 0
TDG_ERR_INVALID = -1
TDG_ERR_CUDA = -2
TDG_ERR_NOMEM = -3
TDG_ERR_TIMEOUT = -4
TDG_ERR_UNSUPPORTED = -5
TDG_ERR_DEVICE = -6

MODE_SM, MODE_CE, MODE_LL, MODE_SERIAL = 0, 1, 2, 3
MODES = {"sm": MODE_SM, "ce": MODE_CE, "ll": MODE_LL, "serial": MODE_SERIAL}
B_KN, B_NK = 0, 1
MOE_ROUTE, MOE_DISPATCH, MOE_COMBINE, MOE_ALL = 1, 2, 4, 7
WHERE = {1: "ag_flag", 2: "pipe", 3: "ll", 4: "moe_expert", 5: "ring", 6: "rs_signal"}

# every symbol include/tdg.h declares
EXPORTS = [
    "tdg_symm_bytes", "tdg_symm_alloc", "tdg_symm_free", "tdg_symm_region", "tdg_symm_at",
    "tdg_symm_flags", "tdg_symm_counters", "tdg_symm_epoch", "tdg_status", "tdg_strerror",
    "tdg_device_info", "tdg_ag_gemm", "tdg_ag_gemm_all_ranks", "tdg_gemm_rs_stage_bytes", "tdg_gemm_rs",
    "tdg_moe_workspace_bytes", "tdg_moe_dispatch_combine", "tdg_moe_dispatch_combine_noalloc",
    "tdg_allreduce_recv_bytes", "tdg_allreduce", "tdg_flash_decode_part_bytes", "tdg_flash_decode",
]
MOE_STATIC_WORKSPACE_BYTES = 2 * 1024 * 1024

_i32, _i64, _u32, _u64 = ctypes.c_int32, ctypes.c_int64, ctypes.c_uint32, ctypes.c_uint64
_sz, _vp = ctypes.c_size_t, ctypes.c_void_p


class TdgFault(ctypes.Structure):
    _fields_ = [("code", _i32), ("where", _u32), ("index", _u32), ("epoch", _u32)]


class AgGemmArgs(ctypes.Structure):
    _fields_ = [("world", ctypes.c_int), ("rank", ctypes.c_int), ("Ms", _i64), ("K", _i64),
                ("N", _i64), ("a_off", _sz), ("g_off", _sz), ("B", _vp), ("C", _vp),
                ("b_layout", ctypes.c_int), ("mode", ctypes.c_int), ("producers", ctypes.c_int),
                ("signal_rows", _i64), ("swizzle", ctypes.c_int), ("timeout_ns", _u64),
                ("ll_off", _sz), ("test_skip_notify", _u64), ("source_order", ctypes.c_int),
                ("c_f32", ctypes.c_int), ("cluster", ctypes.c_int), ("stages", ctypes.c_int),
                ("split_tail", ctypes.c_int), ("producer_items", ctypes.c_int),
                ("producer_warps", ctypes.c_int), ("producer_chunk", ctypes.c_int),
                ("push", ctypes.c_int)]


class AgGemmAllArgs(ctypes.Structure):
    _fields_ = [("world", ctypes.c_int), ("Ms", _i64), ("K", _i64), ("N", _i64), ("a_off", _sz),
                ("g_off", _sz), ("b_off", _sz), ("c_off", _sz), ("b_layout", ctypes.c_int),
                ("mode", ctypes.c_int), ("signal_rows", _i64), ("timeout_ns", _u64),
                ("test_skip_notify", _u64), ("c_f32", ctypes.c_int), ("cluster", ctypes.c_int),
                ("stages", ctypes.c_int), ("push", ctypes.c_int)]


class GemmRsArgs(ctypes.Structure):
    _fields_ = [("world", ctypes.c_int), ("M", _i64), ("K", _i64), ("N", _i64), ("a_off", _sz),
                ("b_off", _sz), ("stage_off", _sz), ("out_off", _sz), ("b_layout", ctypes.c_int),
                ("mode", ctypes.c_int), ("timeout_ns", _u64), ("owner_block", ctypes.c_int),
                ("partial_f32", ctypes.c_int), ("cluster", ctypes.c_int), ("stages", ctypes.c_int),
                ("order", ctypes.c_int), ("red_rows", ctypes.c_int), ("spare", ctypes.c_int)]


class MoeArgs(ctypes.Structure):
    _fields_ = [("world", ctypes.c_int), ("T", _i64), ("H", _i64), ("E", ctypes.c_int),
                ("k", ctypes.c_int), ("x_off", _sz), ("topk_off", _sz), ("gate_off", _sz),
                ("out_off", _sz), ("recv", _vp), ("y", _vp), ("counts", _vp), ("base", _vp),
                ("slot", _vp), ("row_src", _vp), ("row_tok", _vp), ("row_k", _vp),
                ("workspace", _vp), ("workspace_bytes", _sz), ("phases", ctypes.c_int)]


class AllReduceArgs(ctypes.Structure):
    _fields_ = [("world", ctypes.c_int), ("count", _i64), ("x_off", _sz), ("recv_off", _sz),
                ("tile_elems", _i64), ("ctas_per_rank", ctypes.c_int), ("timeout_ns", _u64),
                ("test_skip_signal", _u64)]


class FlashDecodeArgs(ctypes.Structure):
    _fields_ = [("world", ctypes.c_int), ("root", ctypes.c_int), ("B", _i64), ("Hq", _i64),
                ("Hkv", _i64), ("D", _i64), ("S", _i64), ("k_off", _sz), ("v_off", _sz),
                ("part_off", _sz), ("q", _vp), ("out", _vp), ("chunk", _i64),
                ("scale", ctypes.c_float)]


class TdgError(RuntimeError):
    def __init__(self, code, what):
        self.code = code
        super().__init__(f"{what}: {strerror(code)} ({code})")


_lib = None
_lock = threading.Lock()


def lib():
    """Open libtdg.so (raises if it has not been built)."""
    global _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(LIB_PATH):
                raise RuntimeError(
                    f"libtdg.so not found at {LIB_PATH}: build it with "
                    "`python -m tile_centric_comm_gb300.build` (there is no CPU fallback)")
            L = ctypes.CDLL(LIB_PATH)
            L.tdg_symm_bytes.restype = _sz
            L.tdg_symm_bytes.argtypes = [ctypes.c_int, _sz, _sz]
            L.tdg_symm_alloc.restype = ctypes.c_int
            L.tdg_symm_alloc.argtypes = [_vp, _sz, ctypes.c_int, _sz, _sz, ctypes.POINTER(_vp)]
            L.tdg_symm_free.restype = ctypes.c_int
            L.tdg_symm_free.argtypes = [_vp]
            for n in ("tdg_symm_region", "tdg_symm_flags", "tdg_symm_counters"):
                getattr(L, n).restype = _vp
                getattr(L, n).argtypes = [_vp, ctypes.c_int]
            L.tdg_symm_at.restype = _vp
            L.tdg_symm_at.argtypes = [_vp, _vp, ctypes.c_int]
            L.tdg_symm_epoch.restype = _u32
            L.tdg_symm_epoch.argtypes = [_vp]
            L.tdg_status.restype = ctypes.c_int
            L.tdg_status.argtypes = [_vp, _vp, ctypes.POINTER(TdgFault), ctypes.c_int]
            L.tdg_strerror.restype = ctypes.c_char_p
            L.tdg_strerror.argtypes = [ctypes.c_int]
            L.tdg_device_info.restype = ctypes.c_int
            L.tdg_device_info.argtypes = [ctypes.POINTER(ctypes.c_int), ctypes.POINTER(ctypes.c_int)]
            L.tdg_ag_gemm.restype = ctypes.c_int
            L.tdg_ag_gemm.argtypes = [_vp, ctypes.POINTER(AgGemmArgs), _vp, _vp]
            L.tdg_ag_gemm_all_ranks.restype = ctypes.c_int
            L.tdg_ag_gemm_all_ranks.argtypes = [_vp, ctypes.POINTER(AgGemmAllArgs), _vp, _vp]
            L.tdg_gemm_rs_stage_bytes.restype = _sz
            L.tdg_gemm_rs_stage_bytes.argtypes = [ctypes.c_int, _i64, _i64]
            L.tdg_gemm_rs.restype = ctypes.c_int
            L.tdg_gemm_rs.argtypes = [_vp, ctypes.POINTER(GemmRsArgs), _vp]
            L.tdg_moe_workspace_bytes.restype = _sz
            L.tdg_moe_workspace_bytes.argtypes = [ctypes.c_int, _i64, ctypes.c_int]
            L.tdg_moe_dispatch_combine.restype = ctypes.c_int
            L.tdg_moe_dispatch_combine.argtypes = [_vp, ctypes.POINTER(MoeArgs), _vp]
            L.tdg_allreduce_recv_bytes.restype = _sz
            L.tdg_allreduce_recv_bytes.argtypes = [ctypes.c_int, _i64]
            L.tdg_allreduce.restype = ctypes.c_int
            L.tdg_allreduce.argtypes = [_vp, ctypes.POINTER(AllReduceArgs), _vp]
            L.tdg_flash_decode_part_bytes.restype = _sz
            L.tdg_flash_decode_part_bytes.argtypes = [ctypes.c_int, _i64, _i64, _i64, _i64, _i64]
            L.tdg_flash_decode.restype = ctypes.c_int
            L.tdg_flash_decode.argtypes = [_vp, ctypes.POINTER(FlashDecodeArgs), _vp]
            L.tdg_moe_dispatch_combine_noalloc.restype = ctypes.c_int
            L.tdg_moe_dispatch_combine_noalloc.argtypes = [_vp, ctypes.POINTER(MoeArgs), _vp]
            _lib = L
    return _lib


def strerror(code: int) -> str:
    return lib().tdg_strerror(code).decode()


def _check(rc, what):
    if rc != TDG_OK:
        raise TdgError(rc, what)


def _tensor(t, name, dtype, numel, device=None):
    """Check a tensor handed to the library as a raw pointer: the library sees
    neither strides nor dtype, so it must be a contiguous CUDA tensor of the
    documented element type holding at least `numel` elements."""
    import torch
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name}: expected a torch.Tensor, got {type(t).__name__}")
    if t.dtype != dtype:
        raise TypeError(f"{name}: expected {dtype}, got {t.dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{name}: must be contiguous (the library reads it row-major)")
    if t.numel() < numel:
        raise ValueError(f"{name}: holds {t.numel()} elements, needs {numel}")
    if not t.is_cuda:
        raise ValueError(f"{name}: must be a CUDA tensor")
    if device is not None and t.device != device:
        raise ValueError(f"{name}: on {t.device}, the heap is on {device}")
    return t.data_ptr()


def _stream(stream):
    import torch
    if stream is None:
        stream = torch.cuda.current_stream()
    return _vp(stream.cuda_stream)


def device_info():
    sms, sup = ctypes.c_int(0), ctypes.c_int(0)
    _check(lib().tdg_device_info(ctypes.byref(sms), ctypes.byref(sup)), "tdg_device_info")
    return sms.value, bool(sup.value)


class Symm:
    """A symmetric heap of `world` regions carved from one torch allocation."""

    def __init__(self, world: int, region_bytes: int, signals_per_rank: int = 65536,
                 device=None, buffer=None):
        import torch
        region_bytes = (int(region_bytes) + 1023) // 1024 * 1024
        L = lib()
        nbytes = L.tdg_symm_bytes(world, region_bytes, signals_per_rank)
        if buffer is None:
            buffer = torch.empty(nbytes + 1024, dtype=torch.uint8, device=device or "cuda")
        _tensor(buffer, "buffer", torch.uint8, nbytes + 1024)
        self.buf = buffer
        self.base_off = (-buffer.data_ptr()) % 1024
        self.base = buffer.data_ptr() + self.base_off
        self.nbytes = nbytes
        self.world = world
        self.region_bytes = region_bytes
        self.nsig = signals_per_rank
        h = _vp()
        _check(L.tdg_symm_alloc(_vp(self.base), nbytes, world, region_bytes, signals_per_rank,
                                ctypes.byref(h)), "tdg_symm_alloc")
        self.h = h

    def close(self):
        if getattr(self, "h", None):
            lib().tdg_symm_free(self.h)
            self.h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def region_ptr(self, rank: int) -> int:
        return lib().tdg_symm_region(self.h, rank)

    def view(self, rank: int, off: int, shape, dtype):
        """A tensor over region `rank` at byte offset `off`."""
        import torch
        n = 1
        for d in shape:
            n *= int(d)
        esz = torch.empty((), dtype=dtype).element_size()
        if not 0 <= rank < self.world:
            raise ValueError(f"rank {rank} outside [0, {self.world})")
        if off < 0 or off % esz or off + n * esz > self.region_bytes:
            raise ValueError(f"view of {n * esz} bytes at offset {off} does not fit a "
                             f"{self.region_bytes}-byte region with {esz}-byte alignment")
        start = self.base_off + rank * self.region_bytes + off
        return self.buf[start:start + n * esz].view(dtype).view(*shape)

    def flags(self, rank: int, n: int):
        import torch
        if not 0 <= rank < self.world or not 0 <= n <= self.nsig:
            raise ValueError(f"flags({rank}, {n}) outside {self.world} ranks x {self.nsig} words")
        start = lib().tdg_symm_flags(self.h, rank) - self.buf.data_ptr()
        return self.buf[start:start + 4 * n].view(torch.int32)

    def counters(self, rank: int, n: int):
        import torch
        if not 0 <= rank < self.world or not 0 <= n <= self.nsig:
            raise ValueError(f"counters({rank}, {n}) outside {self.world} ranks x {self.nsig} words")
        start = lib().tdg_symm_counters(self.h, rank) - self.buf.data_ptr()
        return self.buf[start:start + 4 * n].view(torch.int32)

    def at(self, ptr: int, rank: int):
        return lib().tdg_symm_at(self.h, _vp(ptr), rank)

    def epoch(self) -> int:
        return lib().tdg_symm_epoch(self.h)

    def status(self, stream=None, clear: bool = True):
        f = TdgFault()
        rc = lib().tdg_status(self.h, _stream(stream), ctypes.byref(f), 1 if clear else 0)
        if rc == TDG_ERR_CUDA:
            raise TdgError(rc, "tdg_status")
        return dict(code=f.code, where=WHERE.get(f.where, f.where), index=f.index, epoch=f.epoch)


def ag_gemm(symm: Symm, rank: int, Ms: int, K: int, N: int, a_off: int, g_off: int, B, C,
            mode="sm", b_layout=B_KN, producers=0, signal_rows=0, swizzle=True,
            timeout_ns=0, ll_off=0, test_skip_notify=0, source_order=0, stream=None,
            side_stream=None, c_f32=False, cluster=0, stages=0, split_tail=False,
            producer_items=0, producer_warps=0, producer_chunk=0, push=False):
    """c_f32: C is float32 (the fp32 accumulator, unrounded) instead of bf16.
    cluster / stages / split_tail / producer_items / producer_warps /
    producer_chunk / push choose the schedule (0 / False: the default for the
    shape); see tdg_ag_gemm_args in include/tdg.h."""
    import torch
    dev = symm.buf.device
    # N == 0 runs the AllGather alone: B and C may then be None
    a = AgGemmArgs(world=symm.world, rank=rank, Ms=Ms, K=K, N=N, a_off=a_off, g_off=g_off,
                   B=None if (N == 0 and B is None) else _tensor(B, "B", torch.bfloat16, K * N, dev),
                   C=None if (N == 0 and C is None) else
                   _tensor(C, "C", torch.float32 if c_f32 else torch.bfloat16, symm.world * Ms * N, dev),
                   b_layout=b_layout, mode=MODES[mode],
                   producers=producers, signal_rows=signal_rows, swizzle=1 if swizzle else 0,
                   timeout_ns=timeout_ns, ll_off=ll_off, test_skip_notify=test_skip_notify,
                   source_order=source_order, c_f32=1 if c_f32 else 0, cluster=cluster,
                   stages=stages, split_tail=1 if split_tail else 0, producer_items=producer_items,
                   producer_warps=producer_warps, producer_chunk=producer_chunk,
                   push=1 if push else 0)
    side = _vp(side_stream.cuda_stream) if side_stream is not None else _vp(None)
    _check(lib().tdg_ag_gemm(symm.h, ctypes.byref(a), _stream(stream), side), "tdg_ag_gemm")


def ag_gemm_all_ranks(symm: Symm, Ms: int, K: int, N: int, a_off: int, g_off: int, b_off: int,
                      c_off: int, mode="ce", b_layout=B_KN, signal_rows=0, timeout_ns=0,
                      test_skip_notify=0, stream=None, side_stream=None, c_f32=False,
                      cluster=0, stages=0, push=False):
    """AllGather+GEMM of every rank in one call: C_r = concat(A_0..A_{W-1}) @ B_r,
    with A_r, the gathered buffers, B_r and C_r all in the heap (offsets).
    c_f32: C_r is float32 (the fp32 accumulator, unrounded) instead of bf16.
    push: the copies go step by step, sender s to destination (s + j) mod W."""
    a = AgGemmAllArgs(world=symm.world, Ms=Ms, K=K, N=N, a_off=a_off, g_off=g_off, b_off=b_off,
                      c_off=c_off, b_layout=b_layout, mode=MODES[mode], signal_rows=signal_rows,
                      timeout_ns=timeout_ns, test_skip_notify=test_skip_notify,
                      c_f32=1 if c_f32 else 0, cluster=cluster, stages=stages,
                      push=1 if push else 0)
    side = _vp(side_stream.cuda_stream) if side_stream is not None else _vp(None)
    _check(lib().tdg_ag_gemm_all_ranks(symm.h, ctypes.byref(a), _stream(stream), side),
           "tdg_ag_gemm_all_ranks")


def gemm_rs_stage_bytes(world: int, M: int, N: int) -> int:
    return lib().tdg_gemm_rs_stage_bytes(world, M, N)


def gemm_rs(symm: Symm, M: int, K: int, N: int, a_off: int, b_off: int, stage_off: int,
            out_off: int, mode="sm", b_layout=B_KN, timeout_ns=0, owner_block=0,
            partial_f32=False, stream=None, cluster=0, stages=0, order=0, red_rows=0, spare=0):
    """partial_f32: push fp32 partials (the staging area must then hold
    2 * gemm_rs_stage_bytes(world, M, N) bytes).  cluster / stages / order /
    red_rows / owner_block / spare choose the schedule (0: the default for the
    shape; spare=n > 0 lets CTA pairs on the SMs that 4-CTA clusters leave
    idle take the last n of the world**2 groups of tiles)."""
    a = GemmRsArgs(world=symm.world, M=M, K=K, N=N, a_off=a_off, b_off=b_off,
                   stage_off=stage_off, out_off=out_off, b_layout=b_layout,
                   mode=MODES[mode], timeout_ns=timeout_ns, owner_block=owner_block,
                   partial_f32=1 if partial_f32 else 0, cluster=cluster, stages=stages,
                   order=order, red_rows=red_rows, spare=spare)
    _check(lib().tdg_gemm_rs(symm.h, ctypes.byref(a), _stream(stream)), "tdg_gemm_rs")


def allreduce_recv_bytes(world: int, count: int) -> int:
    return lib().tdg_allreduce_recv_bytes(world, count)


def allreduce(symm: Symm, count: int, x_off: int, recv_off: int, tile_elems=0, ctas_per_rank=0,
              timeout_ns=0, test_skip_signal=0, stream=None):
    a = AllReduceArgs(world=symm.world, count=count, x_off=x_off, recv_off=recv_off,
                      tile_elems=tile_elems, ctas_per_rank=ctas_per_rank, timeout_ns=timeout_ns,
                      test_skip_signal=test_skip_signal)
    _check(lib().tdg_allreduce(symm.h, ctypes.byref(a), _stream(stream)), "tdg_allreduce")


def flash_decode_part_bytes(world: int, B: int, Hq: int, D: int, S: int, chunk: int = 0) -> int:
    return lib().tdg_flash_decode_part_bytes(world, B, Hq, D, S, chunk)


def flash_decode(symm: Symm, B: int, Hq: int, Hkv: int, D: int, S: int, k_off: int, v_off: int,
                 part_off: int, q, out, root: int = 0, chunk: int = 0, scale: float = 0.0,
                 stream=None):
    import torch
    dev = symm.buf.device
    a = FlashDecodeArgs(world=symm.world, root=root, B=B, Hq=Hq, Hkv=Hkv, D=D, S=S, k_off=k_off,
                        v_off=v_off, part_off=part_off,
                        q=_tensor(q, "q", torch.bfloat16, B * Hq * D, dev),
                        out=_tensor(out, "out", torch.bfloat16, B * Hq * D, dev),
                        chunk=chunk, scale=scale)
    _check(lib().tdg_flash_decode(symm.h, ctypes.byref(a), _stream(stream)), "tdg_flash_decode")


def _moe_args(symm, T, H, E, k, x_off, topk_off, gate_off, out_off, recv, counts, base, slot,
              y, row_src, row_tok, row_k, phases):
    import torch
    dev, W = symm.buf.device, symm.world
    rows = W * T * k

    def opt(t, name, dtype, n):
        return None if t is None else _tensor(t, name, dtype, n, dev)
    return MoeArgs(world=W, T=T, H=H, E=E, k=k, x_off=x_off, topk_off=topk_off,
                   gate_off=gate_off, out_off=out_off,
                   recv=opt(recv, "recv", torch.bfloat16, rows * H),
                   y=opt(y, "y", torch.bfloat16, rows * H),
                   counts=opt(counts, "counts", torch.int64, W * E),
                   base=opt(base, "base", torch.int64, E + 1),
                   slot=opt(slot, "slot", torch.int64, rows),
                   row_src=opt(row_src, "row_src", torch.int32, rows),
                   row_tok=opt(row_tok, "row_tok", torch.int32, rows),
                   row_k=opt(row_k, "row_k", torch.int32, rows),
                   workspace=None, workspace_bytes=0, phases=phases)


def moe_workspace_bytes(world: int, T: int, E: int) -> int:
    return lib().tdg_moe_workspace_bytes(world, T, E)


def moe_dispatch_combine(symm: Symm, T: int, H: int, E: int, k: int, x_off: int, topk_off: int,
                         gate_off: int, out_off: int, recv, counts, base, slot, workspace,
                         y=None, row_src=None, row_tok=None, row_k=None, phases=MOE_ALL,
                         stream=None):
    import torch
    _tensor(workspace, "workspace", torch.uint8, 0, symm.buf.device)
    a = _moe_args(symm, T, H, E, k, x_off, topk_off, gate_off, out_off, recv, counts, base, slot,
                  y, row_src, row_tok, row_k, phases)
    a.workspace = workspace.data_ptr()
    a.workspace_bytes = workspace.numel()
    _check(lib().tdg_moe_dispatch_combine(symm.h, ctypes.byref(a), _stream(stream)),
           "tdg_moe_dispatch_combine")


def moe_dispatch_combine_noalloc(symm: Symm, T: int, H: int, E: int, k: int, x_off: int,
                                 topk_off: int, gate_off: int, out_off: int, recv, counts, base,
                                 slot, y=None, row_src=None, row_tok=None, row_k=None,
                                 phases=MOE_ALL, stream=None):
    """Same as moe_dispatch_combine, for callers that cannot allocate device
    memory when they call: the routing scratch is the library's fixed 2 MiB
    device array, so no workspace is passed.  Raises TdgError (TDG_ERR_NOMEM)
    when world * ceil(T/64) * E exceeds 262144."""
    a = _moe_args(symm, T, H, E, k, x_off, topk_off, gate_off, out_off, recv, counts, base, slot,
                  y, row_src, row_tok, row_k, phases)
    _check(lib().tdg_moe_dispatch_combine_noalloc(symm.h, ctypes.byref(a), _stream(stream)),
           "tdg_moe_dispatch_combine_noalloc")
