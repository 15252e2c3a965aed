"""tile_centric_comm_gb300 -- tile-centric overlapped AllGather+GEMM,
GEMM+ReduceScatter and MoE dispatch/combine for GB300 (sm_103a).

The compute path is the CUDA library ``libtdg.so`` (C ABI declared in
``include/tdg.h``); ``tile_centric_comm_gb300.tdg`` is its thin ctypes binding.
Importing this package loads nothing: the library is opened on first use and
every call fails loudly if it is missing.
"""
__all__ = ["synth", "tdg"]
