"""The C ABI boundary, checked on the CPU: the library builds and loads, exports
every entry point include/tdg.h declares, the ctypes structures match the C
layout (sizes and offsets printed by a C program compiled against the header),
and the host-only helpers compute the documented sizes.  No compute call."""
import ctypes
import os
import re
import subprocess

import pytest

from tile_centric_comm_gb300 import build as tdg_build
from tile_centric_comm_gb300 import tdg

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "tdg.h")


@pytest.fixture(scope="module")
def L():
    tdg_build.build()
    return tdg.lib()


def _declared():
    src = open(HEADER).read()
    return sorted(set(re.findall(r"TDG_API[^;(]*?\b(tdg_\w+)\s*\(", src)))


def test_header_declares_the_binding_exports():
    assert _declared() == sorted(tdg.EXPORTS)


def test_library_exports_every_declared_symbol(L):
    out = subprocess.run(["nm", "-D", "--defined-only", tdg.LIB_PATH], capture_output=True,
                         text=True, check=True).stdout
    exported = set(re.findall(r" T (tdg_\w+)$", out, re.M))
    for name in _declared():
        assert name in exported, name
        assert getattr(L, name) is not None


def test_struct_layouts_match_c(tmp_path):
    prog = tmp_path / "layout.c"
    prog.write_text(r'''
#include <stdio.h>
#include <stddef.h>
#include "tdg.h"
#define F(T, f) printf(#T "." #f " %zu\n", offsetof(T, f))
int main(void) {
  printf("tdg_ag_gemm_args %zu\n", sizeof(tdg_ag_gemm_args));
  printf("tdg_gemm_rs_args %zu\n", sizeof(tdg_gemm_rs_args));
  printf("tdg_moe_args %zu\n", sizeof(tdg_moe_args));
  printf("tdg_fault %zu\n", sizeof(tdg_fault));
  F(tdg_ag_gemm_args, B); F(tdg_ag_gemm_args, signal_rows); F(tdg_ag_gemm_args, timeout_ns);
  F(tdg_ag_gemm_args, test_skip_notify);
  F(tdg_gemm_rs_args, out_off); F(tdg_gemm_rs_args, timeout_ns); F(tdg_gemm_rs_args, partial_f32);
  printf("tdg_allreduce_args %zu\n", sizeof(tdg_allreduce_args));
  printf("tdg_ag_gemm_all_args %zu\n", sizeof(tdg_ag_gemm_all_args));
  F(tdg_ag_gemm_all_args, c_off); F(tdg_ag_gemm_all_args, signal_rows); F(tdg_ag_gemm_all_args, test_skip_notify);
  printf("tdg_flash_decode_args %zu\n", sizeof(tdg_flash_decode_args));
  F(tdg_allreduce_args, timeout_ns); F(tdg_allreduce_args, test_skip_signal); F(tdg_flash_decode_args, out); F(tdg_flash_decode_args, scale);
  F(tdg_moe_args, recv); F(tdg_moe_args, workspace_bytes); F(tdg_moe_args, phases);
  return 0;
}
''')
    exe = tmp_path / "layout"
    subprocess.run(["gcc", "-I", os.path.join(ROOT, "include"), str(prog), "-o", str(exe)],
                   check=True)
    got = dict(l.split() for l in subprocess.run([str(exe)], capture_output=True, text=True,
                                                 check=True).stdout.splitlines())
    assert int(got["tdg_ag_gemm_args"]) == ctypes.sizeof(tdg.AgGemmArgs)
    assert int(got["tdg_gemm_rs_args"]) == ctypes.sizeof(tdg.GemmRsArgs)
    assert int(got["tdg_moe_args"]) == ctypes.sizeof(tdg.MoeArgs)
    assert int(got["tdg_fault"]) == ctypes.sizeof(tdg.TdgFault)
    assert int(got["tdg_allreduce_args"]) == ctypes.sizeof(tdg.AllReduceArgs)
    assert int(got["tdg_flash_decode_args"]) == ctypes.sizeof(tdg.FlashDecodeArgs)
    assert int(got["tdg_ag_gemm_all_args"]) == ctypes.sizeof(tdg.AgGemmAllArgs)
    for key, val in got.items():
        if "." in key:
            s, f = key.split(".")
            cls = {"tdg_ag_gemm_args": tdg.AgGemmArgs, "tdg_gemm_rs_args": tdg.GemmRsArgs,
                   "tdg_moe_args": tdg.MoeArgs, "tdg_allreduce_args": tdg.AllReduceArgs,
                   "tdg_flash_decode_args": tdg.FlashDecodeArgs,
                   "tdg_ag_gemm_all_args": tdg.AgGemmAllArgs}[s]
            assert getattr(cls, f).offset == int(val), key


def test_host_size_helpers(L):
    # heap: regions, then two 256-aligned word areas, then a 256-byte status block
    assert L.tdg_symm_bytes(8, 1 << 20, 1000) == 8 * (1 << 20) + 2 * 32000 + 256
    assert L.tdg_symm_bytes(0, 1024, 1) == 0
    # staging: W partials of (Mo/128) x ceil(N/256) tiles of 128 x 256 bf16
    assert L.tdg_gemm_rs_stage_bytes(8, 8192, 5120) == 8 * 8 * 20 * 128 * 256 * 2
    assert L.tdg_gemm_rs_stage_bytes(2, 256, 520) == 2 * 1 * 3 * 65536
    assert L.tdg_gemm_rs_stage_bytes(3, 256, 8) == 0           # M % W != 0
    # MoE workspace: two int32 tables of W x ceil(T/64) x E
    assert L.tdg_moe_workspace_bytes(8, 4096, 256) == 2 * 8 * 64 * 256 * 4
    assert L.tdg_moe_workspace_bytes(2, 65, 4) == 2 * 2 * 2 * 4 * 4
    # ring AllReduce: W-1 receive slots of count/W float32
    assert L.tdg_allreduce_recv_bytes(8, 1 << 20) == 7 * (1 << 17) * 4
    assert L.tdg_allreduce_recv_bytes(1, 1024) == 0
    # flash decoding partials: W * splits * B * Hq * (D + 2) float32
    assert L.tdg_flash_decode_part_bytes(8, 4, 64, 128, 131072, 512) == 8 * 32 * 4 * 64 * 130 * 4
    assert L.tdg_flash_decode_part_bytes(8, 4, 64, 128, 131072, 0) == 8 * 8 * 4 * 64 * 130 * 4
    assert L.tdg_flash_decode_part_bytes(4, 1, 16, 128, 400, 64) == 4 * 2 * 1 * 16 * 130 * 4
    assert L.tdg_flash_decode_part_bytes(3, 1, 16, 128, 400, 64) == 0        # S % W != 0


def test_strerror_and_invalid_handles(L):
    for code in (0, -1, -2, -3, -4, -5, -6):
        assert len(tdg.strerror(code)) >= 2
    assert L.tdg_symm_region(None, 0) is None
    assert L.tdg_symm_at(None, None, 0) is None
    assert L.tdg_symm_epoch(None) == 0
    assert L.tdg_symm_free(None) == 0
    assert L.tdg_ag_gemm(None, None, None, None) == tdg.TDG_ERR_INVALID
    assert L.tdg_gemm_rs(None, None, None) == tdg.TDG_ERR_INVALID
    assert L.tdg_moe_dispatch_combine(None, None, None) == tdg.TDG_ERR_INVALID
    assert L.tdg_allreduce(None, None, None) == tdg.TDG_ERR_INVALID
    assert L.tdg_flash_decode(None, None, None) == tdg.TDG_ERR_INVALID
    h = ctypes.c_void_p()
    # misaligned base / bad world are rejected before any CUDA call
    assert L.tdg_symm_alloc(ctypes.c_void_p(1024 + 16), 1 << 20, 2, 4096, 16,
                            ctypes.byref(h)) == tdg.TDG_ERR_INVALID
    assert L.tdg_symm_alloc(ctypes.c_void_p(1024), 1 << 20, 0, 4096, 16,
                            ctypes.byref(h)) == tdg.TDG_ERR_INVALID
    assert L.tdg_symm_alloc(ctypes.c_void_p(1024), 100, 2, 4096, 16,
                            ctypes.byref(h)) == tdg.TDG_ERR_NOMEM


def test_binding_tensor_checks_on_the_host():
    """The library sees raw pointers only, so the binding refuses a tensor
    whose dtype, layout or size it cannot describe (checked before the device)."""
    import torch
    good = torch.zeros(4, 8, dtype=torch.bfloat16)
    with pytest.raises(TypeError, match="bfloat16"):
        tdg._tensor(good.float(), "B", torch.bfloat16, 32)
    with pytest.raises(ValueError, match="contiguous"):
        tdg._tensor(good.t(), "B", torch.bfloat16, 32)
    with pytest.raises(ValueError, match="needs 33"):
        tdg._tensor(good, "B", torch.bfloat16, 33)
    with pytest.raises(ValueError, match="CUDA"):
        tdg._tensor(good, "B", torch.bfloat16, 32)
    with pytest.raises(TypeError, match="torch.Tensor"):
        tdg._tensor([0] * 32, "B", torch.bfloat16, 32)
