"""Benchmark of the tile-centric hot path on GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl tdg|reference]

Workload (one "step"): the tensor-parallel MLP layer of Qwen-32B over W=8
logical ranks held in one GPU -- AllGather+GEMM of the up-projection
(A_r 1024x5120 per rank, B 5120x3200) followed by GEMM+ReduceScatter of the
down-projection (A_r 8192x3200, B_r 3200x5120 per rank).  Metric: TFLOP/s of
the two operations together (2*M*N*K counted once per GEMM), with inputs
resident in HBM; L2 is flushed (256 MB write) before every timed step.  The
same run also reports the overlap gain against the serial composition (copy,
then GEMM, then reduce), the end-to-end rate with host buffers, the MoE
dispatch+combine bandwidth, the roofline of the dominant kernel and the CPU
oracle's rate on a bounded sample.

--impl reference times the CPU oracle on a bounded sample of the same
workload each step (the reference arm for this path is the oracle); under
torchrun rank 0 alone runs it.

The path runs on one GPU: its W ranks are logical regions of one device, and
its GEMMs share B slices between the CTA pairs of a cluster by TMA multicast,
which is meant for one GPU's own memory.  With --gpus N > 1 (or under a
torchrun of several processes) rank 0 prints one line with an "unavailable"
key and every rank exits 0 without touching a GPU.
"""
from __future__ import annotations

import argparse
import copy
import json
import os
import statistics
import subprocess
import tempfile
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

AG = dict(W=8, Ms=1024, K=5120, N=3200)          # Qwen-32B MLP up-projection
RS = dict(W=8, M=8192, K=3200, N=5120)           # Qwen-32B MLP down-projection
MOE = dict(W=8, T=4096, H=7168, E=256, k=8)      # MoE dispatch + combine
AG_FLOP = 2 * AG["W"] * AG["Ms"] * AG["K"] * AG["N"]
RS_FLOP = 2 * RS["W"] * RS["M"] * RS["K"] * RS["N"]
STEP_FLOP = AG_FLOP + RS_FLOP
WORKLOAD = ("qwen32b_mlp_tp8: AG-GEMM up-proj (W=8, A_r 1024x5120, B 5120x3200) + "
            "GEMM-RS down-proj (W=8, A_r 8192x3200, B_r 3200x5120), bf16 in, fp32 accumulate, bf16 out")


# DRAM traffic of one rs_gemm_kernel launch at this workload, dram__bytes_read.sum +
# dram__bytes_write.sum from one ncu capture (1.475 GB read + 0.706 GB written).  It is
# reported only while the kernel's code (comments aside) still hashes to the value the capture was taken with.
RS_TRAFFIC = {"sources": "679df334010ed7a3", "bytes": 1_474_665_728 + 705_864_704}
RS_SOURCES = ["tdg_gemm.cuh", "tdg_rs.cu", "tdg_ptx.cuh"]


def rs_sources_hash():
    """Hash of the code (comments and blank space left out) of the files the
    GEMM-RS kernel is built from: a change of wording keeps the capture."""
    import hashlib
    import re
    h = hashlib.sha256()
    for f in RS_SOURCES:
        with open(os.path.join(ROOT, "tile_centric_comm_gb300", "csrc", f), encoding="utf-8") as fh:
            src = fh.read()
        src = re.sub(r"/\*.*?\*/", " ", src, flags=re.S)            # block comments
        src = re.sub(r"//[^\n]*", " ", src)                           # line comments
        h.update(" ".join(src.split()).encode())
    return h.hexdigest()[:16]


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="tdg", choices=["tdg", "reference"])
    ap.add_argument("--mode", default="ce", choices=["sm", "ce", "serial"],
                    help="AG-GEMM overlap: ce = copy engine + flags (default), sm = producer CTAs, "
                         "serial = copy launch then GEMM launch (for measurement only)")
    ap.add_argument("--producers", type=int, default=0)
    ap.add_argument("--signal-rows", type=int, default=0,
                    help="AG rows per signal group (0: the library's default for the mode)")
    ap.add_argument("--no-extras", action="store_true", help="skip serial/e2e/MoE/CPU legs")
    ap.add_argument("--no-cpu", action="store_true")
    ap.add_argument("--only", default="", help="measure one operation alone, not the bench line: "
                    "ag, rs, moe, ring, flash, ag_all (the AG-GEMM of all ranks in one call) or copy "
                    "(the AllGather alone, SERIAL copy launch on --producers CTAs or --mode ce); "
                    "'library' times torch.matmul (cuBLAS) on the AG GEMM shape as context")
    ap.add_argument("--ag-shape", default="", help="W,Ms,K,N for --only ag|library, e.g. 8,2048,8192,7168 "
                    "(the Llama-3-70B gate+up shape)")
    return ap.parse_args()


def dist_env():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return dict(hbm=d["hbm_gbs"], bf16=d["bf16_tflops"], bf16_sus=d["bf16_tflops_sustained"],
                    src="measured")
    return dict(hbm=6800.0, bf16=1900.0, bf16_sus=1700.0, src="fallback")


class Clocks:
    """nvidia-smi samples during the timed region."""

    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        self.index = index
        self.proc = None
        self.path = os.path.join(tempfile.gettempdir(), f"tdg_clocks_{os.getpid()}_{index}.csv")

    def __enter__(self):
        try:
            os.makedirs(os.path.dirname(self.path), exist_ok=True)
            self.f = open(self.path, "w")
            self.proc = subprocess.Popen(["nvidia-smi", f"--id={self.index}", f"--query-gpu={self.Q}",
                                          "--format=csv,noheader,nounits", "-lms", "20"],
                                         stdout=self.f, stderr=subprocess.DEVNULL)
            # the timed region starts only once the sampler is producing lines
            t0 = time.time()
            while time.time() - t0 < 10:
                self.f.flush()
                if os.path.getsize(self.path) > 0:
                    break
                time.sleep(0.05)
            self.start_line = sum(1 for _ in open(self.path))
        except Exception:
            self.proc = None
        return self

    def __exit__(self, *a):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()
            self.f.close()

    def summary(self):
        if self.proc is None or not os.path.exists(self.path):
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        rows = []
        for i, line in enumerate(open(self.path)):
            if i < getattr(self, "start_line", 0):
                continue
            parts = [x.strip() for x in line.split(",")]
            if len(parts) >= 9:
                rows.append(parts)
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
        sm = [float(r[1]) for r in rows if r[1].replace(".", "").isdigit()]
        mx = [float(r[2]) for r in rows if r[2].replace(".", "").isdigit()]
        pw = [float(r[3]) for r in rows if r[3].replace(".", "").isdigit()]
        reasons = set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for r in rows:
            for n, v in zip(names, r[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        loaded = [s for s, p in zip(sm, pw) if p > 300] or sm
        return {"sm_mhz": statistics.median(loaded) if loaded else None,
                "sm_max_mhz": max(mx) if mx else None, "reasons": sorted(reasons),
                "samples": len(rows), "power_w_max": max(pw) if pw else None}


# ------------------------------------------------------------ GPU workload ----
def _dev_bf16(bits, torch):
    import numpy as np
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16).cuda()


def _align(x, a=1024):
    return (x + a - 1) // a * a


class MLP:
    """Inputs of both operations resident in two symmetric heaps."""

    def __init__(self, torch, tdg, synth, mode, producers, signal_rows=0):
        self.torch, self.tdg, self.mode, self.producers = torch, tdg, mode, producers
        self.signal_rows = signal_rows
        ag = synth.ag_inputs(AG["W"], AG["Ms"], AG["K"], AG["N"], "normal", seed=0)
        W, Ms, K, N = AG["W"], AG["Ms"], AG["K"], AG["N"]
        self.ag_a_off = 0
        self.ag_g_off = _align(Ms * K * 2)
        self.ag_host = [torch.from_numpy(a.view("int16")).view(torch.bfloat16).pin_memory()
                        for a in ag.shards]
        self.ag_B_host = torch.from_numpy(ag.B.view("int16")).view(torch.bfloat16).pin_memory()
        del ag
        rs = synth.rs_inputs(RS["W"], RS["M"], RS["K"], RS["N"], "normal", seed=0)
        W, M, K, N = RS["W"], RS["M"], RS["K"], RS["N"]
        self.rs_a_off = 0
        self.rs_b_off = _align(M * K * 2)
        self.rs_s_off = _align(self.rs_b_off + K * N * 2)
        self.rs_o_off = _align(self.rs_s_off + tdg.gemm_rs_stage_bytes(W, M, N))
        self.rs_A_host = [torch.from_numpy(a.view("int16")).view(torch.bfloat16).pin_memory() for a in rs.As]
        self.rs_B_host = [torch.from_numpy(b.view("int16")).view(torch.bfloat16).pin_memory() for b in rs.Bs]
        del rs
        self._alloc_device()
        self.upload_ag()
        self.upload_rs()
        self.h2d_bytes = (sum(t.numel() for t in self.ag_host) + self.ag_B_host.numel()
                          + sum(t.numel() for t in self.rs_A_host)
                          + sum(t.numel() for t in self.rs_B_host)) * 2
        self.d2h_bytes = (self.C_host.numel() + self.out_host.numel()) * 2
        self.h2d_act_bytes = (sum(t.numel() for t in self.ag_host) + sum(t.numel() for t in self.rs_A_host)) * 2

    def _alloc_device(self):
        """Device heaps and outputs (and the pinned host outputs) of one step."""
        torch, tdg = self.torch, self.tdg
        W, Ms, K, N = AG["W"], AG["Ms"], AG["K"], AG["N"]
        self.ag = tdg.Symm(W, _align(self.ag_g_off + W * Ms * K * 2 + 1024), 65536)
        self.ag_B = torch.empty((K, N), dtype=torch.bfloat16, device="cuda")
        self.ag_C = torch.empty((W * Ms, N), dtype=torch.bfloat16, device="cuda")
        W, M, K, N = RS["W"], RS["M"], RS["K"], RS["N"]
        self.rs = tdg.Symm(W, _align(self.rs_o_off + (M // W) * N * 2 + 1024), 65536)
        self.C_host = torch.empty((AG["W"] * AG["Ms"], AG["N"]), dtype=torch.bfloat16).pin_memory()
        self.out_host = torch.empty((RS["W"], RS["M"] // RS["W"], RS["N"]),
                                    dtype=torch.bfloat16).pin_memory()

    def twin(self):
        """A second set of device buffers (and host outputs) over the same
        pinned host inputs, so that consecutive end-to-end steps can alternate
        between two sets: the uploads of one step run while the previous step
        computes and downloads."""
        t = copy.copy(self)
        for k in ("_copy_stream", "_side_stream"):
            t.__dict__.pop(k, None)
        t._alloc_device()
        return t

    def ag_call(self, mode=None, side=None):
        mode = mode or self.mode
        if mode == "ce" and side is None:
            side = self._side()
        self.tdg.ag_gemm(self.ag, 0, AG["Ms"], AG["K"], AG["N"], self.ag_a_off, self.ag_g_off,
                         self.ag_B, self.ag_C, mode=mode, producers=self.producers,
                         signal_rows=self.signal_rows, side_stream=side)

    def _side(self):
        if not hasattr(self, "_side_stream"):
            self._side_stream = self.torch.cuda.Stream()
        return self._side_stream

    def rs_call(self, mode="sm"):
        self.tdg.gemm_rs(self.rs, RS["M"], RS["K"], RS["N"], self.rs_a_off, self.rs_b_off,
                         self.rs_s_off, self.rs_o_off, mode=mode)

    def upload_ag(self, weights=True):
        """host -> device copies of the AG-GEMM inputs (pinned, async); the
        weight B only when `weights`."""
        t = self.torch
        Ms, K = AG["Ms"], AG["K"]
        for s in range(AG["W"]):
            self.ag.view(s, 0, (Ms, K), t.bfloat16).copy_(self.ag_host[s], non_blocking=True)
        if weights:
            self.ag_B.copy_(self.ag_B_host, non_blocking=True)

    def upload_rs(self, weights=True):
        t = self.torch
        M, K, N = RS["M"], RS["K"], RS["N"]
        for r in range(RS["W"]):
            self.rs.view(r, self.rs_a_off, (M, K), t.bfloat16).copy_(self.rs_A_host[r], non_blocking=True)
            if weights:
                self.rs.view(r, self.rs_b_off, (K, N), t.bfloat16).copy_(self.rs_B_host[r], non_blocking=True)

    def download_ag(self):
        self.C_host.copy_(self.ag_C, non_blocking=True)

    def download_rs(self):
        Mo, N = RS["M"] // RS["W"], RS["N"]
        for o in range(RS["W"]):
            self.out_host[o].copy_(self.rs.view(o, self.rs_o_off, (Mo, N), self.torch.bfloat16),
                                   non_blocking=True)

    def e2e_step(self):
        """One step through the public API with host buffers: uploads on a copy
        stream overlap the compute of the previous operation, and the AG output
        downloads while the GEMM-RS runs."""
        t = self.torch
        ms = t.cuda.current_stream()
        if not hasattr(self, "_copy_stream"):
            self._copy_stream = t.cuda.Stream()
        cs = self._copy_stream
        start = t.cuda.Event()
        start.record(ms)
        cs.wait_event(start)               # nothing of this step starts before it
        ag_in, rs_in, ag_done = t.cuda.Event(), t.cuda.Event(), t.cuda.Event()
        with t.cuda.stream(cs):
            self.upload_ag()
            ag_in.record(cs)
            self.upload_rs()
            rs_in.record(cs)
        ms.wait_event(ag_in)
        self.ag_call()
        ag_done.record(ms)
        ms.wait_event(rs_in)
        self.rs_call("sm")
        with t.cuda.stream(cs):
            cs.wait_event(ag_done)
            self.download_ag()
        self.download_rs()
        ms.wait_stream(cs)

    def e2e_pipelined(self, sets, steps, warmup, weights=True):
        """End-to-end throughput with consecutive steps overlapped: step i uses
        buffer set i % 2.  Per step: H2D of all inputs on the upload stream,
        AG-GEMM then GEMM-RS on the compute stream (each waits for its own
        inputs), D2H of both outputs on the download stream.  A set is reused
        only after the download of its previous step has finished.  Returns
        the mean milliseconds per step over `steps` timed steps."""
        t = self.torch
        comp = t.cuda.current_stream()
        up, down = t.cuda.Stream(), t.cuda.Stream()
        free = [t.cuda.Event() for _ in sets]
        for e in free:
            e.record(comp)

        def step(i):
            S = sets[i % len(sets)]
            ag_in, rs_in, ag_done, rs_done = (t.cuda.Event() for _ in range(4))
            up.wait_event(free[i % len(sets)])
            with t.cuda.stream(up):
                S.upload_ag(weights)
                ag_in.record(up)
                S.upload_rs(weights)
                rs_in.record(up)
            comp.wait_event(ag_in)
            S.ag_call()
            ag_done.record(comp)
            comp.wait_event(rs_in)
            S.rs_call("sm")
            rs_done.record(comp)
            down.wait_event(ag_done)
            with t.cuda.stream(down):
                S.download_ag()
                down.wait_event(rs_done)
                S.download_rs()
                free[i % len(sets)].record(down)

        for i in range(warmup):
            step(i)
        t.cuda.synchronize()
        e0, e1 = t.cuda.Event(enable_timing=True), t.cuda.Event(enable_timing=True)
        e0.record(comp)
        up.wait_event(e0)
        for i in range(warmup, warmup + steps):
            step(i)
        comp.wait_stream(up)
        comp.wait_stream(down)
        e1.record(comp)
        t.cuda.synchronize()
        return e0.elapsed_time(e1) / steps

    def check_status(self):
        for s in (self.ag, self.rs):
            st = s.status()
            if st["code"] != 0:
                raise RuntimeError(f"device fault during the bench: {st}")


def timed_steps(torch, fns, steps, warmup, flush):
    """Run `fns` (one callable per part) once per step, flushing L2 before every
    step (outside the events); return per-part lists of device times (ms) of the
    timed steps.  The GPU runs the steps back to back; the host waits once."""
    n = len(fns)
    stream = torch.cuda.current_stream()
    for _ in range(warmup):
        flush.zero_()
        for f in fns:
            f()
    torch.cuda.synchronize()
    evs = []
    for _ in range(steps):
        flush.zero_()
        e = [torch.cuda.Event(enable_timing=True) for _ in range(n + 1)]
        e[0].record(stream)
        for i, f in enumerate(fns):
            f()
            e[i + 1].record(stream)
        evs.append(e)
    torch.cuda.synchronize()
    return [[e[i].elapsed_time(e[i + 1]) for e in evs] for i in range(n)]


def interleaved_steps(torch, variants, rounds, steps, flush):
    """Time several variants of one step in alternating rounds (the order
    rotated every round), so that all of them see the same clock and power
    state: the power cap lowers the clock as a long run goes on, which would
    favour whichever variant ran first.  `variants` maps a name to a list of
    callables (the parts of one step).  Returns {name: [mean ms per part]}."""
    names = list(variants)
    acc = {n: [[] for _ in variants[n]] for n in names}
    for r in range(rounds):
        order = names[r % len(names):] + names[:r % len(names)]
        for n in order:
            parts = timed_steps(torch, variants[n], steps, 1, flush)
            for i, pt in enumerate(parts):
                acc[n][i].extend(pt)
    return {n: [statistics.mean(x) for x in acc[n]] for n in names}


def cpu_oracle_rate(sample_rows_ag=1280, sample_rows_rs=320):
    """The oracle, as it stands, on a bounded sample of the same workload:
    full output rows of AG-GEMM and GEMM-RS.  Returns (TFLOP/s, seconds, desc)."""
    import numpy as np
    import oracle
    from tile_centric_comm_gb300 import synth
    ag = synth.ag_inputs(AG["W"], AG["Ms"], AG["K"], AG["N"], "normal", seed=0)
    rows = np.repeat(np.arange(sample_rows_ag) * 31 % (AG["W"] * AG["Ms"]), AG["N"])
    cols = np.tile(np.arange(AG["N"]), sample_rows_ag)
    t0 = time.perf_counter()
    oracle.ag_gemm_sampled(ag.shards, ag.B, rows, cols)
    t_ag = time.perf_counter() - t0
    del ag
    rs = synth.rs_inputs(RS["W"], RS["M"], RS["K"], RS["N"], "normal", seed=0)
    rows = np.repeat(np.arange(sample_rows_rs) * 127 % RS["M"], RS["N"])
    cols = np.tile(np.arange(RS["N"]), sample_rows_rs)
    t0 = time.perf_counter()
    oracle.gemm_rs_sampled(rs.As, rs.Bs, rows, cols)
    t_rs = time.perf_counter() - t0
    flop = 2.0 * AG["K"] * AG["N"] * sample_rows_ag + 2.0 * RS["W"] * RS["K"] * RS["N"] * sample_rows_rs
    desc = (f"{sample_rows_ag} full output rows of the AG-GEMM ({sample_rows_ag}x{AG['N']} outputs) + "
            f"{sample_rows_rs} full output rows of the GEMM-RS ({sample_rows_rs}x{RS['N']} outputs, "
            f"W={RS['W']} partial sums each), fp64 plain loops")
    return flop / (t_ag + t_rs) / 1e12, t_ag + t_rs, desc


def omp_threads():
    v = os.environ.get("OMP_NUM_THREADS")
    return int(v) if v and v.isdigit() else (os.cpu_count() or 1)


class MoEBench:
    """MoE route + dispatch + combine over 8 ranks x 4096 tokens (HBM bound)."""

    def __init__(self, torch, tdg, synth):
        self.torch, self.tdg = torch, tdg
        W, T, H, E, k = MOE["W"], MOE["T"], MOE["H"], MOE["E"], MOE["k"]
        inp = synth.moe_inputs(W, T, H, E, k, seed=0)
        self.x_off = 0
        self.topk_off = _align(T * H * 2)
        self.gate_off = _align(self.topk_off + T * k * 4)
        self.out_off = _align(self.gate_off + T * k * 4)
        self.symm = tdg.Symm(W, _align(self.out_off + T * H * 2 + 1024), 1024)
        import numpy as np
        for s in range(W):
            self.symm.view(s, self.x_off, (T, H), torch.bfloat16).copy_(_dev_bf16(inp.x[s], torch))
            self.symm.view(s, self.topk_off, (T, k), torch.int32).copy_(torch.from_numpy(np.ascontiguousarray(inp.topk[s])))
            self.symm.view(s, self.gate_off, (T, k), torch.float32).copy_(torch.from_numpy(np.ascontiguousarray(inp.gate[s])))
        total = W * T * k
        self.recv = torch.empty((total, H), dtype=torch.bfloat16, device="cuda")
        self.counts = torch.empty((W, E), dtype=torch.int64, device="cuda")
        self.base = torch.empty(E + 1, dtype=torch.int64, device="cuda")
        self.slot = torch.empty((W, T, k), dtype=torch.int64, device="cuda")
        self.ws = torch.empty(tdg.moe_workspace_bytes(W, T, E), dtype=torch.uint8, device="cuda")
        row = H * 2
        self.bytes_dispatch = W * T * row + total * row      # read x once, write k copies
        self.bytes_combine = total * row + W * T * row       # read k rows, write one

    def call(self, phases):
        W, T, H, E, k = MOE["W"], MOE["T"], MOE["H"], MOE["E"], MOE["k"]
        self.tdg.moe_dispatch_combine(self.symm, T, H, E, k, self.x_off, self.topk_off, self.gate_off,
                                      self.out_off, self.recv, self.counts, self.base, self.slot,
                                      self.ws, phases=phases)


def run_reference(args, rank):
    """The reference arm: the CPU oracle on a bounded sample per step."""
    if rank != 0:
        return
    rates, secs = [], []
    desc = ""
    for it in range(args.warmup + args.steps):
        r, s, desc = cpu_oracle_rate(sample_rows_ag=8, sample_rows_rs=2)
        if it >= args.warmup:
            rates.append(r)
            secs.append(s)
    v = statistics.median(rates)
    line = {"impl": "reference", "metric": "AG-GEMM+GEMM-RS TFLOP/s (qwen32b_mlp_tp8)", "value": v,
            "unit": "TFLOP/s", "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": 1e3 * statistics.mean(secs), "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": WORKLOAD, "sample": desc},
            "cpu_baseline": {"value": v, "unit": "TFLOP/s", "cores": omp_threads(), "kind": "oracle",
                             "sample": desc},
            "e2e": {"value": v, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def leg_moe(torch, tdg, synth, args, flush, pk):
    extras = {}
    # MoE dispatch + combine
    moe = MoEBench(torch, tdg, synth)
    moe.call(tdg.MOE_ROUTE)
    torch.cuda.synchronize()
    mparts = timed_steps(torch, [lambda: moe.call(tdg.MOE_ROUTE), lambda: moe.call(tdg.MOE_DISPATCH),
                                 lambda: moe.call(tdg.MOE_COMBINE)], args.steps, args.warmup, flush)
    m_route, m_disp, m_comb = (statistics.mean(x) for x in mparts)
    bytes_dc = moe.bytes_dispatch + moe.bytes_combine
    extras["moe_dispatch_combine"] = {
        "workload": "8 ranks x 4096 tokens, hidden 7168 bf16, 256 experts, top-8 Zipf(1.2)",
        "route_ms": m_route, "dispatch_ms": m_disp, "combine_ms": m_comb,
        "dispatch_gbs": moe.bytes_dispatch / m_disp / 1e6, "combine_gbs": moe.bytes_combine / m_comb / 1e6,
        "gbs": bytes_dc / (m_disp + m_comb) / 1e6,
        "frac_of_hbm": bytes_dc / (m_disp + m_comb) / 1e6 / pk["hbm"]}
    st = moe.symm.status()
    if st["code"] != 0:
        raise RuntimeError(f"device fault in MoE: {st}")
    del moe
    torch.cuda.empty_cache()
    return extras["moe_dispatch_combine"]


def leg_ag_all(torch, tdg, args, flush, pk):
    """The AG-GEMM of the step for every logical rank in one call (W x the
    work: each rank gathers all shards and multiplies by its own B_r), CE mode
    against its serial twin, timed in interleaved rounds."""
    W, Ms, K, N = AG["W"], AG["Ms"], AG["K"], AG["N"]
    M = W * Ms
    a_off, g_off = 0, _align(Ms * K * 2)
    b_off = _align(g_off + M * K * 2)
    c_off = _align(b_off + K * N * 2)
    sym = tdg.Symm(W, _align(c_off + M * N * 2 + 1024), 65536)
    g = torch.Generator(device="cuda")
    g.manual_seed(0)
    for r in range(W):
        sym.view(r, a_off, (Ms, K), torch.bfloat16).copy_(torch.randn(Ms, K, device="cuda", generator=g))
        sym.view(r, b_off, (K, N), torch.bfloat16).copy_(torch.randn(K, N, device="cuda", generator=g) * 0.02)
    side = torch.cuda.Stream()
    call = lambda mode, push=False: (lambda: tdg.ag_gemm_all_ranks(sym, Ms, K, N, a_off, g_off, b_off, c_off,
                                                                   mode=mode, push=push,
                                                                   side_stream=side if mode == "ce" else None))
    flop = W * AG_FLOP
    res = {"workload": "AG-GEMM Qwen-32B up for all 8 logical ranks in one call (8 x 8192x3200x5120, "
                       "56 remote shard copies)",
           "note": "synthetic N(0,1) shards, 0.02*N(0,1) B_r generated on the device"}
    if args.only == "ag_all" and args.mode == "serial":
        # the serial twin alone (no flag waits: the form an ncu capture can replay)
        ms = statistics.mean(timed_steps(torch, [call("serial")], args.steps, args.warmup, flush)[0])
        res.update({"serial_ms": ms, "serial_tflops": flop / ms / 1e9,
                    "serial_frac_of_bf16_peak": flop / ms / 1e9 / pk["bf16"]})
    else:
        iv = interleaved_steps(torch, {"ce": [call("ce")], "serial": [call("serial")],
                                       "ce_push": [call("ce", True)]}, 3, max(4, args.steps // 5), flush)
        res.update({"ce_ms": iv["ce"][0], "ce_tflops": flop / iv["ce"][0] / 1e9,
                    "ce_frac_of_bf16_peak": flop / iv["ce"][0] / 1e9 / pk["bf16"],
                    "serial_ms": iv["serial"][0], "serial_tflops": flop / iv["serial"][0] / 1e9,
                    "ce_overlap_gain_vs_serial": iv["serial"][0] / iv["ce"][0],
                    "ce_push_ms": iv["ce_push"][0], "ce_push_tflops": flop / iv["ce_push"][0] / 1e9,
                    "ce_push_overlap_gain_vs_serial": iv["serial"][0] / iv["ce_push"][0]})
        res["note"] += "; modes in 3 interleaved rounds"
    st = sym.status()
    if st["code"] != 0:
        raise RuntimeError(f"device fault in the all-ranks AG-GEMM: {st}")
    del sym
    torch.cuda.empty_cache()
    return res


def leg_tp_mlp_all(torch, tdg, args, flush, pk):
    """The Qwen-32B tensor-parallel MLP forward (without the activation) for
    all 8 logical ranks: the all-ranks AG-GEMM writes every C_r into the heap
    and the GEMM-RS reads it there as its A_r (no copy between the two).
    Overlapped (CE + fused RS) against the serial twins, interleaved rounds."""
    W, Ms, H, F = AG["W"], AG["Ms"], AG["K"], AG["N"]     # hidden 5120, ffn shard 3200
    M = W * Ms
    a_off, g_off = 0, _align(Ms * H * 2)
    bu_off = _align(g_off + M * H * 2)
    c_off = _align(bu_off + H * F * 2)
    bd_off = _align(c_off + M * F * 2)
    s_off = _align(bd_off + F * H * 2)
    o_off = _align(s_off + tdg.gemm_rs_stage_bytes(W, M, H))
    sym = tdg.Symm(W, _align(o_off + Ms * H * 2 + 1024), 65536)
    g = torch.Generator(device="cuda")
    g.manual_seed(0)
    for r in range(W):
        sym.view(r, a_off, (Ms, H), torch.bfloat16).copy_(torch.randn(Ms, H, device="cuda", generator=g))
        sym.view(r, bu_off, (H, F), torch.bfloat16).copy_(torch.randn(H, F, device="cuda", generator=g) * 0.02)
        sym.view(r, bd_off, (F, H), torch.bfloat16).copy_(torch.randn(F, H, device="cuda", generator=g) * 0.02)
    side = torch.cuda.Stream()
    over = [lambda: tdg.ag_gemm_all_ranks(sym, Ms, H, F, a_off, g_off, bu_off, c_off, mode="ce", side_stream=side),
            lambda: tdg.gemm_rs(sym, M, F, H, c_off, bd_off, s_off, o_off, mode="sm")]
    ser = [lambda: tdg.ag_gemm_all_ranks(sym, Ms, H, F, a_off, g_off, bu_off, c_off, mode="serial"),
           lambda: tdg.gemm_rs(sym, M, F, H, c_off, bd_off, s_off, o_off, mode="serial")]
    iv = interleaved_steps(torch, {"overlapped": over, "serial": ser}, 3, max(4, args.steps // 5), flush)
    st = sym.status()
    if st["code"] != 0:
        raise RuntimeError(f"device fault in the all-ranks MLP: {st}")
    del sym
    torch.cuda.empty_cache()
    o_ms, s_ms = sum(iv["overlapped"]), sum(iv["serial"])
    flop = W * AG_FLOP + RS_FLOP
    return {"workload": "Qwen-32B TP MLP forward for all 8 logical ranks: all-ranks AG-GEMM up "
                        "(8 x 8192x3200x5120) into the heap, then GEMM-RS down reading it (8 x 8192x5120x3200)",
            "tflop_per_step": flop / 1e12, "ms": o_ms, "tflops": flop / o_ms / 1e9,
            "frac_of_bf16_peak": flop / o_ms / 1e9 / pk["bf16"], "ag_ms": iv["overlapped"][0],
            "rs_ms": iv["overlapped"][1], "serial_ms": s_ms, "serial_tflops": flop / s_ms / 1e9,
            "overlap_gain_vs_serial": s_ms / o_ms,
            "note": "synthetic N(0,1) x, 0.02*N(0,1) weights generated on the device; 3 interleaved rounds"}


def leg_tp_mlp_e2e(torch, tdg, args, pk):
    """The all-ranks TP MLP end to end through the public API with host
    buffers: every step uploads the 8 ranks' activations x_r from pinned host
    memory and downloads the 8 outputs; the weights stay resident (uploaded
    once, as in serving).  Consecutive steps overlap over two heaps (upload,
    compute and download streams)."""
    W, Ms, H, F = AG["W"], AG["Ms"], AG["K"], AG["N"]
    M = W * Ms
    a_off, g_off = 0, _align(Ms * H * 2)
    bu_off = _align(g_off + M * H * 2)
    c_off = _align(bu_off + H * F * 2)
    bd_off = _align(c_off + M * F * 2)
    s_off = _align(bd_off + F * H * 2)
    o_off = _align(s_off + tdg.gemm_rs_stage_bytes(W, M, H))
    gen = torch.Generator(device="cuda")
    gen.manual_seed(0)
    sets = []
    for _ in range(2):
        sym = tdg.Symm(W, _align(o_off + Ms * H * 2 + 1024), 65536)
        for r in range(W):
            sym.view(r, bu_off, (H, F), torch.bfloat16).copy_(torch.randn(H, F, device="cuda", generator=gen) * 0.02)
            sym.view(r, bd_off, (F, H), torch.bfloat16).copy_(torch.randn(F, H, device="cuda", generator=gen) * 0.02)
        sets.append(sym)
    cpu_gen = torch.Generator()
    cpu_gen.manual_seed(0)
    x_host = [torch.randn(Ms, H, generator=cpu_gen).to(torch.bfloat16).pin_memory() for _ in range(W)]
    out_host = [torch.empty(Ms, H, dtype=torch.bfloat16).pin_memory() for _ in range(W)]
    comp = torch.cuda.current_stream()
    up, down, side = torch.cuda.Stream(), torch.cuda.Stream(), torch.cuda.Stream()
    free = [torch.cuda.Event() for _ in sets]
    for e in free:
        e.record(comp)

    def step(i):
        sym = sets[i % 2]
        x_in, done = torch.cuda.Event(), torch.cuda.Event()
        up.wait_event(free[i % 2])
        with torch.cuda.stream(up):
            for r in range(W):
                sym.view(r, a_off, (Ms, H), torch.bfloat16).copy_(x_host[r], non_blocking=True)
            x_in.record(up)
        comp.wait_event(x_in)
        tdg.ag_gemm_all_ranks(sym, Ms, H, F, a_off, g_off, bu_off, c_off, mode="ce", side_stream=side)
        tdg.gemm_rs(sym, M, F, H, c_off, bd_off, s_off, o_off, mode="sm")
        done.record(comp)
        down.wait_event(done)
        with torch.cuda.stream(down):
            for o in range(W):
                out_host[o].copy_(sym.view(o, o_off, (Ms, H), torch.bfloat16), non_blocking=True)
            free[i % 2].record(down)

    for i in range(args.warmup):
        step(i)
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(comp)
    up.wait_event(e0)
    for i in range(args.warmup, args.warmup + args.steps):
        step(i)
    comp.wait_stream(up)
    comp.wait_stream(down)
    e1.record(comp)
    torch.cuda.synchronize()
    ms = e0.elapsed_time(e1) / args.steps
    for sym in sets:
        st = sym.status()
        if st["code"] != 0:
            raise RuntimeError(f"device fault in the all-ranks MLP end to end: {st}")
    del sets
    torch.cuda.empty_cache()
    flop = W * AG_FLOP + RS_FLOP
    return {"workload": "Qwen-32B TP MLP forward for all 8 logical ranks, end to end: x_r of every rank "
                        "uploaded and every out_o downloaded each step, weights resident",
            "value": flop / ms / 1e9, "unit": "TFLOP/s", "ms_per_step": ms,
            "h2d_bytes_per_step": W * Ms * H * 2, "d2h_bytes_per_step": W * Ms * H * 2,
            "frac_of_bf16_peak": flop / ms / 1e9 / pk["bf16"],
            "how": "two heaps, upload / compute / download streams; the AG-GEMM's copies on a side stream"}


def leg_rs_f32(torch, tdg, args, flush, pk):
    """The GEMM-RS of the step with fp32 partials (one rounding, twice the
    staging bytes), overlapped and serial, timed in interleaved rounds."""
    W, M, K, N = RS["W"], RS["M"], RS["K"], RS["N"]
    a_off, b_off = 0, _align(M * K * 2)
    s_off = _align(b_off + K * N * 2)
    o_off = _align(s_off + 2 * tdg.gemm_rs_stage_bytes(W, M, N))
    sym = tdg.Symm(W, _align(o_off + (M // W) * N * 2 + 1024), 65536)
    g = torch.Generator(device="cuda")
    g.manual_seed(0)
    for r in range(W):
        sym.view(r, a_off, (M, K), torch.bfloat16).copy_(torch.randn(M, K, device="cuda", generator=g))
        sym.view(r, b_off, (K, N), torch.bfloat16).copy_(torch.randn(K, N, device="cuda", generator=g) * 0.02)
    call = lambda mode: (lambda: tdg.gemm_rs(sym, M, K, N, a_off, b_off, s_off, o_off, mode=mode,
                                             partial_f32=True))
    iv = interleaved_steps(torch, {"sm": [call("sm")], "serial": [call("serial")]}, 3,
                           max(4, args.steps // 5), flush)
    st = sym.status()
    if st["code"] != 0:
        raise RuntimeError(f"device fault in GEMM-RS with fp32 partials: {st}")
    del sym
    torch.cuda.empty_cache()
    return {"workload": "the step's GEMM-RS (W=8, A_r 8192x3200, B_r 3200x5120) with fp32 partials",
            "sm_ms": iv["sm"][0], "sm_tflops": RS_FLOP / iv["sm"][0] / 1e9,
            "serial_ms": iv["serial"][0], "serial_tflops": RS_FLOP / iv["serial"][0] / 1e9,
            "note": "synthetic N(0,1) A_r, 0.02*N(0,1) B_r generated on the device; modes in 3 interleaved rounds"}


def leg_ring(torch, tdg, synth, args, flush, pk):
    extras = {}
    # ring AllReduce over the 8 logical ranks, 32 Mi float32 per rank
    torch.manual_seed(0)
    W, cnt = 8, 32 * 1024 * 1024
    rsym = tdg.Symm(W, _align(cnt * 4 + tdg.allreduce_recv_bytes(W, cnt) + 2048), 65536)
    for r in range(W):
        rsym.view(r, 0, (cnt,), torch.float32).normal_()
    recv_off = _align(cnt * 4)
    aparts = timed_steps(torch, [lambda: tdg.allreduce(rsym, cnt, 0, recv_off)], args.steps, args.warmup, flush)
    a_ms = statistics.mean(aparts[0])
    st = rsym.status()
    if st["code"] != 0:
        raise RuntimeError(f"device fault in the ring AllReduce: {st}")
    hbm = (5 * W - 4) * cnt * 4   # bytes the ring reads and writes in HBM
    extras["ring_allreduce"] = {
        "workload": "8 logical ranks x 32 Mi float32, ring reduce-scatter + all-gather, 64 Ki-element tiles",
        "ms": a_ms, "hbm_bytes": hbm, "gbs": hbm / a_ms / 1e6, "frac_of_hbm": hbm / a_ms / 1e6 / pk["hbm"],
        "busbw_gbs": 2 * (W - 1) / W * cnt * 4 / a_ms / 1e6}
    del rsym
    torch.cuda.empty_cache()
    return extras["ring_allreduce"]


def leg_ag_config(torch, tdg, synth, args, flush, pk, W, Ms, K, N, dist, workload, modes=("ce", "sm"),
                  variants=None):
    """One AllGather+GEMM config on its own: each overlapped schedule against
    the serial twin (copy launch, then GEMM launch), TFLOP/s and fraction of
    the measured bf16 peak.  `variants` maps a name to (mode, extra args);
    by default one variant per mode."""
    inp = synth.ag_inputs(W, Ms, K, N, dist, seed=0)
    g_off = _align(Ms * K * 2)
    ll_off = _align(g_off + W * Ms * K * 2)    # LL words: 4 bytes per element
    ll_bytes = W * Ms * K * 4 if "ll" in modes else 0
    sym = tdg.Symm(W, _align(ll_off + ll_bytes + 1024), 65536)
    for r in range(W):
        sym.view(r, 0, (Ms, K), torch.bfloat16).copy_(_dev_bf16(inp.shards[r], torch))
    B = _dev_bf16(inp.B, torch)
    C = torch.empty((W * Ms, N), dtype=torch.bfloat16, device="cuda")
    del inp
    side = torch.cuda.Stream()
    flop = 2 * W * Ms * K * N
    if variants is None:
        variants = {m: (m, {}) for m in modes}
    variants = dict({"serial": ("serial", {})}, **variants)

    def call(mode, kw):
        return lambda: tdg.ag_gemm(sym, 0, Ms, K, N, 0, g_off, B, C, mode=mode, ll_off=ll_off,
                                   side_stream=side if mode == "ce" else None, **kw)
    res = {"workload": workload, "note": f"schedules timed in 5 interleaved rounds (same clock state)"}
    for name, (mode, kw) in variants.items():   # warm every schedule once
        timed_steps(torch, [call(mode, kw)], 1, args.warmup, flush)
    iv = interleaved_steps(torch, {n: [call(m, kw)] for n, (m, kw) in variants.items()}, 5,
                           max(4, args.steps // 5), flush)
    times = {n: v[0] for n, v in iv.items()}
    for name in variants:
        res[f"{name}_ms"] = times[name]
        res[f"{name}_tflops"] = flop / times[name] / 1e9
        res[f"{name}_frac_of_bf16_peak"] = flop / times[name] / 1e9 / pk["bf16"]
        if name != "serial":
            res[f"{name}_overlap_gain_vs_serial"] = times["serial"] / times[name]
    st = sym.status()
    if st["code"] != 0:
        raise RuntimeError(f"device fault in {workload}: {st}")
    del sym, B, C
    torch.cuda.empty_cache()
    return res


# push and pull, copy engine and producer CTAs, for the AG configs
AG_SCHEDULES = {"ce": ("ce", {}), "ce_push": ("ce", dict(push=True)), "sm": ("sm", {}),
                "sm_push": ("sm", dict(push=True))}


def leg_ag_copy(torch, tdg, args, flush, pk):
    """The AllGather of the Qwen-32B up-projection alone (N = 0: gathered
    buffer and flags, no GEMM): producer CTAs (the SERIAL copy launch on a
    given number of CTAs) and the copy engine.  Bytes moved = the 8 shards
    (84 MB), each read once and written once."""
    W, Ms, K = AG["W"], AG["Ms"], AG["K"]
    g_off = _align(Ms * K * 2)
    sym = tdg.Symm(W, _align(g_off + W * Ms * K * 2 + 1024), 65536)
    g = torch.Generator(device="cuda")
    g.manual_seed(0)
    for r in range(W):
        sym.view(r, 0, (Ms, K), torch.bfloat16).copy_(torch.randn(Ms, K, device="cuda", generator=g))
    side = torch.cuda.Stream()
    moved = W * Ms * K * 2
    res = {"workload": "AllGather of 8 shards of 1024x5120 bf16 (84 MB moved; read + write 168 MB), no GEMM",
           "bytes_moved": moved}
    for n in (1, 16, 0):
        ms = statistics.mean(timed_steps(torch, [lambda: tdg.ag_gemm(sym, 0, Ms, K, 0, 0, g_off, None, None,
                                                                     mode="serial", producers=n)],
                                         max(4, args.steps // 5), args.warmup, flush)[0])
        ctas = n or sms_of(torch)
        res[f"producers_{n or 'all'}_gbs"] = moved / ms / 1e6
        res[f"producers_{n or 'all'}_gbs_per_cta"] = moved / ms / 1e6 / ctas
        res[f"producers_{n or 'all'}_rw_frac_of_hbm"] = 2 * moved / ms / 1e6 / pk["hbm"]
    ms = statistics.mean(timed_steps(torch, [lambda: tdg.ag_gemm(sym, 0, Ms, K, 0, 0, g_off, None, None,
                                                                 mode="ce", side_stream=side)],
                                     max(4, args.steps // 5), args.warmup, flush)[0])
    res["copy_engine_gbs"] = moved / ms / 1e6
    res["note"] = ("an SM writes to memory at about 63 GB/s at most (TMA bulk or plain stores), so one producer "
                   "CTA moves about 50 GB/s")
    st = sym.status()
    if st["code"] != 0:
        raise RuntimeError(f"device fault in the AllGather alone: {st}")
    del sym
    torch.cuda.empty_cache()
    return res


def sms_of(torch):
    return torch.cuda.get_device_properties(0).multi_processor_count


def leg_autotune(torch, tdg, args, flush, pk):
    """The distributed autotuner on the step's two operations (one process:
    no ranks to agree with): every candidate schedule timed through the C ABI,
    the best one reported beside the library's default."""
    from tile_centric_comm_gb300 import autotune
    out = {}
    W, Ms, K, N = AG["W"], AG["Ms"], AG["K"], AG["N"]
    g_off = _align(Ms * K * 2)
    sym = tdg.Symm(W, _align(g_off + W * Ms * K * 2 + 1024), 65536)
    g = torch.Generator(device="cuda")
    g.manual_seed(0)
    for r in range(W):
        sym.view(r, 0, (Ms, K), torch.bfloat16).copy_(torch.randn(Ms, K, device="cuda", generator=g))
    B = (torch.randn(K, N, device="cuda", generator=g) * 0.02).to(torch.bfloat16)
    C = torch.empty((W * Ms, N), dtype=torch.bfloat16, device="cuda")
    side = torch.cuda.Stream()
    cands = autotune.ag_candidates(W * Ms, Ms, producers=(0,), source_orders=(0,))

    def run(cfg):
        tdg.ag_gemm(sym, 0, Ms, K, N, 0, g_off, B, C, side_stream=side, **cfg)
    best, table = autotune.tune(("ag", W, Ms, K, N), cands, run, warmup=2, iters=20, flush=flush.zero_,
                                use_cache=False, pause=0.2)
    # the first candidate is the library's default schedule in CE mode (pull,
    # the default cluster shape and stage count)
    flop = 2 * W * Ms * K * N
    out["ag_qwen32b_up"] = {"candidates": len(cands), "best": best,
                            "best_tflops": flop / min(r["ms"] for r in table) / 1e9,
                            "default": table[0]["cfg"], "default_tflops": flop / table[0]["ms"] / 1e9,
                            "table": [dict(r["cfg"], tflops=round(flop / r["ms"] / 1e9, 1)) for r in table]}
    del sym, B, C
    torch.cuda.empty_cache()
    W, M, K, N = RS["W"], RS["M"], RS["K"], RS["N"]
    a_off, b_off = 0, _align(M * K * 2)
    s_off = _align(b_off + K * N * 2)
    o_off = _align(s_off + tdg.gemm_rs_stage_bytes(W, M, N))
    sym = tdg.Symm(W, _align(o_off + (M // W) * N * 2 + 1024), 65536)
    for r in range(W):
        sym.view(r, a_off, (M, K), torch.bfloat16).copy_(torch.randn(M, K, device="cuda", generator=g))
        sym.view(r, b_off, (K, N), torch.bfloat16).copy_(torch.randn(K, N, device="cuda", generator=g) * 0.02)
    rc = autotune.rs_candidates(W, M // W, orders=(0,), spares=(0, 2))

    def run_rs(cfg):
        tdg.gemm_rs(sym, M, K, N, a_off, b_off, s_off, o_off, **cfg)
    best, table = autotune.tune(("rs", W, M, K, N), rc, run_rs, warmup=2, iters=50, flush=flush.zero_,
                                use_cache=False, pause=0.2)
    dflt = [r["ms"] for r in table if r["cfg"] == dict(owner_block=W, order=0, cluster=4, stages=0)]
    out["gemm_rs_qwen32b_down"] = {"candidates": len(rc), "best": best,
                                   "best_tflops": RS_FLOP / min(r["ms"] for r in table) / 1e9,
                                   "default": dict(owner_block=W, order=0, cluster=4, stages=0),
                                   "default_tflops": RS_FLOP / dflt[0] / 1e9 if dflt else None,
                                   "table": [dict(r["cfg"], tflops=round(RS_FLOP / r["ms"] / 1e9, 1))
                                             for r in table]}
    st = sym.status()
    if st["code"] != 0:
        raise RuntimeError(f"device fault in the autotune leg: {st}")
    del sym
    torch.cuda.empty_cache()
    out["note"] = ("each candidate timed as a burst of back-to-back calls (20 AG-GEMM / 50 GEMM-RS, L2 flushed "
                   "before each) after a 0.2 s idle pause; 3 rounds with the order rotated, median per candidate")
    return out


def leg_flash(torch, tdg, synth, args, flush, pk):
    extras = {}
    # distributed flash decoding: 4 sequences x 64 heads (8 kv heads, d 128),
    # 128 Ki cached tokens split over the 8 logical ranks
    W, Bq, Hq, Hkv, D, S = 8, 4, 64, 8, 128, 131072
    kvb = Bq * Hkv * (S // W) * D * 2
    part = tdg.flash_decode_part_bytes(W, Bq, Hq, D, S)
    fsym = tdg.Symm(W, _align(2 * _align(kvb) + part + 2048), 4096)
    for r in range(W):
        fsym.view(r, 0, (kvb // 2,), torch.bfloat16).normal_()
        fsym.view(r, _align(kvb), (kvb // 2,), torch.bfloat16).normal_()
    qf = torch.randn((Bq, Hq, D), device="cuda").to(torch.bfloat16)
    of = torch.empty_like(qf)
    fparts = timed_steps(torch, [lambda: tdg.flash_decode(fsym, Bq, Hq, Hkv, D, S, 0, _align(kvb),
                                                          2 * _align(kvb), qf, of)],
                         args.steps, args.warmup, flush)
    f_ms = statistics.mean(fparts[0])
    st = fsym.status()
    if st["code"] != 0:
        raise RuntimeError(f"device fault in flash decoding: {st}")
    fbytes = 2 * kvb * W   # every cached K and V byte is read once
    extras["flash_decode"] = {
        "workload": "4 x 64 heads (8 kv heads, d 128), 128 Ki cached tokens over 8 logical ranks",
        "ms": f_ms, "kv_bytes": fbytes, "gbs": fbytes / f_ms / 1e6, "frac_of_hbm": fbytes / f_ms / 1e6 / pk["hbm"]}
    del fsym, qf, of
    torch.cuda.empty_cache()
    return extras["flash_decode"]


def multi_gpu_unavailable(args, rank, n):
    """--gpus N > 1: this path has no multi-GPU form; rank 0 says so in one
    line, and nothing touches a GPU."""
    if rank != 0:
        return
    print(json.dumps({"impl": "tdg", "metric": "AG-GEMM+GEMM-RS TFLOP/s (qwen32b_mlp_tp8)", "n_gpus": n,
                      "steps": args.steps, "warmup": args.warmup,
                      "unavailable": "the path runs on one GPU (W logical ranks in one device allocation; "
                                     "its GEMMs multicast B slices inside a cluster, from this GPU's own "
                                     "memory), so there is no run on several GPUs"}), flush=True)


def main():
    args = parse()
    rank, world, local = dist_env()
    if args.ag_shape:
        if args.only not in ("ag", "library"):
            raise SystemExit("--ag-shape needs --only ag or --only library")
        W, Ms, K, N = (int(x) for x in args.ag_shape.split(","))
        AG.update(W=W, Ms=Ms, K=K, N=N)
    if args.impl == "reference":
        run_reference(args, rank)
        return
    if world > 1 or args.gpus > 1:
        multi_gpu_unavailable(args, rank, max(world, args.gpus))
        return
    import torch
    from tile_centric_comm_gb300 import synth, tdg
    torch.cuda.set_device(local)
    sms, supported = tdg.device_info()
    if not supported:
        raise SystemExit("libtdg kernels need an sm_103 device")
    pk = peaks()
    flush = torch.empty(256 * 1024 * 1024 // 4, dtype=torch.int32, device="cuda")
    if args.only == "library":
        # context only, not part of the path: the library GEMM on the gathered shape
        M, K, N = AG["W"] * AG["Ms"], AG["K"], AG["N"]
        torch.manual_seed(0)
        a = torch.randn(M, K, device="cuda").to(torch.bfloat16)
        b = (torch.randn(K, N, device="cuda") * 0.02).to(torch.bfloat16)
        c = torch.empty(M, N, device="cuda", dtype=torch.bfloat16)
        with Clocks(local) as clk:
            lp = timed_steps(torch, [lambda: torch.matmul(a, b, out=c)], args.steps, args.warmup, flush)
        ms = statistics.mean(lp[0])
        if rank == 0:
            print(json.dumps({"metric": "library GEMM TFLOP/s (context)", "value": 2 * M * K * N / ms / 1e9,
                              "unit": "TFLOP/s", "ms": ms, "shape": [M, K, N], "steps": args.steps,
                              "warmup": args.warmup, "clocks": clk.summary()}), flush=True)
        return
    if args.only == "ag_all":
        with Clocks(local) as clk:
            res = leg_ag_all(torch, tdg, args, flush, pk)
        if rank == 0:
            key = "serial" if "ce_tflops" not in res else "ce"
            print(json.dumps({"metric": f"all-ranks AG-GEMM TFLOP/s ({key})", "value": res[f"{key}_tflops"],
                              "unit": "TFLOP/s", "n_gpus": 1, "steps": args.steps, "warmup": args.warmup,
                              "higher_is_better": True, "dtype": "bf16",
                              "roofline": {"bound": "tensor", "achieved": res[f"{key}_tflops"], "peak": pk["bf16"],
                                           "unit": "TFLOP/s", "frac": res[f"{key}_tflops"] / pk["bf16"]},
                              "clocks": clk.summary(), "detail": res}), flush=True)
        return
    if args.only == "copy":
        # the AllGather alone (N = 0): the SERIAL copy launch on --producers CTAs
        # (0 = every SM), or the copy engine with --mode ce
        W, Ms, K = AG["W"], AG["Ms"], AG["K"]
        g_off = _align(Ms * K * 2)
        sym = tdg.Symm(W, _align(g_off + W * Ms * K * 2 + 1024), 65536)
        gen = torch.Generator(device="cuda")
        gen.manual_seed(0)
        for r in range(W):
            sym.view(r, 0, (Ms, K), torch.bfloat16).copy_(torch.randn(Ms, K, device="cuda", generator=gen))
        side = torch.cuda.Stream()
        mode = "ce" if args.mode == "ce" else "serial"
        with Clocks(local) as clk:
            cp = timed_steps(torch, [lambda: tdg.ag_gemm(sym, 0, Ms, K, 0, 0, g_off, None, None, mode=mode,
                                                         producers=args.producers,
                                                         side_stream=side if mode == "ce" else None)],
                             args.steps, args.warmup, flush)
        ms = statistics.mean(cp[0])
        moved = W * Ms * K * 2
        if sym.status()["code"] != 0:
            raise RuntimeError(f"device fault in the AllGather alone: {sym.status()}")
        ctas = args.producers or sms
        print(json.dumps({"metric": f"AllGather alone GB/s moved ({mode})", "value": moved / ms / 1e6,
                          "unit": "GB/s", "n_gpus": 1, "steps": args.steps, "warmup": args.warmup,
                          "per_cta_gbs": moved / ms / 1e6 / ctas if mode == "serial" else None,
                          "roofline": {"bound": "hbm", "achieved": 2 * moved / ms / 1e6, "peak": pk["hbm"],
                                       "unit": "GB/s", "frac": 2 * moved / ms / 1e6 / pk["hbm"],
                                       "what": "read + write bytes"},
                          "clocks": clk.summary()}), flush=True)
        return
    if args.only in ("moe", "ring", "flash"):
        leg = {"moe": leg_moe, "ring": leg_ring, "flash": leg_flash}[args.only]
        with Clocks(local) as clk:
            res = leg(torch, tdg, synth, args, flush, pk)
        if rank == 0:
            print(json.dumps({"metric": f"{args.only} GB/s", "value": res["gbs"], "unit": "GB/s",
                              "n_gpus": 1, "steps": args.steps, "warmup": args.warmup,
                              "higher_is_better": True, "dtype": "bf16" if args.only != "ring" else "f32",
                              "roofline": {"bound": "hbm", "achieved": res["gbs"], "peak": pk["hbm"],
                                           "unit": "GB/s", "frac": res["frac_of_hbm"]},
                              "clocks": clk.summary(), "detail": res}), flush=True)
        return
    mlp = MLP(torch, tdg, synth, args.mode, args.producers, args.signal_rows)
    torch.cuda.synchronize()

    # --only rs --mode serial times the serial twin of the GEMM-RS (for captures)
    rs_mode = "serial" if (args.only == "rs" and args.mode == "serial") else "sm"
    fns = [lambda: mlp.ag_call(), lambda: mlp.rs_call(rs_mode)]
    if args.only == "ag":
        fns = fns[:1]
    elif args.only == "rs":
        fns = fns[1:]

    def barrier():
        torch.cuda.synchronize()

    barrier()
    with Clocks(local) as clk:
        parts = timed_steps(torch, fns, args.steps, args.warmup, flush)
    barrier()
    mlp.check_status()
    clocks = clk.summary()
    step_ms = [sum(p[i] for p in parts) for i in range(args.steps)]
    total_ms = sum(step_ms)
    ms_per_step = total_ms / args.steps
    ag_flop = 2 * AG["W"] * AG["Ms"] * AG["K"] * AG["N"]
    flop = (ag_flop if args.only != "rs" else 0) + (RS_FLOP if args.only != "ag" else 0)
    value = flop * args.steps / (total_ms * 1e-3) / 1e12
    launches = 2 * args.steps if not args.only else args.steps
    ag_ms = statistics.mean(parts[0]) if args.only != "rs" else None
    rs_ms = statistics.mean(parts[-1]) if args.only != "ag" else None

    extras = {}
    e2e = None
    cpu = None
    if not args.no_extras and not args.only:
        # the serial composition (same kernels, copy -> GEMM -> reduce) and the
        # other AG mode, timed in rounds interleaved with the overlapped step
        # so that every variant sees the same clock
        other = "sm" if args.mode != "sm" else "ce"
        iv = interleaved_steps(torch, {
            "overlapped": [lambda: mlp.ag_call(), lambda: mlp.rs_call("sm")],
            "serial": [lambda: mlp.ag_call("serial"), lambda: mlp.rs_call("serial")],
            "other": [lambda: mlp.ag_call(other)]}, 5, max(4, args.steps // 5), flush)
        o_ag, o_rs = iv["overlapped"]
        s_ag, s_rs = iv["serial"]
        c_ag = iv["other"][0]
        extras["ag_gemm"] = {"ms": ag_ms, "tflops": AG_FLOP / ag_ms / 1e9,
                             "frac_of_bf16_peak": AG_FLOP / ag_ms / 1e9 / pk["bf16"],
                             "interleaved_ms": o_ag, "serial_ms": s_ag,
                             "overlap_gain_vs_serial": s_ag / o_ag}
        extras["gemm_rs"] = {"ms": rs_ms, "tflops": RS_FLOP / rs_ms / 1e9,
                             "frac_of_bf16_peak": RS_FLOP / rs_ms / 1e9 / pk["bf16"],
                             "interleaved_ms": o_rs, "serial_ms": s_rs,
                             "overlap_gain_vs_serial": s_rs / o_rs}
        extras["overlap_gain_vs_serial"] = (s_ag + s_rs) / (o_ag + o_rs)
        extras["overlap_gain_note"] = ("overlapped and serial steps timed in 5 interleaved rounds "
                                       "(same clock state); 'ms' is the main timed loop")
        extras["ag_gemm"]["mode"] = args.mode
        extras["ag_gemm"][f"{other}_mode_ms"] = c_ag
        extras["ag_gemm"][f"{other}_mode_tflops"] = AG_FLOP / c_ag / 1e9
        extras["ag_gemm"][f"{other}_mode_overlap_gain_vs_serial"] = s_ag / c_ag
        mlp.check_status()
        # end to end through the public API with host buffers: one step at a
        # time, then consecutive steps overlapped over two buffer sets
        barrier()
        eparts = timed_steps(torch, [mlp.e2e_step], args.steps, args.warmup, flush)
        e_one = statistics.mean(eparts[0])
        mlp2 = mlp.twin()
        e_ms = mlp.e2e_pipelined([mlp, mlp2], args.steps, args.warmup)
        # a serving step: the weights (B, B_r) stay resident (uploaded once,
        # before the timed steps); the activations cross every step
        for S in (mlp, mlp2):
            S.upload_ag()
            S.upload_rs()
        torch.cuda.synchronize()
        e_w = mlp.e2e_pipelined([mlp, mlp2], args.steps, args.warmup, weights=False)
        mlp2.check_status()
        del mlp2
        e2e = {"value": STEP_FLOP / e_ms / 1e9, "unit": "TFLOP/s",
               "h2d_bytes_per_step": mlp.h2d_bytes, "d2h_bytes_per_step": mlp.d2h_bytes,
               "ms_per_step": e_ms,
               "how": "consecutive steps overlapped over two device buffer sets (upload, compute and "
                      "download streams); every step copies all its inputs H2D and both outputs D2H",
               "one_step_at_a_time": {"value": STEP_FLOP / e_one / 1e9, "ms_per_step": e_one},
               "weights_resident": {"value": STEP_FLOP / e_w / 1e9, "ms_per_step": e_w,
                                    "h2d_bytes_per_step": mlp.h2d_act_bytes,
                                    "what": "activations (AG shards, RS A_r) H2D every step, outputs D2H; "
                                            "B and B_r uploaded once before the timed steps"}}
        mlp.check_status()
        # context: the library GEMM (cuBLAS through torch.matmul) on the same
        # shapes, with no communication at all (not part of the path)
        a_cat = mlp.ag.view(0, mlp.ag_g_off, (AG["W"] * AG["Ms"], AG["K"]), torch.bfloat16)
        b_rs = [mlp.rs.view(r, mlp.rs_b_off, (RS["K"], RS["N"]), torch.bfloat16) for r in range(RS["W"])]
        a_rs = [mlp.rs.view(r, mlp.rs_a_off, (RS["M"], RS["K"]), torch.bfloat16) for r in range(RS["W"])]
        c_rs = torch.empty((RS["M"], RS["N"]), dtype=torch.bfloat16, device="cuda")
        lparts = timed_steps(torch, [lambda: torch.matmul(a_cat, mlp.ag_B, out=mlp.ag_C),
                                     lambda: [torch.matmul(a_rs[r], b_rs[r], out=c_rs) for r in range(RS["W"])]],
                             args.steps, args.warmup, flush)
        l_ag, l_rs = statistics.mean(lparts[0]), statistics.mean(lparts[1])
        extras["library_gemm_context"] = {
            "what": "torch.matmul (cuBLAS) on the same GEMM shapes, no AllGather / ReduceScatter",
            "ag_shape_tflops": AG_FLOP / l_ag / 1e9, "rs_shapes_tflops": RS_FLOP / l_rs / 1e9}
        del mlp, a_cat, b_rs, a_rs, c_rs
        torch.cuda.empty_cache()
        extras["ag_qwen32b_up_schedules"] = leg_ag_config(
            torch, tdg, synth, args, flush, pk, 8, 1024, 5120, 3200, "normal",
            "AG-GEMM Qwen-32B up: W=8, A_r 1024x5120, B 5120x3200, pull and push", variants=AG_SCHEDULES)
        extras["ag_llama70b_gateup"] = leg_ag_config(
            torch, tdg, synth, args, flush, pk, 8, 2048, 8192, 7168, "normal",
            "AG-GEMM Llama-3-70B gate+up: W=8, A_r 2048x8192, B 8192x7168, pull and push",
            variants=AG_SCHEDULES)
        extras["ag_copy_alone_qwen32b"] = leg_ag_copy(torch, tdg, args, flush, pk)
        extras["autotune"] = leg_autotune(torch, tdg, args, flush, pk)
        extras["ag_tiny"] = leg_ag_config(
            torch, tdg, synth, args, flush, pk, 2, 64, 256, 128, "int2",
            "AG-GEMM tiny: W=2, A_r 64x256, B 256x128, integers (latency bound)", modes=("ce", "sm", "ll"))
        extras["ag_all_ranks_qwen32b_up"] = leg_ag_all(torch, tdg, args, flush, pk)
        extras["tp_mlp_all_ranks_qwen32b"] = leg_tp_mlp_all(torch, tdg, args, flush, pk)
        extras["tp_mlp_all_ranks_qwen32b"]["e2e"] = leg_tp_mlp_e2e(torch, tdg, args, pk)
        extras["gemm_rs_f32_partials"] = leg_rs_f32(torch, tdg, args, flush, pk)
        extras["moe_dispatch_combine"] = leg_moe(torch, tdg, synth, args, flush, pk)
        extras["ring_allreduce"] = leg_ring(torch, tdg, synth, args, flush, pk)
        extras["flash_decode"] = leg_flash(torch, tdg, synth, args, flush, pk)
        if rank == 0 and not args.no_cpu:
            r, s, desc = cpu_oracle_rate()
            cpu = {"value": r, "unit": "TFLOP/s", "cores": omp_threads(), "kind": "oracle", "sample": desc,
                   "seconds": s}

    # roofline of the dominant kernel (the GEMM-RS persistent GEMM, one launch per call)
    dom_ms = rs_ms if rs_ms is not None else ag_ms
    dom_flop = RS_FLOP if rs_ms is not None else ag_flop
    achieved = dom_flop / dom_ms / 1e9
    roofline = {"kernel": "rs_gemm_kernel" if rs_ms is not None else "ag_gemm_kernel",
                "bound": "tensor", "achieved": achieved, "peak": pk["bf16"], "unit": "TFLOP/s",
                "frac": achieved / pk["bf16"],
                "traffic": (RS_TRAFFIC["bytes"] if rs_ms is not None and rs_sources_hash() == RS_TRAFFIC["sources"]
                            else None),
                "traffic_unit": "bytes per launch",
                "algorithmic_bytes": 1_352_000_000 + 755_000_000 if rs_ms is not None else None,
                "peak_kind": f"bf16 dense burst, {pk['src']}",
                "frac_of_sustained": achieved / pk["bf16_sus"]}
    line = {"metric": "AG-GEMM+GEMM-RS TFLOP/s (qwen32b_mlp_tp8)", "value": value, "unit": "TFLOP/s",
            "n_gpus": 1, "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_per_step,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
            "data": "synthetic",
            "config": {"workload": WORKLOAD, "l2": "flushed before every step (256 MB write)",
                       "ag_mode": args.mode, "rs_mode": "sm (push + last-arriver reduction)",
                       "producers": (args.producers or "library default") if args.mode == "sm" else None,
                       "sm_count": sms,
                       "parallelism": "one GPU, 8 logical ranks (symmetric regions of one allocation)"},
            "roofline": roofline, "cpu_baseline": cpu, "e2e": e2e, "gpu_launches": launches,
            "clocks": clocks, "parts": extras}
    print(json.dumps(line), flush=True)


if __name__ == "__main__":
    main()
