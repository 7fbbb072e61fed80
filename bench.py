#!/usr/bin/env python3
"""Benchmark of the CODA GEMM-epilogue hot path on GB300.

Workload (default): the GEMM+RoPE QKV projection, X[4096,4096] x W[4096,12288]
bf16, RoPE on the Q and K heads (head_dim 128, theta 10000, positions
0..4095, adjacent pairs), forward and backward. One step is

  QKV = rope(X W)                      coda_gemm_rope       (fused epilogue)
  dP  = rope^T(A B)                    coda_gemm_rope_bwd   (fused epilogue;
                                       A B stands in for the upstream gradient)
  dX  = dP W^T,  dW = X^T dP           coda_gemm x 2        (plain GEMMs)

4 x 2 M N K = 1.649 TFLOP per step. The unfused comparison runs the same GEMMs
with the identity epilogue plus separate in-place RoPE kernels.

Prints one JSON line (rank 0). `--impl reference` times the float64 CPU oracle
on a bounded sample of the same workload instead. Multi-GPU: replicas only
(every rank runs the whole workload; no collective on the data path).
"""
from __future__ import annotations

import argparse
import hashlib
import re
import json
import os
import subprocess
import sys
import tempfile
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "fused GEMM+epilogue TFLOP/s (% BF16 TC peak) and speedup vs unfused path"
WL = dict(name="rope_qkv_4096", M=4096, K=4096, N=12288, head_dim=128, theta=10000.0, S=4096, rope_cols=8192)
FLOPS_PER_GEMM = 2.0 * WL["M"] * WL["N"] * WL["K"]
FLOPS_PER_STEP = 4 * FLOPS_PER_GEMM


def parse():
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=["coda", "reference"], default="coda")
    ap.add_argument("--no-cpu-baseline", action="store_true", help="skip the CPU oracle leg")
    ap.add_argument("--no-configs", action="store_true",
                    help="skip the per-config fused/unfused entries of the default run")
    ap.add_argument("--suite", action="store_true",
                    help="time every fused operator against its unfused pair on all five workloads "
                         "(one JSON line per operator) instead of the headline step")
    ap.add_argument("--reps", type=int, default=50, help="timed repetitions per operator in --suite (at least)")
    ap.add_argument("--min-seconds", type=float, default=1.0,
                    help="with --suite: raise each entry's repetitions until its timed region lasts this long")
    ap.add_argument("--only", default=None,
                    help="with --suite: run one workload (rmsnorm_chain_tiny, rmsnorm_chain_8192, rope_qkv_4096, "
                         "swiglu_up_4096, lm_head_ce_8192, block_d2048, block_d4096, block_d8192, fp8_rope_qkv_4096, "
                         "fp8_swiglu_up_4096, fp8_lm_head_ce_8192, ce_bwd_f2_bound, gemm_vs_cublas)")
    return ap.parse_args()


def config():
    return {"workload": "GEMM+RoPE QKV projection fwd+bwd: X[4096,4096] x W[4096,12288] bf16, "
                        "RoPE on Q,K (head_dim 128, theta 1e4, positions 0..4095), dX/dW GEMMs",
            "M": WL["M"], "K": WL["K"], "N": WL["N"], "head_dim": WL["head_dim"], "rope_cols": WL["rope_cols"],
            "flops_per_step": FLOPS_PER_STEP, "l2": "flushed between steps (256 MiB write), inputs 256 MiB"}


# ---------------------------------------------------------------- CPU oracle leg

def oracle_sample(inputs, rows):
    """The float64 oracle on the first `rows` tokens of each of the step's four
    GEMMs; returns (seconds, flops)."""
    import oracle as O
    pos = np.arange(rows) % WL["S"]
    X = O.bf16(inputs["X"][:rows])
    A = O.bf16(inputs["A"][:rows])
    W = inputs["_W64"]
    B = inputs["_B64"]
    t0 = time.perf_counter()
    O.gemm_rope(X, W, pos, WL["head_dim"], WL["theta"], WL["rope_cols"])
    dP = O.gemm_rope_bwd(A, B, pos, WL["head_dim"], WL["theta"], WL["rope_cols"])
    O.matmul(dP, W.T)
    O.matmul(X.T, dP)
    return time.perf_counter() - t0, 4 * 2.0 * rows * WL["K"] * WL["N"]


def oracle_prepare(inputs):
    import oracle as O
    inputs["_W64"] = O.bf16(inputs["W"])
    inputs["_B64"] = O.bf16(inputs["B"])


def calibrate_rows(inputs, target_s):
    t, _ = oracle_sample(inputs, 32)
    rows = int(32 * target_s / max(t, 1e-3))
    return max(32, min(WL["M"], rows // 32 * 32))


def cores():
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count()


def cpu_baseline(inputs):
    oracle_prepare(inputs)
    rows = calibrate_rows(inputs, 12.0)
    t, fl = oracle_sample(inputs, rows)
    return {"value": fl / t / 1e12, "unit": "TFLOP/s", "cores": cores(), "kind": "oracle",
            "sample": f"first {rows} of 4096 token rows of each of the 4 GEMMs of one step (float64 NumPy, "
                      f"{t:.1f} s)"}


# ---------------------------------------------------------------- GPU helpers

class Clocks:
    """nvidia-smi sampler running during the timed regions."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        self.index = index
        self.f = tempfile.NamedTemporaryFile("w+", suffix=".csv", delete=False)
        self.p = None

    def start(self):
        try:
            self.p = subprocess.Popen(["nvidia-smi", f"--id={self.index}", f"--query-gpu={self.FIELDS}",
                                       "--format=csv,noheader,nounits", "-lms", "100"],
                                      stdout=self.f, stderr=subprocess.DEVNULL)
        except OSError:
            self.p = None

    def stop(self):
        if self.p is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.p.terminate()
        self.p.wait(timeout=10)
        self.f.flush()
        rows = []
        for line in open(self.f.name):
            parts = [x.strip() for x in line.split(",")]
            if len(parts) >= 9 and parts[1].replace(".", "").isdigit():
                rows.append(parts)
        os.unlink(self.f.name)
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"], "samples": 0}
        sm = np.array([float(r[1]) for r in rows])
        mx = float(rows[0][2])
        load = sm[sm >= 0.5 * mx] if np.any(sm >= 0.5 * mx) else sm
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if r[5 + i].lower().startswith("active")})
        return {"sm_mhz": float(np.median(load)), "sm_max_mhz": mx, "reasons": reasons, "samples": len(rows),
                "power_w_max": max(float(r[3]) for r in rows if r[3].replace(".", "").isdigit())
                if any(r[3].replace(".", "").isdigit() for r in rows) else None}


class NvmlClocks:
    """SM clock and clock-event reasons polled through NVML (ctypes, read-only
    queries) every few milliseconds on a host thread, for timed regions too
    short for the nvidia-smi sampler. Unavailable NVML leaves it empty."""

    REASONS = {0x4: "sw_power_cap", 0x8: "hw_slowdown", 0x20: "sw_thermal_slowdown",
               0x40: "hw_thermal_slowdown", 0x80: "hw_power_brake_slowdown"}

    def __init__(self, device_index):
        import ctypes
        import threading
        self.samples, self.reasons, self.h, self.nv = [], 0, None, None
        self._stop = threading.Event()
        self._t = None
        try:
            nv = ctypes.CDLL("libnvidia-ml.so.1")
            if nv.nvmlInit_v2() != 0:
                return
            import torch
            pr = torch.cuda.get_device_properties(device_index)
            h = ctypes.c_void_p()
            bus = f"{pr.pci_domain_id:08X}:{pr.pci_bus_id:02X}:{pr.pci_device_id:02X}.0".encode()
            if nv.nvmlDeviceGetHandleByPciBusId_v2(ctypes.c_char_p(bus), ctypes.byref(h)) != 0:
                return
            self.nv, self.h = nv, h
        except (OSError, AttributeError, RuntimeError):
            self.nv = None

    def _poll(self):
        import ctypes
        mhz, rs = ctypes.c_uint(), ctypes.c_ulonglong()
        while not self._stop.is_set():
            if self.nv.nvmlDeviceGetClockInfo(self.h, 1, ctypes.byref(mhz)) == 0:  # 1 = SM clock
                self.samples.append(mhz.value)
            if self.nv.nvmlDeviceGetCurrentClocksThrottleReasons(self.h, ctypes.byref(rs)) == 0:
                self.reasons |= rs.value
            self._stop.wait(0.002)

    def start(self):
        if self.nv is not None:
            import threading
            self._t = threading.Thread(target=self._poll, daemon=True)
            self._t.start()
        return self

    def stop(self):
        if self._t is not None:
            self._stop.set()
            self._t.join()
        if self.nv is not None:
            self.nv.nvmlShutdown()
            self.nv = None
        if not self.samples:
            return {"sm_mhz": None, "samples": 0, "source": "nvml unavailable"}
        return {"sm_mhz": float(np.median(self.samples)), "sm_mhz_min": float(min(self.samples)),
                "samples": len(self.samples), "source": "nvml, 2 ms polling",
                "reasons": sorted(v for k, v in self.REASONS.items() if self.reasons & k)}


def measured_peaks():
    """(burst bf16 TFLOP/s, sustained bf16 TFLOP/s, HBM GB/s, source)."""
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return d["bf16_tflops"], d.get("bf16_tflops_sustained", d["bf16_tflops"]), d["hbm_gbs"], "measured"
    return 1900.0, 1700.0, 6800.0, "fallback"


# The sources that define the fused RoPE kernel and its launch: the committed
# ncu traffic applies while these are unchanged.
ROPE_KERNEL_SOURCES = ("ptx.cuh", "gemm_core.cuh", "epilogues.cuh", "gemm_launch.cuh", "host.h", "gemm_fwd.cu",
                       "runtime.cu")


def kernel_src_hash():
    """Hash of the RoPE kernel's sources with comments and blank space removed,
    so that a comment edit does not void the recorded ncu traffic."""
    h = hashlib.sha256()
    for f in ROPE_KERNEL_SOURCES:
        src = open(os.path.join(ROOT, "gemm_epilogue_transformer_gb300", "csrc", f)).read()
        src = re.sub(r"/\*.*?\*/", " ", src, flags=re.S)
        src = re.sub(r"//[^\n]*", " ", src)
        h.update(" ".join(src.split()).encode())
    return h.hexdigest()[:16]


def ncu_traffic(kernel):
    """DRAM bytes per launch from the committed ncu summary, if it was taken on
    the current kernel sources; else None."""
    p = os.path.join(ROOT, "profiles", "ncu_traffic.json")
    if not os.path.exists(p):
        return None
    d = json.load(open(p)).get(kernel)
    if not d or d.get("src_hash") != kernel_src_hash():
        return None
    return d.get("dram_bytes_per_launch")


def max_over_ranks(values, dist, device):
    """Element-wise maximum of per-rank timings (the slowest replica sets the
    job's time); every rank receives the result."""
    import torch
    t = torch.tensor([float(v) for v in values], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return [float(v) for v in t.tolist()]


def main():
    a = parse()
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))

    import coda_inputs as gen
    if a.impl == "reference":
        return reference_arm(a, rank, world)
    if a.suite:
        return suite(a)

    import torch
    torch.cuda.set_device(local)
    dist = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))

    from gemm_epilogue_transformer_gb300 import build_lib
    if rank == 0 or world == 1:
        build_lib.build()
    if dist:
        dist.barrier()
    import gemm_epilogue_transformer_gb300 as G
    G.coda_init(local)

    p = gen.rope_problem(WL["M"], WL["K"], WL["N"], seed=0)
    dev = torch.device("cuda", local)

    def bf(bits):
        return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16)

    host = {k: bf(v).pin_memory() for k, v in p.items()}
    X, W, A, B = (host[k].to(dev) for k in ("X", "W", "A", "B"))
    hd, rc = WL["head_dim"], WL["rope_cols"]
    cos, sin = G.coda_rope_tables(WL["S"], hd, WL["theta"], device=dev)
    M, K, N = WL["M"], WL["K"], WL["N"]
    out = torch.empty((M, N), dtype=torch.bfloat16, device=dev)
    dP = torch.empty((M, N), dtype=torch.bfloat16, device=dev)
    dX = torch.empty((M, K), dtype=torch.bfloat16, device=dev)
    dW = torch.empty((K, N), dtype=torch.bfloat16, device=dev)
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream(dev)

    def fused_step(x, w, a_, b_, ev=None, outs=None):
        o, p_, dx, dw = outs if outs is not None else (out, dP, dX, dW)
        if ev is not None:
            ev[0].record(stream)
        G.coda_gemm_rope(x, w, cos, sin, hd, rc, out=o)
        if ev is not None:
            ev[1].record(stream)
        G.coda_gemm_rope_bwd(a_, b_, cos, sin, hd, rc, out=p_)
        G.coda_gemm(p_, w, transB=True, out=dx)
        G.coda_gemm(x, p_, transA=True, out=dw)

    def unfused_step():
        G.coda_gemm(X, W, out=out)
        G.coda_unfused_rope(out, cos, sin, hd, rc)
        G.coda_gemm(A, B, out=dP)
        G.coda_unfused_rope_bwd(dP, cos, sin, hd, rc)
        G.coda_gemm(dP, W, transB=True, out=dX)
        G.coda_gemm(X, dP, transA=True, out=dW)

    def barrier():
        torch.cuda.synchronize(dev)
        if dist:
            dist.barrier()
        torch.cuda.synchronize(dev)

    def timed(step_fn, steps, kernel_events=False):
        ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(steps)]
        kev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(steps)]
        barrier()
        for i in range(steps):
            flush.zero_()
            ev[i][0].record(stream)
            step_fn(kev[i] if kernel_events else None)
            ev[i][1].record(stream)
        barrier()
        step_ms = [s.elapsed_time(e) for s, e in ev]
        k_ms = [s.elapsed_time(e) for s, e in kev] if kernel_events else None
        timed.last = (step_ms, k_ms)
        return float(np.mean(step_ms)), (float(np.mean(k_ms)) if k_ms else None)

    clocks = Clocks(local)
    clocks.start()
    for _ in range(a.warmup):
        fused_step(X, W, A, B)
        unfused_step()
    torch.cuda.synchronize(dev)
    G.coda_device_status(clear=True)

    # NVTX ranges name the phases for profilers (ncu --nvtx --nvtx-include "fused/")
    nvtx = torch.cuda.nvtx
    nvtx.range_push("fused")
    clk_fused = NvmlClocks(local).start()
    ms_fused, ms_rope = timed(lambda ev: fused_step(X, W, A, B, ev), a.steps, kernel_events=True)
    clk_fused = clk_fused.stop()
    step_ms_all, rope_ms_all = timed.last
    nvtx.range_pop()
    nvtx.range_push("unfused")
    ms_unfused, _ = timed(lambda ev: unfused_step(), a.steps)
    nvtx.range_pop()

    # The headline kernel back to back with no L2 flush in between (its inputs,
    # 128 MiB, then partly stay in the 126 MiB L2): the other cache regime.
    # One event pair spans the batch: back-to-back launches overlap through
    # programmatic dependent launch, which per-launch events would cut.
    ev_u = (torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
    for _ in range(3):
        G.coda_gemm_rope(X, W, cos, sin, hd, rc, out=out)
    barrier()
    ev_u[0].record(stream)
    for _ in range(a.steps):
        G.coda_gemm_rope(X, W, cos, sin, hd, rc, out=out)
    ev_u[1].record(stream)
    barrier()
    ms_rope_unflushed = ev_u[0].elapsed_time(ev_u[1]) / a.steps

    # End to end through the public API: every step copies its four inputs from
    # pinned host memory to the device, runs the step, and copies its three
    # results back to pinned host memory. Serial: all on the compute stream.
    # Pipelined (the reported e2e): host-to-device copies on one copy stream,
    # device-to-host copies on another, double-buffered device inputs and
    # outputs and two sets of host result buffers, so step i's copies overlap
    # the neighbouring steps' compute and each other; every step still moves
    # all of its bytes inside the timed region.
    names_in = ("X", "W", "A", "B")
    d_in = [{k: torch.empty_like(host[k], device=dev) for k in names_in} for _ in range(2)]
    d_out = [(torch.empty_like(out), torch.empty_like(dP), torch.empty_like(dX), torch.empty_like(dW))
             for _ in range(2)]
    h_res = [(torch.empty((M, N), dtype=torch.bfloat16).pin_memory(),
              torch.empty((M, K), dtype=torch.bfloat16).pin_memory(),
              torch.empty((K, N), dtype=torch.bfloat16).pin_memory()) for _ in range(2)]

    def e2e_serial_step(_ev):
        di, do, hr = d_in[0], d_out[0], h_res[0]
        for k in names_in:
            di[k].copy_(host[k], non_blocking=True)
        fused_step(di["X"], di["W"], di["A"], di["B"], outs=do)
        hr[0].copy_(do[0], non_blocking=True)
        hr[1].copy_(do[2], non_blocking=True)
        hr[2].copy_(do[3], non_blocking=True)

    s_h2d = torch.cuda.Stream(dev)
    s_d2h = torch.cuda.Stream(dev)

    def e2e_pipelined(steps):
        ev = lambda: torch.cuda.Event(enable_timing=False)  # noqa: E731
        in_ready, in_free = [ev(), ev()], [ev(), ev()]
        out_ready, out_free = [ev(), ev()], [ev(), ev()]
        t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        barrier()
        t0.record(stream)
        for j in range(2):
            in_free[j].record(stream)
            out_free[j].record(stream)
        for i in range(steps):
            j = i % 2
            with torch.cuda.stream(s_h2d):
                s_h2d.wait_event(in_free[j])
                for k in names_in:
                    d_in[j][k].copy_(host[k], non_blocking=True)
                in_ready[j].record(s_h2d)
            stream.wait_event(in_ready[j])
            stream.wait_event(out_free[j])
            fused_step(d_in[j]["X"], d_in[j]["W"], d_in[j]["A"], d_in[j]["B"], outs=d_out[j])
            in_free[j].record(stream)
            out_ready[j].record(stream)
            with torch.cuda.stream(s_d2h):
                s_d2h.wait_event(out_ready[j])
                h_res[j][0].copy_(d_out[j][0], non_blocking=True)
                h_res[j][1].copy_(d_out[j][2], non_blocking=True)
                h_res[j][2].copy_(d_out[j][3], non_blocking=True)
                out_free[j].record(s_d2h)
        for j in range(2):
            stream.wait_event(out_free[j])
        t1.record(stream)
        barrier()
        return t0.elapsed_time(t1) / steps

    # At least 50 steps for the end-to-end figures, whatever --steps is: the pipelined loop fills
    # and drains its copy streams once per run, about one step's copies, which 20 steps would
    # charge at 5 % of the figure. Every step still moves all of its bytes.
    e2e_steps = max(50, min(a.steps, 200))
    for _ in range(2):
        e2e_serial_step(None)
    nvtx.range_push("e2e_serial")
    ms_e2e_serial, _ = timed(e2e_serial_step, e2e_steps)
    nvtx.range_pop()
    e2e_pipelined(3)
    nvtx.range_push("e2e")
    ms_e2e = e2e_pipelined(e2e_steps)
    nvtx.range_pop()
    clk = clocks.stop()
    status = G.coda_device_status(clear=True)
    h2d = sum(host[k].numel() * 2 for k in ("X", "W", "A", "B"))
    d2h = (M * N + M * K + K * N) * 2

    if dist:
        ms_fused, ms_unfused, ms_e2e, ms_e2e_serial, ms_rope = max_over_ranks(
            [ms_fused, ms_unfused, ms_e2e, ms_e2e_serial, ms_rope], dist, dev)

    if rank != 0:
        if dist:
            dist.destroy_process_group()
        return 0

    peak_tf, peak_tf_sus, _, peak_kind = measured_peaks()
    achieved = FLOPS_PER_GEMM / (ms_rope * 1e-3) / 1e12
    ach_unflushed = FLOPS_PER_GEMM / (ms_rope_unflushed * 1e-3) / 1e12
    traffic = ncu_traffic("coda_gemm_rope")
    line = {
        "metric": METRIC,
        "value": world * FLOPS_PER_STEP / (ms_fused * 1e-3) / 1e12,
        "unit": "TFLOP/s",
        "n_gpus": world,
        "steps": a.steps,
        "warmup": a.warmup,
        "ms_per_step": ms_fused,
        "ms_per_step_median": float(np.median(step_ms_all)),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "bf16",
        "data": "synthetic (seeded N(0,1) activations, N(0,1/K) weights, bf16)",
        "config": config(),
        "speedup_vs_unfused": ms_unfused / ms_fused,
        "unfused_ms_per_step": ms_unfused,
        "pct_bf16_peak": 100.0 * (FLOPS_PER_STEP / (ms_fused * 1e-3) / 1e12) / peak_tf,
        "clocks": clk,
        "e2e": {"value": world * FLOPS_PER_STEP / (ms_e2e * 1e-3) / 1e12, "unit": "TFLOP/s",
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "ms_per_step": ms_e2e,
                "pipeline": "copy streams overlap compute, double-buffered", "steps": e2e_steps,
                "serial_ms_per_step": ms_e2e_serial,
                "serial_value": world * FLOPS_PER_STEP / (ms_e2e_serial * 1e-3) / 1e12},
        "gpu_launches": 4 * a.steps,
        "roofline": {"kernel": "coda_gemm_rope (gemm_epilogue_kernel<EpiRope<1>>)", "bound": "tensor",
                     "achieved": achieved, "peak": peak_tf, "unit": "TFLOP/s", "frac": achieved / peak_tf,
                     "peak_source": f"bf16_tflops (burst) of {peak_kind}", "traffic": traffic,
                     "ms_per_launch": ms_rope, "ms_per_launch_median": float(np.median(rope_ms_all)),
                     "peak_sustained": peak_tf_sus, "frac_sustained": achieved / peak_tf_sus,
                     "sm_mhz": clk_fused.get("sm_mhz"), "clock": clk_fused,
                     "unflushed": {"ms_per_launch": ms_rope_unflushed, "achieved": ach_unflushed,
                                   "frac": ach_unflushed / peak_tf, "launches": a.steps,
                                   "l2": "no flush between back-to-back launches, mean over the batch"}},
        "device_status": status,
    }
    if not a.no_configs and world == 1:
        # every other config, fused against unfused (median of alternating reps)
        del host, d_in, d_out, h_res, flush
        torch.cuda.empty_cache()
        R = Runner(G, dev, reps=50)
        entries = []
        for name in CONFIG_WORKLOADS:
            entries += run_workload(R, name)
        line["configs"] = {f"{e['workload']}/{e['op']}": e for e in entries}
        status |= G.coda_device_status(clear=True)
        line["device_status"] = status
    if not a.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(p)
    print(json.dumps(line), flush=True)
    if dist:
        dist.destroy_process_group()
    return 0


def reference_arm(a, rank, world):
    """The float64 CPU oracle on a bounded sample of each step (rank 0 only)."""
    if rank != 0:
        return 0
    import coda_inputs as gen
    p = gen.rope_problem(WL["M"], WL["K"], WL["N"], seed=0)
    oracle_prepare(p)
    rows = calibrate_rows(p, 2.0)
    for _ in range(a.warmup):
        oracle_sample(p, rows)
    ts, fl = [], 0.0
    for _ in range(a.steps):
        t, fl = oracle_sample(p, rows)
        ts.append(t)
    ms = 1e3 * float(np.mean(ts))
    value = fl / (ms * 1e-3) / 1e12
    sample = f"first {rows} of 4096 token rows of each of the 4 GEMMs of one step (float64 NumPy)"
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": world,
        "steps": a.steps, "warmup": a.warmup, "ms_per_step": ms, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic (seeded, same inputs as the GPU arm)",
        "config": config(),
        "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": cores(), "kind": "oracle", "sample": sample},
        "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


# ---------------------------------------------------------------- operator suite

class Runner:
    """Times fused sequences against their unfused twins. Repetitions of the
    two (and of the dominant kernel alone) alternate, with the L2 flushed
    before every one, so clock and power drift over the run affect every
    column alike. Each entry samples the SM clock while it runs."""

    def __init__(self, G, dev, reps, min_s=1.0, max_reps=2000):
        import torch
        self.G, self.dev, self.reps, self.min_s, self.max_reps = G, dev, reps, min_s, max_reps
        self.stream = torch.cuda.current_stream(dev)
        self.flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)
        self.peak_tf, self.peak_tf_sus, self.peak_bw, self.peak_kind = measured_peaks()

    def _time_unflushed(self, fn, reps):
        """Mean time of fn over `reps` back-to-back calls with no L2 flush
        between them (the other cache regime: inputs may partly stay in L2).
        One event pair spans the whole batch: the kernels are launched with
        programmatic dependent launch, so a call's prologue overlaps the
        previous call's tail, which events around each call would cut."""
        import torch
        s, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        fn()
        torch.cuda.synchronize(self.dev)
        s.record(self.stream)
        for _ in range(reps):
            fn()
        e.record(self.stream)
        torch.cuda.synchronize(self.dev)
        return s.elapsed_time(e) / reps

    def _time(self, fns, reps):
        import torch
        ev = [[(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in fns]
              for _ in range(reps)]
        torch.cuda.synchronize(self.dev)
        for r in range(reps):
            for (s, e), fn in zip(ev[r], fns):
                self.flush.zero_()
                s.record(self.stream)
                fn()
                e.record(self.stream)
        torch.cuda.synchronize(self.dev)
        return [[ev[r][i][0].elapsed_time(ev[r][i][1]) for r in range(reps)] for i in range(len(fns))]

    def roofline(self, ms, flops, nbytes, peak_mult=1.0):
        """Fraction of the kernel's roofline: max(F / P, B / BW) / t, against
        the burst and the sustained bf16 peak (times peak_mult for FP8)."""
        t_hbm = nbytes / (self.peak_bw * 1e9) if nbytes else 0.0
        out = {"ms": ms, "tflops": flops / (ms * 1e-3) / 1e12 if flops else None,
               "gbs": nbytes / (ms * 1e-3) / 1e9 if nbytes else None}
        for key, pk in (("frac", self.peak_tf), ("frac_sustained", self.peak_tf_sus)):
            t_tc = flops / (pk * peak_mult * 1e12) if flops else 0.0
            out[key] = max(t_tc, t_hbm) / (ms * 1e-3)
        out["bound"] = "tensor" if flops and flops / (self.peak_tf * peak_mult * 1e12) >= t_hbm else "hbm"
        return out

    def entry(self, workload, op, flops, fused, unfused, launches, kernels=(), peak_mult=1.0, fused_bytes=None):
        """kernels: (name, fn, flops, bytes) of the sequence's dominant kernel(s),
        each timed alone; an empty list means `fused` is one kernel (its bytes
        in fused_bytes)."""
        fns = [fused, unfused] + [k[1] for k in kernels]
        for _ in range(3):
            for fn in fns:
                fn()
        one = self._time(fns, 1)
        round_ms = sum(x[0] for x in one) + 0.05 * len(fns)
        reps = int(min(self.max_reps, max(self.reps, np.ceil(1e3 * self.min_s / round_ms))))
        clk = NvmlClocks(self.dev.index or 0).start()
        t = self._time(fns, reps)
        c = clk.stop()
        tn = self._time_unflushed(fused, min(reps, 200))
        fm, um = float(np.median(t[0])), float(np.median(t[1]))
        e = {"workload": workload, "op": op, "fused_ms": fm, "fused_min_ms": float(np.min(t[0])),
             "fused_unflushed_ms": tn,
             "unfused_ms": um, "unfused_min_ms": float(np.min(t[1])), "speedup_vs_unfused": um / fm,
             "fused_tflops": flops / (fm * 1e-3) / 1e12 if flops else None, "reps": reps,
             "kernels": launches, "sm_mhz": c.get("sm_mhz"), "clock_reasons": c.get("reasons"),
             "clock_samples": c.get("samples")}
        if peak_mult != 1.0:
            e["peak_note"] = f"FP8 peak taken as {peak_mult:g} x the bf16 peak"
        if kernels:
            e["dominant"] = []
            for (name, _, kf, kb), tk in zip(kernels, t[2:]):
                e["dominant"].append({"kernel": name, **self.roofline(float(np.median(tk)), kf, kb, peak_mult)})
        else:
            e["dominant"] = [{"kernel": "the fused kernel", **self.roofline(fm, flops, fused_bytes or 0, peak_mult)}]
        return e


def _dev_normal(gen_t, dev):
    import torch

    def normal(shape, std=1.0, mean=0.0):
        x = torch.randn(shape, generator=gen_t, device=dev, dtype=torch.float32)
        return (x * std + mean).to(torch.bfloat16)
    return normal


def rms_chain_entries(R, name, M, Kd):
    """GEMM-RMSNorm-GEMM forward and backward (d = N = K = Kd)."""
    import torch
    G, dev = R.G, R.dev
    g = torch.Generator(device=dev)
    g.manual_seed(0)
    nrm = _dev_normal(g, dev)
    d_ = Kd
    x, W0, z = nrm((M, Kd)), nrm((Kd, d_), Kd ** -0.5), nrm((M, d_))
    gam, W1 = nrm((d_,), 0.1, 1.0), nrm((d_, d_), d_ ** -0.5)
    dO, Wn = nrm((M, Kd)), nrm((Kd, d_), Kd ** -0.5)
    nb = G.coda_num_col_tiles(d_)
    h1 = torch.empty((M, d_), dtype=torch.bfloat16, device=dev)
    h2, h0, Y = (torch.empty_like(h1) for _ in range(3))
    psq = torch.empty((M, nb), dtype=torch.float32, device=dev)
    r = torch.empty((M,), dtype=torch.float32, device=dev)

    def fused_fwd():
        G.coda_gemm_res_rmsprep(x, W0, z, gam, h1=h1, h2=h2, psq=psq)
        G.coda_rms_reduce(psq, d_, 1e-6, r=r)
        G.coda_gemm_rowscale(h2, W1, r, out=Y)

    def unfused_fwd():
        G.coda_gemm(x, W0, out=h0)
        G.coda_unfused_add(h0, z, out=h1)
        nn, _ = G.coda_unfused_rmsnorm(h1, gam, 1e-6)
        G.coda_gemm(nn, W1, out=Y)

    fl = 2.0 * M * Kd * d_
    b1 = 2.0 * (M * Kd + Kd * d_ + 3 * M * d_ + d_) + 4.0 * M * nb
    out = [R.entry(name, "fwd", 2 * fl, fused_fwd, unfused_fwd, "3 fused (2 GEMM + aux) vs 4 unfused",
                   kernels=[("coda_gemm_res_rmsprep (GEMM1: h1, h2, row partials)",
                             lambda: G.coda_gemm_res_rmsprep(x, W0, z, gam, h1=h1, h2=h2, psq=psq), fl, b1)])]
    fused_fwd()
    st = {}

    def fused_bwd():
        dY_, _, pd = G.coda_gemm_rowdot(dO, Wn, Y, r)
        s_ = G.coda_rowdot_reduce(pd, d_)
        dh, pdg = G.coda_gemm_rmsnorm_bwd(dY_, W1, h1, gam, r, s_)
        G.coda_colsum_reduce(pdg)
        st["dY"], st["s"] = dY_, s_

    def unfused_bwd():
        dY_ = G.coda_gemm(dO, Wn)
        Gd = G.coda_gemm(dY_, W1, transB=True)
        _, pdg = G.coda_unfused_rmsnorm_bwd(Gd, h1, gam, r)
        G.coda_colsum_reduce(pdg)

    fused_bwd()
    b2 = 2.0 * (M * d_ + d_ * d_ + 2 * M * d_ + d_) + 4.0 * (2 * M + (M // 32 + 1) * d_)
    out.append(R.entry(name, "bwd", 2 * fl, fused_bwd, unfused_bwd,
                       "dY GEMM + rowdot + RMSNorm-bwd GEMM + 2 aux vs 2 GEMM + rmsnorm_bwd + colsum",
                       kernels=[("coda_gemm_rmsnorm_bwd (dgrad of GEMM2: dh1, dgamma partials)",
                                 lambda: G.coda_gemm_rmsnorm_bwd(st["dY"], W1, h1, gam, r, st["s"]), fl, b2)]))
    return out


def rope_entries(R):
    import torch
    G, dev = R.G, R.dev
    M, K, N, hd, rc = 4096, 4096, 12288, 128, 8192
    g = torch.Generator(device=dev)
    g.manual_seed(0)
    nrm = _dev_normal(g, dev)
    X, W, A_, B_ = nrm((M, K)), nrm((K, N), K ** -0.5), nrm((M, K)), nrm((K, N), K ** -0.5)
    c, sn = G.coda_rope_tables(4096, hd, 10000.0, device=dev)
    out = torch.empty((M, N), dtype=torch.bfloat16, device=dev)
    fl, by = 2.0 * M * N * K, 2.0 * (M * K + K * N + M * N) + 8.0 * 4096 * hd // 2
    return [R.entry("rope_qkv_4096", "fwd", fl, lambda: G.coda_gemm_rope(X, W, c, sn, hd, rc, out=out),
                    lambda: (G.coda_gemm(X, W, out=out), G.coda_unfused_rope(out, c, sn, hd, rc)), "1 vs 2",
                    fused_bytes=by),
            R.entry("rope_qkv_4096", "bwd", fl, lambda: G.coda_gemm_rope_bwd(A_, B_, c, sn, hd, rc, out=out),
                    lambda: (G.coda_gemm(A_, B_, out=out), G.coda_unfused_rope_bwd(out, c, sn, hd, rc)), "1 vs 2",
                    fused_bytes=by),
            R.entry("rope_qkv_4096", "plain_gemm", fl, lambda: G.coda_gemm(X, W, out=out),
                    lambda: G.coda_gemm(X, W, out=out), "identity epilogue, both columns the same kernel",
                    fused_bytes=2.0 * (M * K + K * N + M * N))]


def swiglu_entries(R):
    import torch
    G, dev = R.G, R.dev
    M, K, F = 4096, 4096, 14336
    g = torch.Generator(device=dev)
    g.manual_seed(0)
    nrm = _dev_normal(g, dev)
    X, Wgu, dYs, Wd = nrm((M, K)), nrm((K, 2 * F), K ** -0.5), nrm((M, K)), nrm((F, K), F ** -0.5)
    A = torch.empty((M, F), dtype=torch.bfloat16, device=dev)
    GU = torch.empty((M, 2 * F), dtype=torch.bfloat16, device=dev)
    dA = torch.empty((M, F), dtype=torch.bfloat16, device=dev)
    dGU = torch.empty_like(GU)
    fl = 2.0 * M * 2 * F * K
    by = 2.0 * (M * K + K * 2 * F + M * F)
    out = [R.entry("swiglu_up_4096", "fwd", fl, lambda: G.coda_gemm_swiglu(X, Wgu, out=A),
                   lambda: (G.coda_gemm(X, Wgu, out=GU), G.coda_unfused_swiglu(GU)), "1 vs 2 (no GU saved)",
                   fused_bytes=by),
           R.entry("swiglu_up_4096", "fwd_save_gu", fl, lambda: G.coda_gemm_swiglu(X, Wgu, out=A, gu=GU),
                   lambda: (G.coda_gemm(X, Wgu, out=GU), G.coda_unfused_swiglu(GU)),
                   "1 vs 2 (GU saved for backward)", fused_bytes=by + 2.0 * M * 2 * F)]
    G.coda_gemm_swiglu(X, Wgu, out=A, gu=GU)
    out.append(R.entry("swiglu_up_4096", "bwd", fl / 2, lambda: G.coda_gemm_swiglu_bwd(dYs, Wd, GU, out=dGU),
                       lambda: (G.coda_gemm(dYs, Wd, transB=True, out=dA), G.coda_unfused_swiglu_bwd(dA, GU)),
                       "1 vs 2", fused_bytes=2.0 * (M * K + F * K + 2 * M * 2 * F)))
    return out


def ce_entries(R):
    import torch
    G, dev = R.G, R.dev
    M, K, V = 8192, 4096, 32768
    g = torch.Generator(device=dev)
    g.manual_seed(0)
    nrm = _dev_normal(g, dev)
    H, W = nrm((M, K)), nrm((K, V), K ** -0.5)
    y = torch.randint(0, V, (M,), generator=g, device=dev, dtype=torch.int32)
    logits = torch.empty((M, V), dtype=torch.bfloat16, device=dev)
    st = {}
    nb = G.coda_num_col_tiles(V)

    def fused_ce():
        pm, ps, pa, tg = G.coda_gemm_ce_lse(H, W, y)
        st["lse"] = G.coda_ce_reduce(pm, ps, pa, tg)[0]

    def unfused_ce():
        G.coda_gemm(H, W, out=logits)
        G.coda_unfused_ce_fwd(logits, y)

    fl = 2.0 * M * V * K
    b_in = 2.0 * (M * K + K * V) + 4.0 * M
    out = [R.entry("lm_head_ce_8192", "fwd", fl, fused_ce, unfused_ce,
                   "GEMM+partials + reduce vs GEMM (bf16 logits) + CE",
                   kernels=[("coda_gemm_ce_lse (online LSE partials)", lambda: G.coda_gemm_ce_lse(H, W, y), fl,
                             b_in + 12.0 * M * nb + 4.0 * M)])]
    fused_ce()
    lse = st["lse"]
    out.append(R.entry("lm_head_ce_8192", "bwd_dlogits", fl,
                       lambda: G.coda_gemm_ce_bwd(H, W, y, lse, 1.0 / M, out=logits),
                       lambda: (G.coda_gemm(H, W, out=logits), G.coda_unfused_ce_bwd(logits, y, lse, 1.0 / M)),
                       "recompute GEMM with dl epilogue vs recompute GEMM + CE-bwd kernel",
                       fused_bytes=b_in + 4.0 * M + 2.0 * M * V))
    return out


def block_entries(R, dm):
    """One period of the block-level chain (RoPE-path and SwiGLU-path
    GEMM-residual-RMSNorm-GEMM structures) at 16K tokens, forward and forward +
    backward, fused sequence vs unfused sequence."""
    import torch
    import coda_inputs as gen
    G, dev = R.G, R.dev
    c = gen.WORKLOADS[f"block_d{dm}"]
    M, d, F, hd, rc, S = c["M"], c["d"], c["F"], c["head_dim"], c["rope_cols"], c["S"]
    g = torch.Generator(device=dev)
    g.manual_seed(0)
    nrm = _dev_normal(g, dev)
    t = dict(P=nrm((M, F)), Wd=nrm((F, d), F ** -0.5), x=nrm((M, d)), gamma1=nrm((d,), 0.1, 1.0),
             Wqkv=nrm((d, 3 * d), d ** -0.5), O=nrm((M, d)), Wo=nrm((d, d), d ** -0.5),
             gamma2=nrm((d,), 0.1, 1.0), Wgu=nrm((d, 2 * F), d ** -0.5), dQKV=nrm((M, 3 * d)),
             gh=nrm((M, d)), Wdn=nrm((F, d), F ** -0.5))
    cos, sin = G.coda_rope_tables(S, hd, c["theta"], device=dev)
    fl_fwd = 2.0 * M * d * (3 * F + 4 * d)
    fused = G.CodaBlock(t, hd, rc, cos, sin, c["eps"])
    unfused = G.CodaBlock(t, hd, rc, cos, sin, c["eps"], unfused=True)
    name = f"block_d{dm}"
    fl_up = 2.0 * M * d * 2 * F
    up_bytes = 2.0 * (M * d + d * 2 * F + M * F + M * 2 * F) + 4.0 * M
    out = [R.entry(name, "fwd", fl_fwd, fused.fwd, unfused.fwd_unfused, "6 fused launches vs 10 unfused",
                   kernels=[("coda_gemm_rowscale_swiglu (SwiGLU up-projection, GU saved)",
                             lambda: G.coda_gemm_rowscale_swiglu(fused.h2g, t["Wgu"], fused.r2, out=fused.a,
                                                                 gu=fused.gu), fl_up, up_bytes)])]
    fused.fwd().bwd()
    unfused.fwd_unfused()
    nbF = G.coda_num_col_tiles(F)
    b1_bytes = 2.0 * (M * d + F * d + 2 * M * 2 * F) + 4.0 * (M + M * nbF)
    res_bytes = 2.0 * (M * 2 * F + d * 2 * F + 3 * M * d + d) + 4.0 * (2 * M + (M // 32) * d)
    out.append(R.entry(
        name, "fwd_bwd", 3 * fl_fwd, lambda: fused.fwd().bwd(), lambda: unfused.fwd_unfused().bwd_unfused(),
        "19 fused launches vs 26 unfused",
        kernels=[("coda_gemm_rmsnorm_bwd_res (dh2 = RMSNorm-bwd of the SwiGLU path, K = 2F)",
                  lambda: G.coda_gemm_rmsnorm_bwd_res(fused.dgur, t["Wgu"], fused.h2, t["gamma2"], fused.r2,
                                                      fused.s2, t["gh"]), fl_up, res_bytes),
                 ("coda_gemm_swiglu_bwd_rowdot (SwiGLU backward with the row statistic)",
                  lambda: G.coda_gemm_swiglu_bwd_rowdot(t["gh"], t["Wdn"], fused.gu, fused.r2), fl_up / 2,
                  b1_bytes)]))
    return out


def fp8_entries(R, want):
    """FP8 (E4M3) mainloop variants: the fused kernel against the FP8 plain GEMM
    plus the same stand-alone kernels. The percentage is of the FP8 dense peak,
    taken as twice the measured BF16 peak (the nominal FP8 / BF16 ratio)."""
    import torch
    import coda_inputs as gen
    G, dev = R.G, R.dev
    out = []

    def u8(bits):
        return torch.from_numpy(np.ascontiguousarray(bits, dtype=np.uint8)).to(dev)

    name = "fp8_rope_qkv_4096"
    if want(name):
        w = gen.WORKLOADS[name]
        p = gen.fp8_problem(w["M"], w["K"], w["N"], seed=0)
        X, Wt, al = u8(p["A"]), u8(p["B"]), p["sA"] * p["sB"]
        c, sn = G.coda_rope_tables(w["S"], w["head_dim"], w["theta"], device=dev)
        o = torch.empty((w["M"], w["N"]), dtype=torch.bfloat16, device=dev)
        hd, rc = w["head_dim"], w["rope_cols"]
        fl = 2.0 * w["M"] * w["N"] * w["K"]
        by = 1.0 * (w["M"] + w["N"]) * w["K"] + 2.0 * w["M"] * w["N"]
        out.append(R.entry(name, "fwd", fl, lambda: G.coda_gemm_rope_fp8(X, Wt, al, c, sn, hd, rc, out=o),
                           lambda: (G.coda_gemm_fp8(X, Wt, al, out=o), G.coda_unfused_rope(o, c, sn, hd, rc)),
                           "1 vs 2", peak_mult=2.0, fused_bytes=by))
        out.append(R.entry(name, "plain_gemm", fl, lambda: G.coda_gemm_fp8(X, Wt, al, out=o),
                           lambda: G.coda_gemm_fp8(X, Wt, al, out=o), "identity epilogue, both columns the same kernel",
                           peak_mult=2.0, fused_bytes=by))
        del p, X, Wt, o
    name = "fp8_swiglu_up_4096"
    if want(name):
        w = gen.WORKLOADS[name]
        p = gen.fp8_problem(w["M"], w["K"], w["N"], seed=0)
        X, Wt, al = u8(p["A"]), u8(p["B"]), p["sA"] * p["sB"]
        F = w["N"] // 2
        A = torch.empty((w["M"], F), dtype=torch.bfloat16, device=dev)
        GU = torch.empty((w["M"], 2 * F), dtype=torch.bfloat16, device=dev)
        fl = 2.0 * w["M"] * w["N"] * w["K"]
        by = 1.0 * (w["M"] + w["N"]) * w["K"] + 2.0 * w["M"] * F
        out.append(R.entry(name, "fwd", fl, lambda: G.coda_gemm_swiglu_fp8(X, Wt, al, out=A),
                           lambda: (G.coda_gemm_fp8(X, Wt, al, out=GU), G.coda_unfused_swiglu(GU)),
                           "1 vs 2 (no GU saved)", peak_mult=2.0, fused_bytes=by))
        out.append(R.entry(name, "fwd_save_gu", fl, lambda: G.coda_gemm_swiglu_fp8(X, Wt, al, out=A, gu=GU),
                           lambda: (G.coda_gemm_fp8(X, Wt, al, out=GU), G.coda_unfused_swiglu(GU)),
                           "1 vs 2 (GU saved for backward)", peak_mult=2.0, fused_bytes=by + 4.0 * w["M"] * F))
        del p, X, Wt, A, GU
    name = "fp8_lm_head_ce_8192"
    if want(name):
        w = gen.WORKLOADS[name]
        p = gen.fp8_problem(w["M"], w["K"], w["N"], seed=0, labels=True)
        H, Wt, al = u8(p["A"]), u8(p["B"]), p["sA"] * p["sB"]
        y = torch.from_numpy(p["labels"]).to(dev)
        logits = torch.empty((w["M"], w["N"]), dtype=torch.bfloat16, device=dev)
        fl = 2.0 * w["M"] * w["N"] * w["K"]
        st = {}

        def fused_ce():
            pm, ps, pa, tg = G.coda_gemm_ce_lse_fp8(H, Wt, al, y)
            st["lse"] = G.coda_ce_reduce(pm, ps, pa, tg)[0]

        out.append(R.entry(name, "fwd", fl, fused_ce, lambda: (G.coda_gemm_fp8(H, Wt, al, out=logits),
                                                               G.coda_unfused_ce_fwd(logits, y)),
                           "GEMM+partials + reduce vs GEMM (bf16 logits) + CE", peak_mult=2.0,
                           kernels=[("coda_gemm_ce_lse_fp8", lambda: G.coda_gemm_ce_lse_fp8(H, Wt, al, y), fl,
                                     1.0 * (w["M"] + w["N"]) * w["K"])]))
        fused_ce()
        lse = st["lse"]
        out.append(R.entry(name, "bwd_dlogits", fl,
                           lambda: G.coda_gemm_ce_bwd_fp8(H, Wt, al, y, lse, 1.0 / w["M"], out=logits),
                           lambda: (G.coda_gemm_fp8(H, Wt, al, out=logits),
                                    G.coda_unfused_ce_bwd(logits, y, lse, 1.0 / w["M"])),
                           "recompute GEMM with dl epilogue vs recompute GEMM + CE-bwd kernel", peak_mult=2.0,
                           fused_bytes=1.0 * (w["M"] + w["N"]) * w["K"] + 2.0 * w["M"] * w["N"]))
        del p, H, Wt, logits
    return out


def ce_f2_entries(R):
    """Bound on what consuming the cross-entropy gradient on chip could save
    (dl never stored, never re-read): the backward as built (the recompute GEMM
    whose epilogue writes dl, then dH = dl W^T and dW = H^T dl) against the same
    three GEMMs with the recompute GEMM storing nothing (its forward twin, which
    keeps only per-tile statistics). The difference is the dl write plus the
    dl-forming epilogue; a fused design would still run all three contractions."""
    import torch
    G, dev = R.G, R.dev
    M, K, V = 8192, 4096, 32768
    g = torch.Generator(device=dev)
    g.manual_seed(0)
    nrm = _dev_normal(g, dev)
    H, W = nrm((M, K)), nrm((K, V), K ** -0.5)
    y = torch.randint(0, V, (M,), generator=g, device=dev, dtype=torch.int32)
    pm, ps, pa, tg = G.coda_gemm_ce_lse(H, W, y)
    lse = G.coda_ce_reduce(pm, ps, pa, tg)[0]
    dl = torch.empty((M, V), dtype=torch.bfloat16, device=dev)
    dH = torch.empty((M, K), dtype=torch.bfloat16, device=dev)
    dW = torch.empty((K, V), dtype=torch.bfloat16, device=dev)
    G.coda_gemm_ce_bwd(H, W, y, lse, 1.0 / M, out=dl)

    def built():
        G.coda_gemm_ce_bwd(H, W, y, lse, 1.0 / M, out=dl)
        G.coda_gemm(dl, W, transB=True, out=dH)
        G.coda_gemm(H, dl, transA=True, out=dW)

    def bound():
        G.coda_gemm_ce_lse(H, W, y)
        G.coda_gemm(dl, W, transB=True, out=dH)
        G.coda_gemm(H, dl, transA=True, out=dW)

    e = R.entry("lm_head_ce_8192", "bwd_chain_f2_bound", 3 * 2.0 * M * V * K, built, bound,
                "fused column: dl-forming GEMM + dH + dW as built; unfused column: the same three GEMMs "
                "with the recompute GEMM storing no dl (the most an on-chip dl could save)")
    e["f2_max_gain"] = e["fused_ms"] / e["unfused_ms"]
    return [e]


def cublas_entries(R):
    """The library's plain GEMM (identity epilogue) next to cuBLAS (torch.matmul)
    on the same operands: the mainloop's distance from the vendor library. The
    `unfused` column is cuBLAS here."""
    import torch
    G, dev = R.G, R.dev
    g = torch.Generator(device=dev)
    g.manual_seed(0)
    nrm = _dev_normal(g, dev)
    out = []
    for M, N, K in ((4096, 12288, 4096), (4096, 14336, 4096), (8192, 8192, 8192), (16384, 28672, 4096)):
        A, B = nrm((M, K)), nrm((K, N), K ** -0.5)
        C = torch.empty((M, N), dtype=torch.bfloat16, device=dev)
        C2 = torch.empty_like(C)
        e = R.entry(f"gemm_vs_cublas_{M}x{N}x{K}", "plain_gemm", 2.0 * M * N * K,
                    lambda: G.coda_gemm(A, B, out=C), lambda: torch.matmul(A, B, out=C2),
                    "fused column: coda_gemm (identity epilogue); unfused column: torch.matmul (cuBLAS)",
                    fused_bytes=2.0 * (M * K + K * N + M * N))
        e["coda_over_cublas_throughput"] = e["unfused_ms"] / e["fused_ms"]
        out.append(e)
        del A, B, C, C2
    return out


# The workloads of the default run's `configs` object (every config but the
# headline's), and of --suite.
CONFIG_WORKLOADS = ("rmsnorm_chain_tiny", "swiglu_up_4096", "rmsnorm_chain_8192", "lm_head_ce_8192", "block_d4096")
SUITE_WORKLOADS = ("rmsnorm_chain_tiny", "rmsnorm_chain_8192", "rope_qkv_4096", "swiglu_up_4096",
                   "lm_head_ce_8192", "block_d2048", "block_d4096", "block_d8192", "fp8_rope_qkv_4096",
                   "fp8_swiglu_up_4096", "fp8_lm_head_ce_8192", "ce_bwd_f2_bound", "gemm_vs_cublas")


def run_workload(R, name):
    import torch
    if name == "rmsnorm_chain_tiny":
        out = rms_chain_entries(R, name, 256, 512)
    elif name == "rmsnorm_chain_8192":
        out = rms_chain_entries(R, name, 8192, 8192)
    elif name == "rope_qkv_4096":
        out = rope_entries(R)
    elif name == "swiglu_up_4096":
        out = swiglu_entries(R)
    elif name == "lm_head_ce_8192":
        out = ce_entries(R)
    elif name.startswith("block_d"):
        out = block_entries(R, int(name[len("block_d"):]))
    elif name == "ce_bwd_f2_bound":
        out = ce_f2_entries(R)
    elif name == "gemm_vs_cublas":
        out = cublas_entries(R)
    elif name.startswith("fp8_"):
        out = fp8_entries(R, lambda n: n == name)
    else:
        raise ValueError(f"unknown workload {name}")
    torch.cuda.synchronize(R.dev)
    torch.cuda.empty_cache()
    return out


def suite(a):
    """Fused vs unfused time of every operator on every workload; one JSON line each."""
    import torch
    from gemm_epilogue_transformer_gb300 import build_lib
    build_lib.build()
    import gemm_epilogue_transformer_gb300 as G
    G.coda_init(0)
    R = Runner(G, torch.device("cuda", 0), a.reps, min_s=a.min_seconds)
    for name in SUITE_WORKLOADS:
        if a.only is None or a.only == name:
            for e in run_workload(R, name):
                print(json.dumps(e), flush=True)
    status = G.coda_device_status(clear=True)
    print(json.dumps({"suite": "done", "device_status": status}), flush=True)
    return 0 if status == 0 else 1


if __name__ == "__main__":
    sys.exit(main())
