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
    ap.add_argument("--suite", action="store_true",
                    help="time every fused operator against its unfused pair on all five workloads "
                         "(one JSON line per operator) instead of the headline step")
    ap.add_argument("--reps", type=int, default=20, help="timed repetitions per operator in --suite")
    ap.add_argument("--only", default=None,
                    help="with --suite: run one workload (rmsnorm_chain_tiny, rmsnorm_chain_8192, rope_qkv_4096, "
                         "swiglu_up_4096, lm_head_ce_8192, block_d2048, block_d4096, block_d8192, fp8_rope_qkv_4096, "
                         "fp8_swiglu_up_4096, fp8_lm_head_ce_8192)")
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


def measured_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return d["bf16_tflops"], d["hbm_gbs"], "measured"
    return 1900.0, 6800.0, "fallback"


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
    ms_fused, ms_rope = timed(lambda ev: fused_step(X, W, A, B, ev), a.steps, kernel_events=True)
    nvtx.range_pop()
    nvtx.range_push("unfused")
    ms_unfused, _ = timed(lambda ev: unfused_step(), a.steps)
    nvtx.range_pop()

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

    e2e_steps = max(3, min(a.steps, 50))
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

    peak_tf, _, peak_kind = measured_peaks()
    achieved = FLOPS_PER_GEMM / (ms_rope * 1e-3) / 1e12
    traffic = ncu_traffic("coda_gemm_rope")
    line = {
        "metric": METRIC,
        "value": world * FLOPS_PER_STEP / (ms_fused * 1e-3) / 1e12,
        "unit": "TFLOP/s",
        "n_gpus": world,
        "steps": a.steps,
        "warmup": a.warmup,
        "ms_per_step": ms_fused,
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
                "pipeline": "copy streams overlap compute, double-buffered",
                "serial_ms_per_step": ms_e2e_serial,
                "serial_value": world * FLOPS_PER_STEP / (ms_e2e_serial * 1e-3) / 1e12},
        "gpu_launches": 4 * a.steps,
        "roofline": {"kernel": "coda_gemm_rope (gemm_epilogue_kernel<EpiRope<1>>)", "bound": "tensor",
                     "achieved": achieved, "peak": peak_tf, "unit": "TFLOP/s", "frac": achieved / peak_tf,
                     "peak_source": f"bf16_tflops (burst) of {peak_kind}", "traffic": traffic,
                     "ms_per_launch": ms_rope},
        "device_status": status,
    }
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

def suite(a):
    """Fused vs unfused time of every operator on the five workloads; one JSON line each."""
    import torch
    import coda_inputs as gen
    from gemm_epilogue_transformer_gb300 import build_lib
    build_lib.build()
    import gemm_epilogue_transformer_gb300 as G
    G.coda_init(0)
    dev = torch.device("cuda", 0)
    stream = torch.cuda.current_stream(dev)
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)
    peak_tf, peak_bw, peak_kind = measured_peaks()

    def d(bits):
        return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16).to(dev)

    def graph_of(fn):
        """Capture fn's launches into a CUDA graph (after one direct run) and return its replay."""
        side = torch.cuda.Stream(dev)
        side.wait_stream(stream)
        with torch.cuda.stream(side):
            fn()
        stream.wait_stream(side)
        torch.cuda.synchronize(dev)
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=side):
            fn()
        graphs.append(g)
        return g.replay

    graphs = []

    def once(fn):
        flush.zero_()
        s, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        s.record(stream)
        fn()
        e.record(stream)
        e.synchronize()
        return s.elapsed_time(e)

    def report(workload, op, flops, fused, unfused, launches, peak_mult=1.0):
        # fused and unfused repetitions alternate, so clock and power drift over
        # the run affect both columns alike
        for _ in range(3):
            fused()
            unfused()
        tf, tu = [], []
        for _ in range(a.reps):
            tf.append(once(fused))
            tu.append(once(unfused))
        fm, fmin = float(np.median(tf)), float(np.min(tf))
        um, umin = float(np.median(tu)), float(np.min(tu))
        pk = peak_tf * peak_mult
        line = {"suite": workload, "op": op, "fused_ms": fm, "fused_min_ms": fmin, "unfused_ms": um,
                "unfused_min_ms": umin, "speedup_vs_unfused": um / fm,
                "fused_tflops": flops / (fm * 1e-3) / 1e12 if flops else None,
                "pct_bf16_peak": 100 * flops / (fm * 1e-3) / 1e12 / pk if flops else None,
                "kernels": launches, "reps": a.reps,
                "peak": (f"{pk:.1f} TFLOP/s ({peak_kind} bf16 x {peak_mult:g})" if peak_mult != 1.0
                         else f"{peak_tf} TFLOP/s ({peak_kind})")}
        print(json.dumps(line), flush=True)

    # -- GEMM-RMSNorm-GEMM (tiny and 8192)
    def want(name):
        return a.only is None or a.only == name

    for name, M, Kd, bwdK in (("rmsnorm_chain_tiny", 256, 512, 512), ("rmsnorm_chain_8192", 8192, 8192, 8192)):
        if not want(name):
            continue
        p = gen.rms_chain(M, Kd, Kd, Kd, seed=0, bwd_K=bwdK)
        x, W0, z, g, W1, dO, Wn = (d(p[k]) for k in ("x", "W0", "z", "gamma", "W1", "dO", "Wn"))
        d_ = Kd
        nb = G.coda_num_col_tiles(d_)
        h1 = torch.empty((M, d_), dtype=torch.bfloat16, device=dev)
        h2, h0, n, Y, dY, dYr, Gm, dh1 = (torch.empty_like(h1) for _ in range(8))
        psq = torch.empty((M, nb), dtype=torch.float32, device=dev)
        pdot = torch.empty_like(psq)
        r = torch.empty((M,), dtype=torch.float32, device=dev)
        ru = torch.empty_like(r)

        def fused_fwd():
            G.coda_gemm_res_rmsprep(x, W0, z, g, h1=h1, h2=h2, psq=psq)
            G.coda_rms_reduce(psq, d_, 1e-6, r=r)
            G.coda_gemm_rowscale(h2, W1, r, out=Y)

        def unfused_fwd():
            G.coda_gemm(x, W0, out=h0)
            G.coda_unfused_add(h0, z, out=h1)
            nn, rr = G.coda_unfused_rmsnorm(h1, g, 1e-6)
            G.coda_gemm(nn, W1, out=Y)

        report(name, "fwd", 2 * 2.0 * M * Kd * d_, fused_fwd, unfused_fwd, "3 fused (2 GEMM + aux) vs 4 unfused")
        if M * Kd <= 256 * 512:
            # the tiny chain is launch-bound: the same sequences replayed from CUDA graphs
            report(name, "fwd_graph", 2 * 2.0 * M * Kd * d_, graph_of(fused_fwd), graph_of(unfused_fwd),
                   "the same launches, each sequence replayed from one CUDA graph")
        fused_fwd()

        def fused_bwd():
            dY_, dYr_, pd = G.coda_gemm_rowdot(dO, Wn, Y, r)
            s_ = G.coda_rowdot_reduce(pd, d_)
            dh, pdg = G.coda_gemm_rmsnorm_bwd(dY_, W1, h1, g, r, s_)
            G.coda_colsum_reduce(pdg)

        def unfused_bwd():
            dY_ = G.coda_gemm(dO, Wn)
            Gd = G.coda_gemm(dY_, W1, transB=True)
            dh, pdg = G.coda_unfused_rmsnorm_bwd(Gd, h1, g, r)
            G.coda_colsum_reduce(pdg)

        report(name, "bwd", 2 * 2.0 * M * Kd * d_, fused_bwd, unfused_bwd,
               "dY GEMM + rowdot + RMSNorm-bwd GEMM + 2 aux vs 2 GEMM + rmsnorm_bwd + colsum")
        del p, x, W0, z, g, W1, dO, Wn, h1, h2, h0, n, Y, dY, dYr, Gm, dh1
        torch.cuda.empty_cache()

    # -- GEMM + RoPE
    M, K, N, hd, rc = 4096, 4096, 12288, 128, 8192
    if want("rope_qkv_4096"):
        rope_suite(G, gen, d, dev, report, M, K, N, hd, rc)
    if want("swiglu_up_4096"):
        swiglu_suite(G, gen, d, dev, report)
    if want("lm_head_ce_8192"):
        ce_suite(G, gen, d, dev, report)
    for dm in sorted(gen.BLOCK_SIZES):
        if want(f"block_d{dm}"):
            block_suite(G, gen, dev, report, dm)
    fp8_suite(G, gen, dev, report, want)
    status = G.coda_device_status(clear=True)
    print(json.dumps({"suite": "done", "device_status": status}), flush=True)
    return 0 if status == 0 else 1


def rope_suite(G, gen, d, dev, report, M, K, N, hd, rc):
    import torch
    p = gen.rope_problem(M, K, N, seed=0)
    X, W, A_, B_ = (d(p[k]) for k in ("X", "W", "A", "B"))
    c, sn = G.coda_rope_tables(4096, hd, 10000.0, device=dev)
    out = torch.empty((M, N), dtype=torch.bfloat16, device=dev)
    report("rope_qkv_4096", "fwd", 2.0 * M * N * K, lambda: G.coda_gemm_rope(X, W, c, sn, hd, rc, out=out),
           lambda: (G.coda_gemm(X, W, out=out), G.coda_unfused_rope(out, c, sn, hd, rc)), "1 vs 2")
    report("rope_qkv_4096", "bwd", 2.0 * M * N * K, lambda: G.coda_gemm_rope_bwd(A_, B_, c, sn, hd, rc, out=out),
           lambda: (G.coda_gemm(A_, B_, out=out), G.coda_unfused_rope_bwd(out, c, sn, hd, rc)), "1 vs 2")
    report("rope_qkv_4096", "plain_gemm", 2.0 * M * N * K, lambda: G.coda_gemm(X, W, out=out),
           lambda: G.coda_gemm(X, W, out=out), "identity epilogue, both columns the same kernel")
    del p, X, W, A_, B_, out
    torch.cuda.empty_cache()


def swiglu_suite(G, gen, d, dev, report):
    import torch
    M, K, F = 4096, 4096, 14336
    p = gen.swiglu_problem(M, K, F, seed=0)
    X, Wgu, dYs, Wd = (d(p[k]) for k in ("X", "Wgu", "dY", "Wd"))
    A = torch.empty((M, F), dtype=torch.bfloat16, device=dev)
    GU = torch.empty((M, 2 * F), dtype=torch.bfloat16, device=dev)
    dA = torch.empty((M, F), dtype=torch.bfloat16, device=dev)
    dGU = torch.empty_like(GU)
    report("swiglu_up_4096", "fwd", 2.0 * M * 2 * F * K, lambda: G.coda_gemm_swiglu(X, Wgu, out=A),
           lambda: (G.coda_gemm(X, Wgu, out=GU), G.coda_unfused_swiglu(GU)), "1 vs 2 (no GU saved)")
    report("swiglu_up_4096", "fwd_save_gu", 2.0 * M * 2 * F * K,
           lambda: G.coda_gemm_swiglu(X, Wgu, out=A, gu=GU),
           lambda: (G.coda_gemm(X, Wgu, out=GU), G.coda_unfused_swiglu(GU)), "1 vs 2 (GU saved for backward)")
    report("swiglu_up_4096", "bwd", 2.0 * M * F * K, lambda: G.coda_gemm_swiglu_bwd(dYs, Wd, GU, out=dGU),
           lambda: (G.coda_gemm(dYs, Wd, transB=True, out=dA), G.coda_unfused_swiglu_bwd(dA, GU)), "1 vs 2")
    del p, X, Wgu, dYs, Wd, A, GU, dA, dGU
    torch.cuda.empty_cache()


def ce_suite(G, gen, d, dev, report):
    import torch
    M, K, V = 8192, 4096, 32768
    p = gen.ce_problem(M, K, V, seed=0)
    H, W = d(p["H"]), d(p["W"])
    y = torch.from_numpy(p["labels"]).to(dev)
    logits = torch.empty((M, V), dtype=torch.bfloat16, device=dev)
    st = {}

    def fused_ce():
        pm, ps, pa, tg = G.coda_gemm_ce_lse(H, W, y)
        st["lse"] = G.coda_ce_reduce(pm, ps, pa, tg)[0]

    def unfused_ce():
        G.coda_gemm(H, W, out=logits)
        G.coda_unfused_ce_fwd(logits, y)

    report("lm_head_ce_8192", "fwd", 2.0 * M * V * K, fused_ce, unfused_ce, "GEMM+partials + reduce vs GEMM (bf16 logits) + CE")
    fused_ce()
    lse = st["lse"]
    report("lm_head_ce_8192", "bwd_dlogits", 2.0 * M * V * K,
           lambda: G.coda_gemm_ce_bwd(H, W, y, lse, 1.0 / M, out=logits),
           lambda: (G.coda_gemm(H, W, out=logits), G.coda_unfused_ce_bwd(logits, y, lse, 1.0 / M)),
           "recompute GEMM with dl epilogue vs recompute GEMM + CE-bwd kernel")


def fp8_suite(G, gen, dev, report, want):
    """FP8 (E4M3) mainloop variants: the fused kernel against the FP8 plain GEMM
    plus the same stand-alone kernels. The percentage is of the FP8 dense peak,
    taken as twice the measured BF16 peak (the nominal FP8 / BF16 ratio)."""
    import torch

    def u8(bits):
        return torch.from_numpy(np.ascontiguousarray(bits, dtype=np.uint8)).to(dev)

    name = "fp8_rope_qkv_4096"
    if want(name):
        w = gen.WORKLOADS[name]
        p = gen.fp8_problem(w["M"], w["K"], w["N"], seed=0)
        X, Wt, al = u8(p["A"]), u8(p["B"]), p["sA"] * p["sB"]
        c, sn = G.coda_rope_tables(w["S"], w["head_dim"], w["theta"], device=dev)
        out = torch.empty((w["M"], w["N"]), dtype=torch.bfloat16, device=dev)
        hd, rc = w["head_dim"], w["rope_cols"]
        fl = 2.0 * w["M"] * w["N"] * w["K"]
        report(name, "fwd", fl, lambda: G.coda_gemm_rope_fp8(X, Wt, al, c, sn, hd, rc, out=out),
               lambda: (G.coda_gemm_fp8(X, Wt, al, out=out), G.coda_unfused_rope(out, c, sn, hd, rc)), "1 vs 2",
               peak_mult=2.0)
        report(name, "plain_gemm", fl, lambda: G.coda_gemm_fp8(X, Wt, al, out=out),
               lambda: G.coda_gemm_fp8(X, Wt, al, out=out), "identity epilogue, both columns the same kernel",
               peak_mult=2.0)
        del p, X, Wt, out
    name = "fp8_swiglu_up_4096"
    if want(name):
        w = gen.WORKLOADS[name]
        p = gen.fp8_problem(w["M"], w["K"], w["N"], seed=0)
        X, Wt, al = u8(p["A"]), u8(p["B"]), p["sA"] * p["sB"]
        F = w["N"] // 2
        A = torch.empty((w["M"], F), dtype=torch.bfloat16, device=dev)
        GU = torch.empty((w["M"], 2 * F), dtype=torch.bfloat16, device=dev)
        fl = 2.0 * w["M"] * w["N"] * w["K"]
        report(name, "fwd", fl, lambda: G.coda_gemm_swiglu_fp8(X, Wt, al, out=A),
               lambda: (G.coda_gemm_fp8(X, Wt, al, out=GU), G.coda_unfused_swiglu(GU)), "1 vs 2 (no GU saved)",
               peak_mult=2.0)
        report(name, "fwd_save_gu", fl, lambda: G.coda_gemm_swiglu_fp8(X, Wt, al, out=A, gu=GU),
               lambda: (G.coda_gemm_fp8(X, Wt, al, out=GU), G.coda_unfused_swiglu(GU)),
               "1 vs 2 (GU saved for backward)", peak_mult=2.0)
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

        report(name, "fwd", fl, fused_ce, lambda: (G.coda_gemm_fp8(H, Wt, al, out=logits),
                                                   G.coda_unfused_ce_fwd(logits, y)),
               "GEMM+partials + reduce vs GEMM (bf16 logits) + CE", peak_mult=2.0)
        fused_ce()
        lse = st["lse"]
        report(name, "bwd_dlogits", fl, lambda: G.coda_gemm_ce_bwd_fp8(H, Wt, al, y, lse, 1.0 / w["M"], out=logits),
               lambda: (G.coda_gemm_fp8(H, Wt, al, out=logits), G.coda_unfused_ce_bwd(logits, y, lse, 1.0 / w["M"])),
               "recompute GEMM with dl epilogue vs recompute GEMM + CE-bwd kernel", peak_mult=2.0)
        del p, H, Wt, logits
    torch.cuda.empty_cache()


def block_suite(G, gen, dev, report, dm):
    """One period of the block-level chain (RoPE-path and SwiGLU-path
    GEMM-residual-RMSNorm-GEMM structures) at 16K tokens, forward and forward +
    backward, fused sequence vs unfused sequence. Inputs are drawn on the
    device (seeded torch generator) with the distributions of
    coda_inputs.block_problem: a host-side draw of the 70B-scale tensors would
    take longer than the timing itself."""
    import torch
    c = gen.WORKLOADS[f"block_d{dm}"]
    M, d, F, hd, rc, S = c["M"], c["d"], c["F"], c["head_dim"], c["rope_cols"], c["S"]
    g = torch.Generator(device=dev)
    g.manual_seed(0)

    def normal(shape, std=1.0, mean=0.0):
        t = torch.randn(shape, generator=g, device=dev, dtype=torch.float32)
        return (t * std + mean).to(torch.bfloat16)

    t = dict(P=normal((M, F)), Wd=normal((F, d), F ** -0.5), x=normal((M, d)), gamma1=normal((d,), 0.1, 1.0),
             Wqkv=normal((d, 3 * d), d ** -0.5), O=normal((M, d)), Wo=normal((d, d), d ** -0.5),
             gamma2=normal((d,), 0.1, 1.0), Wgu=normal((d, 2 * F), d ** -0.5), dQKV=normal((M, 3 * d)),
             gh=normal((M, d)), Wdn=normal((F, d), F ** -0.5))
    cos, sin = G.coda_rope_tables(S, hd, c["theta"], device=dev)
    fl_fwd = 2.0 * M * d * (3 * F + 4 * d)
    fused = G.CodaBlock(t, hd, rc, cos, sin, c["eps"])
    unfused = G.CodaBlock(t, hd, rc, cos, sin, c["eps"], unfused=True)
    name = f"block_d{dm}"
    report(name, "fwd", fl_fwd, fused.fwd, unfused.fwd_unfused, "6 fused launches vs 10 unfused")
    fused.fwd()
    unfused.fwd_unfused()
    report(name, "fwd_bwd", 3 * fl_fwd, lambda: fused.fwd().bwd(), lambda: unfused.fwd_unfused().bwd_unfused(),
           "19 fused launches vs 26 unfused")
    del t, fused, unfused
    torch.cuda.empty_cache()


if __name__ == "__main__":
    sys.exit(main())
