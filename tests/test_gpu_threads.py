"""Host threads launching concurrently.

A fresh process starts four threads before any kernel of the library has run,
so the per-kernel first-use set-up (shared-memory attribute, cluster
occupancy query), the creation of each stream's stream-K workspace and the
launch settings are exercised under concurrency.
Each thread runs a mix of fused kernels and auxiliary reductions on its own
stream; one thread keeps switching the tile setting between automatic and
SM pairs (the same variant at these shapes, so bit-identical results). Afterwards the same calls
run serially, and every concurrent result must equal its serial twin bit for
bit."""
import os
import subprocess
import sys
import textwrap

import pytest

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

CHILD = textwrap.dedent("""
    import sys, threading
    import torch
    import gemm_epilogue_transformer_gb300 as coda

    coda.coda_init(0)
    coda.coda_set_stream_k(2)  # the split wherever it applies: only the 1800 x 3400 x 1096 GEMM below
    g = torch.Generator(device="cuda").manual_seed(5)
    def bf(*s, std=1.0):
        return (torch.randn(*s, device="cuda", generator=g) * std).bfloat16()
    x, W0, z = bf(1000, 512), bf(512, 768, std=512 ** -0.5), bf(1000, 768)
    gam = (1 + 0.1 * torch.randn(768, device="cuda", generator=g)).bfloat16()
    W1 = bf(768, 640, std=768 ** -0.5)
    X, Wr = bf(700, 384), bf(384, 1536, std=384 ** -0.5)
    Wgu = bf(384, 2 * 520, std=384 ** -0.5)
    H, Wv = bf(600, 256), bf(256, 3000, std=256 ** -0.5)
    y = torch.randint(0, 3000, (600,), device="cuda", dtype=torch.int32, generator=g)
    Ak, Bk = bf(1800, 1096), bf(1096, 3400, std=1096 ** -0.5)
    torch.cuda.synchronize()

    def step():
        c, s = coda.coda_rope_tables(1024, 128, 1e4)
        h1, h2, psq = coda.coda_gemm_res_rmsprep(x, W0, z, gam)
        r = coda.coda_rms_reduce(psq, 768, 1e-6)
        Y = coda.coda_gemm_rowscale(h2, W1, r)
        q = coda.coda_gemm_rope(X, Wr, c, s, 128, 1024)
        a, gu = coda.coda_gemm_swiglu(X, Wgu, want_gu=True)
        pm, ps, pa, t = coda.coda_gemm_ce_lse(H, Wv, y)
        lse, lrow, lmean, am = coda.coda_ce_reduce(pm, ps, pa, t)
        Ck = coda.coda_gemm(Ak, Bk)   # stream-K split: each stream's first use creates its workspace
        return [h1, h2, r, Y, q, a, gu, lse, lrow, lmean, am, Ck]

    N_THREADS, REPS = 4, 6
    results = [[] for _ in range(N_THREADS)]
    errors = []
    start = threading.Barrier(N_THREADS)

    def worker(i):
        try:
            st = torch.cuda.Stream()
            start.wait()
            with torch.cuda.stream(st):
                for rep in range(REPS):
                    if i == 0:
                        coda.coda_set_cta_group(2 if rep % 2 else 0)
                    results[i].append([o.clone() for o in step()])
            st.synchronize()
        except Exception as e:  # reported by the parent through the exit code
            errors.append(f"thread {i}: {e!r}")

    threads = [threading.Thread(target=worker, args=(i,)) for i in range(N_THREADS)]
    for t in threads:
        t.start()
    for t in threads:
        t.join()
    torch.cuda.synchronize()
    if errors:
        print("\\n".join(errors))
        sys.exit(2)
    coda.coda_set_cta_group(0)
    ref = [o.clone() for o in step()]
    torch.cuda.synchronize()
    bad = 0
    for i in range(N_THREADS):
        for rep, outs in enumerate(results[i]):
            for k, (o, e) in enumerate(zip(outs, ref)):
                if not torch.equal(o, e):
                    bad += 1
                    print(f"thread {i} rep {rep} output {k} differs")
    status = coda.coda_device_status(clear=True)
    print("status", status, "mismatches", bad)
    sys.exit(0 if bad == 0 and status == 0 else 3)
""")


def test_concurrent_host_threads(coda):
    env = dict(os.environ)
    env["PYTHONPATH"] = ROOT + os.pathsep + env.get("PYTHONPATH", "")
    r = subprocess.run([sys.executable, "-c", CHILD], cwd=ROOT, env=env, capture_output=True, text=True,
                       timeout=300)
    assert r.returncode == 0, f"exit {r.returncode}\n{r.stdout[-3000:]}\n{r.stderr[-3000:]}"
