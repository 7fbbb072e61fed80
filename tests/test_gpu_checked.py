"""The checked build (libcoda_checked.so, compiled with CODA_CHECKED=1) tests
the index of every direct global load and store of the fused epilogues against
the extent of the tensor it touches and sets CODA_DEVST_BOUNDS instead of
making the access (the stream-K split's partial accumulators and arrival words
included). This test reruns the fused, edge, sentinel, block-chain, FP8 and
stream-K parity suites in a child process that loads the checked build: every
parity assertion must still hold and no read of the status word may show the
bounds bit (tests/conftest.py fails any such read)."""
import os
import subprocess
import sys

import pytest

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SUITES = ["tests/test_gpu_fused.py", "tests/test_gpu_edges.py", "tests/test_gpu_sentinels.py",
          "tests/test_gpu_block.py", "tests/test_gpu_fp8.py", "tests/test_gpu_streamk.py"]


def test_parity_suites_on_the_checked_build():
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from gemm_epilogue_transformer_gb300 import build_lib
    path = build_lib.build(checked=True)
    env = dict(os.environ, CODA_LIBRARY=path)
    probe = subprocess.run([sys.executable, "-c", "import gemm_epilogue_transformer_gb300._lib as L; "
                            "print(L.LIB_PATH); L.load()"], cwd=ROOT, env=env, capture_output=True, text=True,
                           timeout=300)
    assert probe.returncode == 0 and probe.stdout.strip() == path, probe.stdout + probe.stderr
    r = subprocess.run([sys.executable, "-m", "pytest", "-x", "-q", "-m", "gpu", "-p", "no:cacheprovider", *SUITES],
                       cwd=ROOT, env=env, capture_output=True, text=True, timeout=1500)
    assert r.returncode == 0, r.stdout[-4000:] + r.stderr[-2000:]
    assert " passed" in r.stdout
