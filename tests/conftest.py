import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a GB300 (sm_103a) GPU and the built CUDA library")
    config.addinivalue_line("markers", "slow: full-size parity case (minutes)")


import pytest  # noqa: E402


@pytest.fixture(scope="session")
def coda():
    """The product binding on cuda:0, built for sm_103a if needed."""
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from gemm_epilogue_transformer_gb300 import build_lib
    build_lib.build()
    import gemm_epilogue_transformer_gb300 as G
    if os.environ.get("CODA_LIBRARY"):
        # a run on the checked build: any read of the status word that shows
        # CODA_DEVST_BOUNDS fails at once, even in a test that clears the word
        read = G.coda_device_status

        def checked_status(clear=True):
            st = read(clear)
            assert st < 0 or not st & 4, f"checked build: an epilogue access fell outside its tensor (status {st})"
            return st
        G.coda_device_status = checked_status
    G.coda_init(0)
    G.coda_device_status(clear=True)
    yield G
    assert G.coda_device_status(clear=True) == 0, "device status word set during the tests"
