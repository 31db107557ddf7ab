import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (GB300, sm_103a) and the built CUDA library")


import pytest  # noqa: E402


@pytest.fixture
def stall_hooks(monkeypatch):
    """(on, off): switch the kernels' bounded-wait test hooks on (every pipeline stage expects 16
    bytes no copy delivers and every wait gives up after 20 ms) and off again.  The library reads
    them from the environment when asked to (pkv_debug_reload_env); they are off after the test
    whatever happens."""
    import paged_kv_cache_266_gb300 as pkv

    def on():
        monkeypatch.setenv("PKV_TEST_WAIT_LIMIT_MS", "20")
        monkeypatch.setenv("PKV_TEST_STALL_COPIES", "1")
        pkv.pkv_debug_reload_env()

    def off():
        monkeypatch.delenv("PKV_TEST_WAIT_LIMIT_MS", raising=False)
        monkeypatch.delenv("PKV_TEST_STALL_COPIES", raising=False)
        pkv.pkv_debug_reload_env()

    yield on, off
    off()
