import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (GB300, sm_103a)")
    # The binding loads the compiled library at import; build it first if it is
    # missing or stale (nvcc is present wherever the tests run).
    from paged_kv_cache_308_gb300 import build
    build.build()
