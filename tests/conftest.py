import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (GB300, sm_103a); parity tests through the C ABI")
    config.addinivalue_line("markers", "slow: long-running CPU test")


@pytest.fixture(scope="session", autouse=True)
def _built_cpu_libs():
    """Compile the oracle, the row generator (gcc) and libhs.so (nvcc, sm_103a) once."""
    import oracle
    import workloads
    from hierarchical_sparse_attention_gb300 import build as hs_build
    oracle.build()
    workloads.build_rowgen()
    hs_build.build()
    yield
