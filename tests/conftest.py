import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and the built library")
    config.addinivalue_line("markers", "slow: full-size workloads")
    # build the CUDA library (nvcc cross-compiles without a GPU) and the C
    # oracle before any test module imports them
    import __graft_entry__
    __graft_entry__._build_module().build()
    import oracle
    oracle.build()
