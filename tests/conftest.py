import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and the built libq4k")


@pytest.fixture(scope="session")
def oracle_mod():
    import oracle
    oracle.build()
    return oracle


@pytest.fixture(scope="session")
def q4k():
    """The GPU library binding, built in-tree if needed. Fails loudly without it."""
    from gguf_q4_dequant_gb300 import build as q4k_build
    q4k_build.build()
    import gguf_q4_dequant_gb300 as lib
    return lib


# worst |err| / tolerance per (workload, M, X dtype), filled by the full-size
# parity tests and printed at the end of the run
PARITY = {}


@pytest.fixture(scope="session")
def parity_record():
    return PARITY


def pytest_terminal_summary(terminalreporter):
    if PARITY:
        terminalreporter.write_line("worst |err| / tolerance over the sampled outputs, per (workload, M, X dtype):")
        for k in sorted(PARITY):
            terminalreporter.write_line(f"  workload {k[0]} M={k[1]} {k[2]}: {PARITY[k]:.4f}")
