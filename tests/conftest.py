import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (GB300, sm_103a)")


@pytest.fixture(scope="session")
def oracle_built():
    """Compile the CPU oracle only."""
    import oracle
    oracle.build()
    return True


@pytest.fixture(scope="session")
def built():
    """Compile the oracle, the product library and the input generator (in-tree)."""
    import oracle
    import radixattention_prefix_shared_tree_gb300._compile as comp
    import synth.native as sn
    oracle.build()
    comp.build()
    sn.build()
    return True


@pytest.fixture(scope="session")
def cuda(built):
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    return torch.device("cuda:0")


def pytest_terminal_summary(terminalreporter):
    """Every attention comparison's count of elements above 1e-2 and the
    largest excess (tests/tolerance.py records them)."""
    mod = sys.modules.get("tests.tolerance")
    if mod is None:
        return
    for line in mod.summary_lines():
        terminalreporter.write_line(line)
