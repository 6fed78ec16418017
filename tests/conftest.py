import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (GB300)")
    config.addinivalue_line("markers", "slow: long-running oracle checks")


import pytest  # noqa: E402


@pytest.fixture(scope="session")
def tp():
    """The built library's binding (builds libtp.so in-tree if needed)."""
    from megatron_tensor_transformer_gate_gb300 import binding, build
    build.build()
    binding.lib()
    return binding
