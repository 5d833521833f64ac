import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)
HERE = os.path.dirname(os.path.abspath(__file__))
if HERE not in sys.path:
    sys.path.insert(0, HERE)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a)")
    config.addinivalue_line("markers", "slow: long-running CPU oracle case")


def golden_path(name: str) -> str:
    return os.path.join(HERE, "golden", name)


@pytest.fixture(scope="session", autouse=True)
def _built_cpu_side():
    import oracle
    import synth
    oracle.build()
    synth.build(device=False)


@pytest.fixture(scope="session")
def k3_layer():
    """The full 896-expert K3-shaped layer (15.7 GB), generated on the GPU once."""
    import torch
    import synth
    from harness import device_layer_weights
    wts = device_layer_weights(synth.WORKLOADS["decode1"])
    yield wts
    del wts
    torch.cuda.empty_cache()
