import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

GOLDEN = os.path.join(ROOT, "tests", "golden")


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (B300, sm_103a)")


def read_golden(name):
    """Parse a ``key = values  # comment`` fixture into {key: [floats]}."""
    out = {}
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.split("#", 1)[0].strip()
            if not line or "=" not in line:
                continue
            k, v = line.split("=", 1)
            out[k.strip()] = [float(x) for x in v.split()]
    return out


@pytest.fixture(scope="session")
def cuda_lib():
    """The compiled library on a GPU machine (skips when no GPU is present)."""
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from decode_attention_kv_softmax_b300 import kvdec
    kvdec.load()
    return kvdec
