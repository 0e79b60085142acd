import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line(
        "markers", "gpu: needs a CUDA GPU (sm_103a) and the built CUDA library")


@pytest.fixture(scope="session")
def golden_dir():
    return os.path.join(ROOT, "tests", "golden")


@pytest.fixture(scope="session")
def full_moe():
    """Router + 256 routed experts + 1 shared expert at full size (~22.6 GB of bf16
    weights), drawn once on the GPU and shared by every test that needs them."""
    import torch
    from hybrid_linear_attention_gated_gb300 import inputs
    from tests.gpu_common import FULL, f64, require_gpu
    dev = require_gpu()
    w = inputs.moe_weights(FULL["E"], FULL["Hd"], FULL["I"], FULL["n_shared"],
                           inputs.generator(3, dev), device=dev)
    w["W_r64"] = f64(w["W_r"])
    yield w
    w.clear()
    torch.cuda.empty_cache()
