"""The failure-detection path of the tensor-core projections, without a real stall.

A bounded device wait that gives up must not fail the launch or poison the context: it
records HLA_ERR_DEVICE_TIMEOUT in the device status word, which hla_device_status() reports
once and clears.  The test hook makes one wait give up on a barrier that nothing arrives at,
before any tensor memory is allocated or any copy or MMA is issued, so nothing is in flight
when the wait runs out.  The next launch without the hook must compute the right result.
"""

import pytest
import torch

import oracle
from hybrid_linear_attention_gated_gb300 import hla, inputs
from tests.gpu_common import PROJ_FROB_REL_F32, f64, max_rel, require_gpu

pytestmark = pytest.mark.gpu

HLA_ERR_DEVICE_TIMEOUT = 6


def test_forced_wait_timeout_is_reported_once_and_the_context_stays_usable():
    dev = require_gpu()
    M, N, K = 64, 1024, 2048  # 64 tokens: the tensor-core path
    g = inputs.generator(77)
    x = inputs.activations(M, K, g).to(dev)
    W = inputs.weight((N, K), g).to(dev)
    y = torch.full((M, N), 7.0, device=dev)
    torch.cuda.synchronize()
    assert hla.hla_device_status() == 0
    try:
        hla.hla_test_force_wait_timeout(1)
        # split 1: no workspace, the kernel writes y directly (here: it writes nothing)
        hla.skinny_proj_splitk(M, N, K, x, W, None, y, hla.HLA_F32, 1, None, 0)
        assert hla.hla_last_variant().startswith("skinny_proj<tt64,")
        torch.cuda.synchronize()
    finally:
        hla.hla_test_force_wait_timeout(0)
    assert hla.hla_device_status() == HLA_ERR_DEVICE_TIMEOUT   # reported ...
    assert hla.hla_device_status() == 0                        # ... once, then cleared
    assert torch.all(y == 7.0)                                 # the given-up launch wrote nothing

    # the context is still usable and the next launch is right
    hla.skinny_proj_splitk(M, N, K, x, W, None, y, hla.HLA_F32, 1, None, 0)
    torch.cuda.synchronize()
    assert hla.hla_device_status() == 0
    assert max_rel(f64(y), oracle.moe.linear(f64(x), f64(W))) < PROJ_FROB_REL_F32
