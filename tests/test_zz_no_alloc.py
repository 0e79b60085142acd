"""skinny_proj_splitk_noalloc against skinny_proj_splitk, through the C ABI.

The no-alloc entry point serves callers that cannot allocate device memory when they
run a projection (a server that fixes its memory budget at start-up, a plugin whose host
owns every allocation): its split-K partials live in one fixed device array inside the
library instead of a caller workspace.  It must give the workspace version's results,
call after call, even though every call reuses the partials the previous call left.
This file is collected last so that a run stopping at the first failure has run every
other test first.
"""

import pytest
import torch

import oracle
from hybrid_linear_attention_gated_gb300 import hla, inputs
from tests.gpu_common import PROJ_FROB_REL_BF16, PROJ_FROB_REL_F32, f64, max_rel, require_gpu

pytestmark = pytest.mark.gpu


def _case(dev, M, N, K, out, res, seed):
    g = inputs.generator(seed)
    x = inputs.activations(M, K, g).to(dev)
    W = inputs.weight((N, K), g).to(dev)
    r = inputs.activations(M, N, g).to(dev) if res else None
    dt = torch.bfloat16 if out == hla.HLA_BF16 else torch.float32
    return x, W, r, torch.empty(M, N, device=dev, dtype=dt), torch.empty(M, N, device=dev, dtype=dt)


def test_noalloc_matches_workspace_version_on_consecutive_calls():
    dev = require_gpu()
    # two calls in a row with different shapes; both split K, so both go through the array
    cases = [(4, 1024, 2048, hla.HLA_F32, False, 61), (64, 7168, 4096, hla.HLA_BF16, True, 62)]
    for M, N, K, out, res, seed in cases:
        x, W, r, y_ref, y = _case(dev, M, N, K, out, res, seed)
        nb = hla.skinny_proj_splitk_workspace_size(M, N, K, 0)
        assert 0 < nb <= hla.HLA_NOALLOC_SCRATCH_BYTES
        ws = torch.empty(nb, dtype=torch.uint8, device=dev)
        hla.skinny_proj_splitk(M, N, K, x, W, r, y_ref, out, 0, ws, nb)
        ws_variant = hla.hla_last_variant()
        hla.skinny_proj_splitk_noalloc(M, N, K, x, W, r, y, out, 0)
        variant = hla.hla_last_variant()
        torch.cuda.synchronize()
        # a tensor-core launch (M = 64) reports a bounded wait that gave up only here
        assert hla.hla_device_status() == 0
        assert variant.startswith("skinny_proj_noalloc") and "split1>" not in variant
        # the same kernels with the same split, in the same order: the same bits
        assert variant[len("skinny_proj_noalloc"):] == ws_variant[len("skinny_proj"):], (variant, ws_variant)
        assert torch.equal(y, y_ref)
        # and element by element against the oracle's x W^T (+ residual)
        ref = oracle.moe.linear(f64(x), f64(W)) + (f64(r) if res else 0.0)
        tol = PROJ_FROB_REL_BF16 if out == hla.HLA_BF16 else PROJ_FROB_REL_F32
        assert max_rel(f64(y), ref) < tol


def test_noalloc_rejects_partials_larger_than_its_array():
    dev = require_gpu()
    M, N, K, split = 64, 16416, 7168, 8  # 8 x 64 x 16416 x 4 bytes > 16 MiB
    x = torch.zeros(M, K, dtype=torch.bfloat16, device=dev)
    W = torch.zeros(N, K, dtype=torch.bfloat16, device=dev)
    y = torch.full((M, N), 7.0, device=dev)
    n0 = hla.hla_launch_count()
    status = hla.load().skinny_proj_splitk_noalloc(M, N, K, x.data_ptr(), W.data_ptr(), None,
                                                   y.data_ptr(), hla.HLA_F32, split,
                                                   torch.cuda.current_stream().cuda_stream)
    assert status == 4  # HLA_ERR_WORKSPACE
    assert hla.hla_launch_count() == n0
    torch.cuda.synchronize()
    assert torch.all(y == 7.0)
