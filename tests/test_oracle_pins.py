"""The oracle against facts that do not come from it (CPU only)."""

import numpy as np

import oracle
from oracle import kda, moe, layer, numerics
from tests.oracle_pins import (kda_pin_failures, spec_pin_failures, moe_pin_failures,
                               layer_pin_failures, fused_pin_failures,
                               extend_pin_failures)


def test_kda_step_pins():
    assert kda_pin_failures(kda.kda_step) == []


def test_spec_window_pins():
    assert spec_pin_failures(kda.kda_step, kda.spec_verify, kda.accept_prefix, kda.spec_replay) == []


def test_fused_replay_verify_pins():
    assert fused_pin_failures(kda.kda_step, kda.spec_replay_verify) == []


def test_extend_pins():
    assert extend_pin_failures(kda.kda_step, kda.extend) == []


def test_moe_pins():
    assert moe_pin_failures(moe.route_topk, moe.moe_forward, moe.swiglu_expert, moe.rmsnorm,
                            moe.linear, numerics.round_bf16, numerics.silu) == []


def test_layer_pins():
    assert layer_pin_failures(layer.qkvg_epilogue, layer.decode_layer, kda.kda_step,
                              moe.rmsnorm, numerics.round_bf16) == []


def test_oracle_is_independent_of_the_library():
    """The oracle imports nothing from the CUDA library package."""
    import os
    root = os.path.dirname(oracle.__file__)
    for name in os.listdir(root):
        if name.endswith(".py"):
            src = open(os.path.join(root, name)).read()
            assert "hybrid_linear_attention_gated_gb300" not in src, name
            assert "ctypes" not in src and "torch" not in src, name


def test_warm_state_is_sequential_steps():
    rng = np.random.default_rng(5)
    n, dk, dv = 6, 3, 2
    q, k = rng.standard_normal((n, dk)), rng.standard_normal((n, dk))
    v, al, be = rng.standard_normal((n, dv)), rng.uniform(0.1, 0.9, (n, dk)), rng.uniform(0, 1, n)
    S = np.zeros((dk, dv))
    for t in range(n):
        S, _ = kda.kda_step(S, q[t], k[t], v[t], al[t], be[t])
    assert np.array_equal(kda.warm_state((dk, dv), q, k, v, al, be), S)
