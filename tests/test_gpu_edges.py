"""Edge cases on the GPU: the rule's degenerate cases, the largest sizes the C ABI accepts, and
the widest router and expert set, each against the oracle (or an exact closed form)."""

import numpy as np
import pytest
import torch

import oracle
from hybrid_linear_attention_gated_gb300 import hla, inputs
from tests.gpu_common import (FULL, KDA_MAX_REL, LAYER_FROB_REL, MOE_FROB_REL, ROUTER_W_REL,
                              ExpertCache, f64, frob_rel, max_rel, require_gpu, warm_states)
from tests.test_gpu_moe import tie_free_activations

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def dev():
    return require_gpu()


def _decode(S, u, dev):
    B, H, d = u["q"].shape
    o = torch.empty(B, H, d, device=dev)
    hla.kda_decode_step(B, H, d, d, S, None, u["q"], u["k"], u["v"], u["alpha"], u["beta"], o)
    torch.cuda.synchronize()
    return o


@pytest.mark.parametrize("d", [64, 128])
def test_kda_no_write_no_decay_leaves_state_bitwise(dev, d):
    """beta = 0 and alpha = 1: the state is untouched bit for bit and o = S^T q."""
    B, H = 2, 4
    S0 = warm_states(11, B, H, d)
    u = inputs.kda_inputs((B,), H, d, d, inputs.generator(110 + d))
    u["alpha"] = torch.ones_like(u["alpha"])
    u["beta"] = torch.zeros_like(u["beta"])
    ud = {k: v.to(dev) for k, v in u.items()}
    S = S0.to(dev)
    o = _decode(S, ud, dev)
    assert torch.equal(S.cpu(), S0)
    o_ref = np.einsum("bhij,bhi->bhj", f64(S0), f64(u["q"]))
    assert max_rel(f64(o), o_ref) < KDA_MAX_REL


def test_kda_no_write_is_exact_decay(dev):
    """beta = 0: the new state is diag(alpha) S, each entry the correctly rounded fp32 product,
    so it equals the oracle's fp64 product rounded to fp32 exactly."""
    B, H, d = 3, 8, 128
    S0 = warm_states(12, B, H, d)
    u = inputs.kda_inputs((B,), H, d, d, inputs.generator(120))
    u["beta"] = torch.zeros_like(u["beta"])
    ud = {k: v.to(dev) for k, v in u.items()}
    S = S0.to(dev)
    _decode(S, ud, dev)
    S_ref, _ = oracle.kda.kda_step(f64(S0), f64(u["q"]), f64(u["k"]), f64(u["v"]), f64(u["alpha"]),
                                   f64(u["beta"]))
    assert np.array_equal(S.cpu().numpy(), oracle.numerics.round_f32(S_ref).astype(np.float32))


def test_kda_decode_batch_256(dev):
    """256 sequences x 32 heads (536 MB of state): sampled heads against the oracle."""
    B, H, d = 256, 32, 128
    S0 = warm_states(13, B, H, d)
    u = inputs.kda_inputs((B,), H, d, d, inputs.generator(130))
    S = S0.to(dev)
    o = _decode(S, {k: v.to(dev) for k, v in u.items()}, dev)
    for b, h in [(0, 0), (77, 5), (128, 31), (255, 17)]:
        S_ref, o_ref = oracle.kda.kda_step(f64(S0[b, h]), f64(u["q"][b, h]), f64(u["k"][b, h]),
                                           f64(u["v"][b, h]), f64(u["alpha"][b, h]), f64(u["beta"][b, h]))
        assert max_rel(f64(S[b, h]), S_ref) < KDA_MAX_REL
        assert max_rel(f64(o[b, h]), o_ref) < KDA_MAX_REL


def _moe_case(dev, M, Hd, I, E, k, ns, seed):
    g = inputs.generator(seed)
    w = inputs.moe_weights(E, Hd, I, ns, g)
    x, _ = tie_free_activations(M, Hd, f64(w["W_r"]), k, seed)
    wd = {kk: vv.to(dev) for kk, vv in w.items()}
    xd = x.to(dev)
    idx = torch.empty(M, k, dtype=torch.int32, device=dev)
    wt = torch.empty(M, k, device=dev)
    rb = hla.moe_route_topk_workspace_size(M, Hd, E)
    rws = torch.empty(max(rb, 256), dtype=torch.uint8, device=dev)
    hla.moe_route_topk(M, Hd, E, k, xd, wd["W_r"], idx, wt, None, rws, rb)
    res = inputs.activations(M, Hd, g).to(dev)
    y = torch.empty(M, Hd, dtype=torch.bfloat16, device=dev)
    nb = hla.moe_expert_forward_workspace_size(M, Hd, I, E, k, ns)
    ws = torch.empty(nb, dtype=torch.uint8, device=dev)
    hla.moe_expert_forward(M, Hd, I, E, k, ns, xd, idx, wt, wd["W_gate"], wd["W_up"], wd["W_down"],
                           wd.get("Ws_gate"), wd.get("Ws_up"), wd.get("Ws_down"), res, y, ws, nb)
    torch.cuda.synchronize()
    idx_ref, w_ref, _ = oracle.moe.route_topk(f64(x), f64(w["W_r"]), k)
    assert np.array_equal(idx.cpu().numpy(), idx_ref)
    assert max_rel(f64(wt), w_ref) < ROUTER_W_REL
    shared = [(f64(w["Ws_gate"][s]), f64(w["Ws_up"][s]), f64(w["Ws_down"][s])) for s in range(ns)]
    y_ref = oracle.moe.moe_forward(f64(x), idx_ref, w_ref,
                                   (f64(w["W_gate"]), f64(w["W_up"]), f64(w["W_down"])), shared,
                                   residual=f64(res))
    assert frob_rel(f64(y), y_ref) < MOE_FROB_REL


def test_widest_router_and_expert_set(dev):
    """1022 routed experts + 2 shared (the 1024-unit limit), top-16 (the largest k)."""
    _moe_case(dev, M=3, Hd=256, I=128, E=1022, k=16, ns=2, seed=140)


def test_moe_256_tokens(dev):
    """256 tokens (the largest batch): 16 token groups for the shared expert, several per
    routed expert."""
    _moe_case(dev, M=256, Hd=256, I=128, E=16, k=2, ns=1, seed=141)


def test_decode_layer_256_tokens(dev, full_moe):
    """The full-size layer at its largest batch, 256 tokens, on sampled sequences."""
    M, H, D = 256, 32, 128
    w = inputs.layer_weights(FULL["Hd"], H, D, D, inputs.generator(4, dev), device=dev)
    w.update({k: full_moe[k] for k in ("W_r", "W_gate", "W_up", "W_down", "Ws_gate", "Ws_up", "Ws_down")})
    L = hla.make_layer(FULL["Hd"], H, D, D, FULL["E"], FULL["k"], FULL["I"], FULL["n_shared"], 1e-6, w)
    p = dict(H=H, dk=D, dv=D, top_k=FULL["k"], eps=1e-6, gamma_attn=f64(w["gamma_attn"]),
             gamma_moe=f64(w["gamma_moe"]), W_qkvgb=f64(w["W_qkvgb"]), W_o=f64(w["W_o"]),
             W_r=full_moe["W_r64"])
    x = inputs.activations(M, FULL["Hd"], inputs.generator(4500))
    S0 = warm_states(4, M, H, D)
    S = S0.to(dev)
    y = torch.empty(M, FULL["Hd"], dtype=torch.bfloat16, device=dev)
    nb = hla.hla_decode_layer_workspace_size(L, M)
    ws = torch.empty(nb, dtype=torch.uint8, device=dev)
    hla.hla_decode_layer(L, M, x.to(dev), S, None, y, ws, nb, prefetch_stream=torch.cuda.Stream())
    torch.cuda.synchronize()
    cache = ExpertCache(full_moe)
    checked = 0
    for m in (0, 101, 200, 255):
        y_ref, S_ref, aux = oracle.layer.decode_layer(f64(x)[m:m + 1], f64(S0)[m:m + 1], p, cache,
                                                       cache.shared())
        top = np.sort(aux["logits"][0])[::-1][:FULL["k"] + 1]
        if np.any(-np.diff(top) < 1e-3):
            continue  # a near tie in routing: the two sides may legitimately pick differently
        assert frob_rel(f64(y)[m:m + 1], y_ref) < LAYER_FROB_REL, m
        assert frob_rel(f64(S)[m:m + 1], S_ref) < LAYER_FROB_REL, m
        checked += 1
    assert checked >= 1
