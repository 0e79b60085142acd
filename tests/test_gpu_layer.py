"""The full hybrid decode layer (hidden 7168, 32 KDA heads of 128, 256 experts top-8 + 1
shared) through the C-ABI executor, against the oracle's composed layer on every sequence
(a sequence whose router logits hold a near tie is compared on its state only)."""

import numpy as np
import pytest
import torch

import oracle
from hybrid_linear_attention_gated_gb300 import hla, inputs
from tests.gpu_common import (FULL, LAYER_FROB_REL, ExpertCache, f64, frob_rel, require_gpu,
                              warm_states)

pytestmark = pytest.mark.gpu

H, D = 32, 128
ROUTER_MARGIN = 1e-3   # y is not compared for a token whose oracle top-(k+1) logits are closer than this


@pytest.fixture(scope="module")
def dev():
    return require_gpu()


@pytest.fixture(scope="module")
def layer(dev, full_moe):
    w = inputs.layer_weights(FULL["Hd"], H, D, D, inputs.generator(4, dev), device=dev)
    w.update({k: full_moe[k] for k in ("W_r", "W_gate", "W_up", "W_down", "Ws_gate", "Ws_up", "Ws_down")})
    L = hla.make_layer(FULL["Hd"], H, D, D, FULL["E"], FULL["k"], FULL["I"], FULL["n_shared"], 1e-6, w)
    p = dict(H=H, dk=D, dv=D, top_k=FULL["k"], eps=1e-6, gamma_attn=f64(w["gamma_attn"]),
             gamma_moe=f64(w["gamma_moe"]), W_qkvgb=f64(w["W_qkvgb"]), W_o=f64(w["W_o"]),
             W_r=full_moe["W_r64"])
    return w, L, p


def _run(dev, L, M, x, S, prefetch=False):
    y = torch.empty(M, FULL["Hd"], dtype=torch.bfloat16, device=dev)
    nb = hla.hla_decode_layer_workspace_size(L, M)
    ws = torch.empty(nb, dtype=torch.uint8, device=dev)
    side = torch.cuda.Stream() if prefetch else 0
    hla.hla_decode_layer(L, M, x, S, None, y, ws, nb, prefetch_stream=side)
    return y


@pytest.mark.parametrize("M", [1, 8, 64])
def test_decode_layer(dev, full_moe, layer, M):
    w, L, p = layer
    x = inputs.activations(M, FULL["Hd"], inputs.generator(4000 + M))
    S0 = warm_states(4, M, H, D)
    S = S0.to(dev)
    y = _run(dev, L, M, x.to(dev), S)
    torch.cuda.synchronize()
    assert hla.hla_last_variant().startswith("decode_layer")
    cache = ExpertCache(full_moe)
    y_ref, S_ref, aux = oracle.layer.decode_layer(f64(x), f64(S0), p, cache, cache.shared())
    S_got, y_got = f64(S), f64(y)
    ties = 0
    for m in range(M):
        # the state does not depend on the routing: every sequence
        assert frob_rel(S_got[m], S_ref[m]) < LAYER_FROB_REL, m
        top = np.sort(aux["logits"][m])[::-1][:FULL["k"] + 1]
        if np.any(-np.diff(top) < ROUTER_MARGIN):
            ties += 1
            continue  # a near tie in routing: the two sides may legitimately pick differently
        assert frob_rel(y_got[m], y_ref[m]) < LAYER_FROB_REL, m
    assert ties <= M // 4, ties


@pytest.mark.parametrize("M,mask", [(8, "7"), (64, None), (64, "7")])
def test_layer_prefetch_is_bitwise_neutral(dev, layer, M, mask, monkeypatch):
    """Every prefetch choice (default policy, or all of them forced) leaves results bit-identical."""
    if mask is not None:
        monkeypatch.setenv("HLA_PREFETCH_MASK", mask)
    w, L, p = layer
    x = inputs.activations(M, FULL["Hd"], inputs.generator(4100 + M)).to(dev)
    S0 = warm_states(4, M, H, D)
    S1, S2 = S0.to(dev), S0.to(dev)
    y1 = _run(dev, L, M, x, S1)
    y2 = _run(dev, L, M, x, S2, prefetch=True)
    torch.cuda.synchronize()
    assert torch.equal(y1, y2) and torch.equal(S1, S2)


@pytest.mark.parametrize("M", [8, 64])
def test_layer_in_cuda_graph_matches_eager(dev, layer, M):
    """Captured with its prefetch stream (at batch 64 the side-stream fork/join is captured too)."""
    w, L, p = layer
    x = inputs.activations(M, FULL["Hd"], inputs.generator(4200 + M)).to(dev)
    S0 = warm_states(4, M, H, D)
    S_eager = S0.to(dev)
    y_eager = _run(dev, L, M, x, S_eager, prefetch=True)
    S_graph = S0.to(dev)
    y = torch.empty(M, FULL["Hd"], dtype=torch.bfloat16, device=dev)
    nb = hla.hla_decode_layer_workspace_size(L, M)
    ws = torch.empty(nb, dtype=torch.uint8, device=dev)
    side = torch.cuda.Stream()
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    stream = torch.cuda.Stream()
    with torch.cuda.stream(stream):
        with torch.cuda.graph(g, stream=stream):
            hla.hla_decode_layer(L, M, x, S_graph, None, y, ws, nb, prefetch_stream=side)
    S_graph.copy_(S0.to(dev))
    g.replay()
    torch.cuda.synchronize()
    assert torch.equal(y, y_eager) and torch.equal(S_graph, S_eager)


@pytest.mark.parametrize("M", [1, 64])
def test_layer_shared_experts_on_side_stream(dev, layer, M, monkeypatch):
    """HLA_SHARED_STREAM=1: the layer forks the shared experts onto its side stream before the
    router.  The state is untouched by the placement (bit-identical), the output is close to
    the default placement, and a captured CUDA graph reproduces the eager call bit for bit."""
    w, L, p = layer
    x = inputs.activations(M, FULL["Hd"], inputs.generator(4400 + M)).to(dev)
    S0 = warm_states(4, M, H, D)
    S_def = S0.to(dev)
    y_def = _run(dev, L, M, x, S_def, prefetch=True)
    monkeypatch.setenv("HLA_SHARED_STREAM", "1")
    S_side = S0.to(dev)
    y_side = _run(dev, L, M, x, S_side, prefetch=True)
    torch.cuda.synchronize()
    assert torch.equal(S_side, S_def)
    assert frob_rel(f64(y_side), f64(y_def)) < 2e-3
    y = torch.empty(M, FULL["Hd"], dtype=torch.bfloat16, device=dev)
    nb = hla.hla_decode_layer_workspace_size(L, M)
    ws = torch.empty(nb, dtype=torch.uint8, device=dev)
    side = torch.cuda.Stream()
    S_graph = S0.to(dev)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    stream = torch.cuda.Stream()
    with torch.cuda.stream(stream):
        with torch.cuda.graph(g, stream=stream):
            hla.hla_decode_layer(L, M, x, S_graph, None, y, ws, nb, prefetch_stream=side)
    S_graph.copy_(S0.to(dev))
    g.replay()
    torch.cuda.synchronize()
    assert torch.equal(y, y_side) and torch.equal(S_graph, S_side)



@pytest.mark.parametrize("M", [1, 8, 64])
def test_layer_programmatic_launch_is_bitwise_neutral(dev, layer, M, monkeypatch):
    """The layer's kernels chained by programmatic dependent launch (each loads its weights or
    state before waiting for its predecessor) give the same bits as plain launches, eager and
    captured in a CUDA graph with the prefetch stream."""
    w, L, p = layer
    x = inputs.activations(M, FULL["Hd"], inputs.generator(4600 + M)).to(dev)
    S0 = warm_states(4, M, H, D)
    out = {}
    for mode in ("0", "1"):
        monkeypatch.setenv("HLA_PDL", mode)
        S = S0.to(dev)
        y = _run(dev, L, M, x, S, prefetch=True)
        out[mode] = (y, S, hla.hla_last_variant())
    torch.cuda.synchronize()
    assert "<pdl>" in out["1"][2] and "<pdl>" not in out["0"][2]
    assert torch.equal(out["0"][0], out["1"][0]) and torch.equal(out["0"][1], out["1"][1])
    monkeypatch.setenv("HLA_PDL", "1")
    y = torch.empty(M, FULL["Hd"], dtype=torch.bfloat16, device=dev)
    nb = hla.hla_decode_layer_workspace_size(L, M)
    ws = torch.empty(nb, dtype=torch.uint8, device=dev)
    side = torch.cuda.Stream()
    S_graph = S0.to(dev)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    stream = torch.cuda.Stream()
    with torch.cuda.stream(stream):
        with torch.cuda.graph(g, stream=stream):
            hla.hla_decode_layer(L, M, x, S_graph, None, y, ws, nb, prefetch_stream=side)
    for _ in range(2):  # replays after the first see the previous replay's workspace contents
        S_graph.copy_(S0.to(dev))
        g.replay()
        torch.cuda.synchronize()
        assert torch.equal(y, out["0"][0]) and torch.equal(S_graph, out["0"][1])


@pytest.mark.parametrize("M", [1, 8, 64])
def test_layer_state_pool_matches_identity(dev, layer, M):
    """The layer with its states in a larger slot pool (state_idx: a seeded permutation) gives the
    bits of the layer on the same states stored in order, and leaves every other slot untouched."""
    w, L, p = layer
    x = inputs.activations(M, FULL["Hd"], inputs.generator(4800 + M)).to(dev)
    S0 = warm_states(6, M, H, D)
    ref_S = S0.to(dev)
    ref_y = _run(dev, L, M, x, ref_S)
    P = M + 5
    perm = torch.randperm(P, generator=inputs.generator(4801 + M))[:M].to(torch.int32)
    pool0 = torch.randn(P, H, D, D, generator=inputs.generator(4802 + M)).mul_(0.05)
    pool0[perm.long()] = S0
    pool = pool0.to(dev)
    y = torch.empty(M, FULL["Hd"], dtype=torch.bfloat16, device=dev)
    nb = hla.hla_decode_layer_workspace_size(L, M)
    ws = torch.empty(nb, dtype=torch.uint8, device=dev)
    hla.hla_decode_layer(L, M, x, pool, perm.to(dev), y, ws, nb, prefetch_stream=0)
    torch.cuda.synchronize()
    assert torch.equal(y, ref_y)
    got = pool.cpu()
    assert torch.equal(got[perm.long()], ref_S.cpu())
    others = torch.ones(P, dtype=torch.bool)
    others[perm.long()] = False
    assert torch.equal(got[others], pool0[others])
