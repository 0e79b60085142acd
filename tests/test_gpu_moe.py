"""Skinny projections, RMSNorm, router top-k and routed + shared experts on the GPU vs the oracle."""

import numpy as np
import pytest
import torch

import oracle
from hybrid_linear_attention_gated_gb300 import hla, inputs
from tests.gpu_common import (FULL, MOE_FROB_REL, PROJ_FROB_REL_BF16, PROJ_FROB_REL_F32,
                              ROUTER_W_REL, ExpertCache, f64, frob_rel, max_rel, require_gpu)

pytestmark = pytest.mark.gpu

TIE_GAP = 1e-5  # minimum gap between adjacent top-(k+1) sigmoid scores of a test token


@pytest.fixture(scope="module")
def dev():
    return require_gpu()


def _ws(nbytes, dev):
    return torch.empty(max(int(nbytes), 256), dtype=torch.uint8, device=dev)


def tie_free_activations(M, Hd, W_r64, k, seed, device="cpu"):
    """x ~ N(0,1) bf16 [M, Hd]; a token whose top-(k+1) oracle scores come within TIE_GAP of
    each other is redrawn from the next sub-seed.  Returns (x, number of redraws)."""
    rows, redraws = [], 0
    for m in range(M):
        sub = 0
        while True:
            x = inputs.activations(1, Hd, inputs.generator(seed * 1000 + m * 97 + sub))
            s = np.sort(oracle.numerics.sigmoid(f64(x) @ W_r64.T)[0])[::-1][:k + 1]
            if np.all(-np.diff(s) >= TIE_GAP):
                break
            sub += 1
            redraws += 1
        rows.append(x)
    return torch.cat(rows).to(device), redraws


# ----------------------------------------------------------------------------- projections

@pytest.mark.parametrize("M,N,K,split,res,out", [
    (1, 7168, 4096, 0, True, hla.HLA_BF16), (2, 256, 7168, 0, False, hla.HLA_F32),
    (3, 1028, 256, 1, False, hla.HLA_F32), (13, 1000, 512, 3, True, hla.HLA_BF16),
    (64, 7168, 4096, 0, True, hla.HLA_BF16), (64, 2048, 7168, 2, False, hla.HLA_F32),
    (256, 96, 256, 0, False, hla.HLA_F32), (9, 16, 32, 1, True, hla.HLA_F32)])
def test_skinny_proj(dev, M, N, K, split, res, out):
    g = inputs.generator(M * 7 + N)
    x = inputs.activations(M, K, g)
    W = inputs.weight((N, K), g)
    r = inputs.activations(M, N, g) if res else None
    y = torch.empty(M, N, device=dev, dtype=torch.bfloat16 if out == hla.HLA_BF16 else torch.float32)
    nb = hla.skinny_proj_splitk_workspace_size(M, N, K, split)
    ws = _ws(nb, dev)
    hla.skinny_proj_splitk(M, N, K, x.to(dev), W.to(dev), r.to(dev) if res else None, y, out, split,
                           ws, ws.numel())
    torch.cuda.synchronize()
    ref = oracle.moe.linear(f64(x), f64(W)) + (f64(r) if res else 0.0)
    tol = PROJ_FROB_REL_BF16 if out == hla.HLA_BF16 else PROJ_FROB_REL_F32
    assert frob_rel(f64(y), ref) < tol


@pytest.mark.parametrize("M,N,K,split,res,out", [
    (1, 1024, 544, 1, False, hla.HLA_F32), (1, 16416, 7168, 0, False, hla.HLA_F32),
    (5, 256, 7168, 7, True, hla.HLA_BF16), (8, 2048, 1024, 3, True, hla.HLA_F32),
    (12, 512, 2048, 5, False, hla.HLA_BF16), (31, 7168, 4096, 0, True, hla.HLA_BF16)])
def test_dense_cross_item_bitwise(dev, M, N, K, split, res, out, monkeypatch):
    """The persistent streaming kernel whose load ring runs across items gives the same bits as
    one item per warp, and matches the oracle.  K slices of 17, 11/10 and 13/12 steps move the
    ring's phase at item boundaries; 8- and 16-token tiles, split and direct epilogues."""
    g = inputs.generator(700 + M + N)
    x = inputs.activations(M, K, g).to(dev)
    W = inputs.weight((N, K), g).to(dev)
    r = inputs.activations(M, N, g).to(dev) if res else None
    dt = torch.bfloat16 if out == hla.HLA_BF16 else torch.float32
    nb = hla.skinny_proj_splitk_workspace_size(M, N, K, split)
    ws = _ws(nb, dev)
    ys, variants = {}, {}
    for xi in ("1", "0"):
        monkeypatch.setenv("HLA_DENSE_XITEM", xi)
        ys[xi] = torch.empty(M, N, device=dev, dtype=dt)
        hla.skinny_proj_splitk(M, N, K, x, W, r, ys[xi], out, split, ws, ws.numel())
        variants[xi] = hla.hla_last_variant()
    torch.cuda.synchronize()
    assert ",xi," in variants["1"] and ",xi," not in variants["0"], variants
    assert torch.equal(ys["1"], ys["0"])
    ref = oracle.moe.linear(f64(x), f64(W)) + (f64(r) if res else 0.0)
    tol = PROJ_FROB_REL_BF16 if out == hla.HLA_BF16 else PROJ_FROB_REL_F32
    assert frob_rel(f64(ys["1"]), ref) < tol


@pytest.mark.parametrize("M", [1, 8, 64])
def test_proj_residual_rmsnorm(dev, M):
    """o-projection + residual + RMSNorm in one epilogue: bit-identical to skinny_proj_splitk
    followed by hla_rmsnorm (same split), and within tolerance of the oracle."""
    N, K = 7168, 4096
    g = inputs.generator(90 + M)
    x, W = inputs.activations(M, K, g).to(dev), inputs.weight((N, K), g).to(dev)
    res, gam = inputs.activations(M, N, g).to(dev), inputs.gains(N, g).to(dev)
    r1 = torch.empty(M, N, dtype=torch.bfloat16, device=dev)
    xn1 = torch.empty_like(r1)
    nb = hla.skinny_proj_residual_rmsnorm_workspace_size(M, N, K, 0)
    ws = _ws(nb, dev)
    hla.skinny_proj_residual_rmsnorm(M, N, K, x, W, res, gam, 1e-6, r1, xn1, 0, ws, nb)
    split = int(hla.hla_last_variant().split("split")[1].rstrip(">"))
    r2 = torch.empty_like(r1)
    xn2 = torch.empty_like(r1)
    ws2 = _ws(hla.skinny_proj_splitk_workspace_size(M, N, K, split), dev)
    hla.skinny_proj_splitk(M, N, K, x, W, res, r2, hla.HLA_BF16, split, ws2, ws2.numel())
    hla.hla_rmsnorm(M, N, r2, gam, 1e-6, xn2)
    torch.cuda.synchronize()
    assert torch.equal(r1, r2) and torch.equal(xn1, xn2)
    r_ref = oracle.moe.linear(f64(x), f64(W)) + f64(res)
    assert frob_rel(f64(r1), r_ref) < PROJ_FROB_REL_BF16
    xn_ref = oracle.moe.rmsnorm(oracle.numerics.round_bf16(r_ref), f64(gam), 1e-6)
    assert frob_rel(f64(xn1), xn_ref) < PROJ_FROB_REL_BF16


@pytest.mark.parametrize("M,N,K", [(2, 1032, 512), (3, 9216, 256), (1, 8, 64)])
def test_proj_residual_rmsnorm_shapes(dev, M, N, K):
    """The fused epilogue at widths that leave cluster CTAs partly or wholly empty and at a width
    past 128 groups of 8 per CTA: bit-identical to the projection followed by hla_rmsnorm."""
    g = inputs.generator(95 + N)
    x, W = inputs.activations(M, K, g).to(dev), inputs.weight((N, K), g).to(dev)
    res, gam = inputs.activations(M, N, g).to(dev), inputs.gains(N, g).to(dev)
    r1 = torch.empty(M, N, dtype=torch.bfloat16, device=dev)
    xn1 = torch.empty_like(r1)
    nb = hla.skinny_proj_residual_rmsnorm_workspace_size(M, N, K, 0)
    ws = _ws(nb, dev)
    hla.skinny_proj_residual_rmsnorm(M, N, K, x, W, res, gam, 1e-6, r1, xn1, 0, ws, nb)
    split = int(hla.hla_last_variant().split("split")[1].rstrip(">"))
    r2, xn2 = torch.empty_like(r1), torch.empty_like(r1)
    ws2 = _ws(hla.skinny_proj_splitk_workspace_size(M, N, K, split), dev)
    hla.skinny_proj_splitk(M, N, K, x, W, res, r2, hla.HLA_BF16, split, ws2, ws2.numel())
    hla.hla_rmsnorm(M, N, r2, gam, 1e-6, xn2)
    torch.cuda.synchronize()
    assert torch.equal(r1, r2) and torch.equal(xn1, xn2)
    r_ref = oracle.moe.linear(f64(x), f64(W)) + f64(res)
    xn_ref = oracle.moe.rmsnorm(oracle.numerics.round_bf16(r_ref), f64(gam), 1e-6)
    assert frob_rel(f64(xn1), xn_ref) < PROJ_FROB_REL_BF16


def test_split_counts_agree(dev):
    M, N, K = 4, 512, 2048
    g = inputs.generator(3)
    x, W = inputs.activations(M, K, g).to(dev), inputs.weight((N, K), g).to(dev)
    outs = []
    for split in (1, 2, 5, 16):
        y = torch.empty(M, N, device=dev)
        ws = _ws(hla.skinny_proj_splitk_workspace_size(M, N, K, split), dev)
        hla.skinny_proj_splitk(M, N, K, x, W, None, y, hla.HLA_F32, split, ws, ws.numel())
        outs.append(y)
    torch.cuda.synchronize()
    for y in outs[1:]:
        assert frob_rel(f64(y), f64(outs[0])) < 1e-5


@pytest.mark.parametrize("M,N,K", [(32, 1000, 4000), (33, 16416, 512), (64, 7168, 4096),
                                   (100, 300, 2048), (128, 128, 64), (200, 1030, 1024),
                                   (256, 256, 7168)])
def test_tensor_core_projection(dev, M, N, K, monkeypatch):
    """tcgen05 + TMA path (32..256 tokens): ragged rows, K not a multiple of the 64-wide TMA
    box (zero-filled tail), every tile width; against the oracle and the mma.sync path."""
    g = inputs.generator(M * 3 + N + K)
    x = inputs.activations(M, K, g).to(dev)
    W = inputs.weight((N, K), g).to(dev)
    y = torch.empty(M, N, device=dev)
    ws = _ws(hla.skinny_proj_splitk_workspace_size(M, N, K, 0), dev)
    assert hla.hla_device_status() == 0
    hla.skinny_proj_splitk(M, N, K, x, W, None, y, hla.HLA_F32, 0, ws, ws.numel())
    variant = hla.hla_last_variant()
    torch.cuda.synchronize()
    assert hla.hla_device_status() == 0
    tt = int(variant.split("tt")[1].split(",")[0])
    assert tt >= 32 and tt >= M, variant
    ref = oracle.moe.linear(f64(x), f64(W))
    assert frob_rel(f64(y), ref) < PROJ_FROB_REL_F32
    monkeypatch.setenv("HLA_DENSE_TC", "0")
    y2 = torch.empty(M, N, device=dev)
    ws2 = _ws(hla.skinny_proj_splitk_workspace_size(M, N, K, 0), dev)
    hla.skinny_proj_splitk(M, N, K, x, W, None, y2, hla.HLA_F32, 0, ws2, ws2.numel())
    assert "tt16" in hla.hla_last_variant()
    torch.cuda.synchronize()
    assert frob_rel(f64(y), f64(y2)) < 1e-5


def test_tensor_core_split_counts_agree(dev):
    M, N, K = 64, 640, 2048
    g = inputs.generator(4)
    x, W = inputs.activations(M, K, g).to(dev), inputs.weight((N, K), g).to(dev)
    r = inputs.activations(M, N, g).to(dev)
    outs = []
    for split in (1, 2, 3, 8, 32):
        y = torch.empty(M, N, device=dev, dtype=torch.bfloat16)
        ws = _ws(hla.skinny_proj_splitk_workspace_size(M, N, K, split), dev)
        hla.skinny_proj_splitk(M, N, K, x, W, r, y, hla.HLA_BF16, split, ws, ws.numel())
        outs.append(y)
    torch.cuda.synchronize()
    ref = oracle.moe.linear(f64(x), f64(W)) + f64(r)
    for y in outs:
        assert frob_rel(f64(y), ref) < PROJ_FROB_REL_BF16
    assert hla.hla_device_status() == 0


@pytest.mark.parametrize("M,Hd,H,d", [(1, 256, 4, 64), (5, 512, 2, 128), (64, 1024, 4, 128)])
def test_qkvg_projection(dev, M, Hd, H, d):
    g = inputs.generator(M + Hd)
    x = inputs.activations(M, Hd, g)
    W = inputs.weight((4 * H * d + H, Hd), g, std=0.05)
    outs = dict(q=torch.empty(M, H, d, dtype=torch.bfloat16, device=dev),
                k=torch.empty(M, H, d, dtype=torch.bfloat16, device=dev),
                v=torch.empty(M, H, d, dtype=torch.bfloat16, device=dev),
                alpha=torch.empty(M, H, d, device=dev), beta=torch.empty(M, H, device=dev))
    ws = _ws(hla.kda_qkvg_proj_workspace_size(M, Hd, H, d, d, 0), dev)
    hla.kda_qkvg_proj(M, Hd, H, d, d, x.to(dev), W.to(dev), outs["q"], outs["k"], outs["v"],
                      outs["alpha"], outs["beta"], 0, ws, ws.numel())
    torch.cuda.synchronize()
    q, k, v, al, be = oracle.layer.qkvg_epilogue(oracle.moe.linear(f64(x), f64(W)), H, d, d)
    # bf16 outputs: both sides round to bf16, so they may differ by one bf16 ulp (2^-8 rel)
    for name, ref in (("q", q), ("k", k), ("v", v)):
        assert max_rel(f64(outs[name]), ref) < 1e-2, name
        assert frob_rel(f64(outs[name]), ref) < 4e-3, name
    assert max_rel(f64(outs["alpha"]), al) < 1e-4
    assert max_rel(f64(outs["beta"]), be) < 1e-4


@pytest.mark.parametrize("M,Hd", [(1, 7168), (64, 7168), (3, 256), (2, 8), (5, 40), (1, 8200),
                                  (2, 16384)])
def test_rmsnorm(dev, M, Hd):
    """One thread-block cluster per row: rows narrower than the cluster (CTAs with no columns),
    and rows wider than 128 groups of 8 per CTA (the looped path)."""
    g = inputs.generator(M + 5)
    x, gam = inputs.activations(M, Hd, g), inputs.gains(Hd, g)
    y = torch.empty(M, Hd, dtype=torch.bfloat16, device=dev)
    hla.hla_rmsnorm(M, Hd, x.to(dev), gam.to(dev), 1e-6, y)
    torch.cuda.synchronize()
    ref = oracle.moe.rmsnorm(f64(x), f64(gam), 1e-6)
    assert max_rel(f64(y), ref) < 1e-2 and frob_rel(f64(y), ref) < 4e-3


# ----------------------------------------------------------------------------- tiny MoE

@pytest.mark.parametrize("n_shared", [0, 1])
def test_tiny_moe(dev, n_shared):
    """16 experts, top-2, hidden 256, intermediate 128, one token, seed 0."""
    M, Hd, I, E, k = 1, 256, 128, 16, 2
    g = inputs.generator(0)
    w = inputs.moe_weights(E, Hd, I, n_shared, g)
    x, redraws = tie_free_activations(M, Hd, f64(w["W_r"]), k, 0)
    wd = {kk: (vv.to(dev) if vv is not None else None) for kk, vv in w.items()}
    idx = torch.empty(M, k, dtype=torch.int32, device=dev)
    wt = torch.empty(M, k, device=dev)
    logits = torch.empty(M, E, device=dev)
    ws = _ws(hla.moe_route_topk_workspace_size(M, Hd, E), dev)
    hla.moe_route_topk(M, Hd, E, k, x.to(dev), wd["W_r"], idx, wt, logits, ws, ws.numel())
    y = torch.empty(M, Hd, dtype=torch.bfloat16, device=dev)
    nb = hla.moe_expert_forward_workspace_size(M, Hd, I, E, k, n_shared)
    ws2 = _ws(nb, dev)
    hla.moe_expert_forward(M, Hd, I, E, k, n_shared, x.to(dev), idx, wt, wd["W_gate"], wd["W_up"],
                           wd["W_down"], wd["Ws_gate"], wd["Ws_up"], wd["Ws_down"], None, y, ws2, nb)
    torch.cuda.synchronize()
    idx_ref, w_ref, lg_ref = oracle.moe.route_topk(f64(x), f64(w["W_r"]), k)
    assert np.array_equal(idx.cpu().numpy(), idx_ref)
    assert max_rel(f64(wt), w_ref) < ROUTER_W_REL
    assert frob_rel(f64(logits), lg_ref) < 1e-5
    shared = [(f64(w["Ws_gate"][0]), f64(w["Ws_up"][0]), f64(w["Ws_down"][0]))] if n_shared else []
    y_ref = oracle.moe.moe_forward(f64(x), idx_ref, w_ref,
                                   (f64(w["W_gate"]), f64(w["W_up"]), f64(w["W_down"])), shared)
    assert frob_rel(f64(y), y_ref) < MOE_FROB_REL


@pytest.mark.parametrize("M,ks", [(20, "0"), (20, "3"), (40, "0")])
def test_shared_experts_on_tensor_core_path(dev, M, ks, monkeypatch):
    """With HLA_SHARED_TC=1, past 16 tokens the shared experts run as dense SwiGLU products on
    tcgen05 (not as grouped work units); with a forced K split of the routed gate/up the two
    paths coexist."""
    monkeypatch.setenv("HLA_SHARED_TC", "1")
    if ks != "0":
        monkeypatch.setenv("HLA_MOE_SPLIT", ks)
    Hd, I, E, k, ns = 256, 128, 16, 2, 2
    g = inputs.generator(70 + M)
    w = inputs.moe_weights(E, Hd, I, ns, g)
    x, _ = tie_free_activations(M, Hd, f64(w["W_r"]), k, 70 + M)
    wd = {kk: vv.to(dev) for kk, vv in w.items()}
    idx_ref, w_ref, _ = oracle.moe.route_topk(f64(x), f64(w["W_r"]), k)
    idx = torch.from_numpy(idx_ref.astype("int32")).to(dev)
    wt = torch.from_numpy(w_ref.astype("float32")).to(dev)
    res = inputs.activations(M, Hd, g).to(dev)
    y = torch.empty(M, Hd, dtype=torch.bfloat16, device=dev)
    nb = hla.moe_expert_forward_workspace_size(M, Hd, I, E, k, ns)
    ws = _ws(nb, dev)
    hla.moe_expert_forward(M, Hd, I, E, k, ns, x.to(dev), idx, wt, wd["W_gate"], wd["W_up"],
                           wd["W_down"], wd["Ws_gate"], wd["Ws_up"], wd["Ws_down"], res, y, ws, nb)
    variant = hla.hla_last_variant()
    torch.cuda.synchronize()
    assert "shared_tc" in variant and (ks == "0" or f"ks{ks}" in variant), variant
    assert hla.hla_device_status() == 0
    shared = [(f64(w["Ws_gate"][s]), f64(w["Ws_up"][s]), f64(w["Ws_down"][s])) for s in range(ns)]
    y_ref = oracle.moe.moe_forward(f64(x), idx_ref, w_ref,
                                   (f64(w["W_gate"]), f64(w["W_up"]), f64(w["W_down"])), shared,
                                   residual=f64(res))
    assert frob_rel(f64(y), y_ref) < MOE_FROB_REL


@pytest.mark.parametrize("M", [1, 5, 40])
def test_shared_experts_on_side_stream(dev, M, monkeypatch):
    """With HLA_SHARED_STREAM=1 and a side stream, the shared experts run there as dense
    SwiGLU products (split K, their own partial buffers) while the routed experts run on the
    main stream; the combine waits for both."""
    monkeypatch.setenv("HLA_SHARED_STREAM", "1")
    Hd, I, E, k, ns = 256, 128, 16, 2, 2
    g = inputs.generator(170 + M)
    w = inputs.moe_weights(E, Hd, I, ns, g)
    x, _ = tie_free_activations(M, Hd, f64(w["W_r"]), k, 170 + M)
    wd = {kk: vv.to(dev) for kk, vv in w.items()}
    idx_ref, w_ref, _ = oracle.moe.route_topk(f64(x), f64(w["W_r"]), k)
    idx = torch.from_numpy(idx_ref.astype("int32")).to(dev)
    wt = torch.from_numpy(w_ref.astype("float32")).to(dev)
    res = inputs.activations(M, Hd, g).to(dev)
    y = torch.empty(M, Hd, dtype=torch.bfloat16, device=dev)
    nb = hla.moe_expert_forward_workspace_size(M, Hd, I, E, k, ns)
    ws = _ws(nb, dev)
    side = torch.cuda.Stream()
    hla.moe_expert_forward(M, Hd, I, E, k, ns, x.to(dev), idx, wt, wd["W_gate"], wd["W_up"],
                           wd["W_down"], wd["Ws_gate"], wd["Ws_up"], wd["Ws_down"], res, y, ws, nb,
                           prefetch_stream=side)
    variant = hla.hla_last_variant()
    torch.cuda.synchronize()
    assert "shared_side" in variant, variant
    shared = [(f64(w["Ws_gate"][s]), f64(w["Ws_up"][s]), f64(w["Ws_down"][s])) for s in range(ns)]
    y_ref = oracle.moe.moe_forward(f64(x), idx_ref, w_ref,
                                   (f64(w["W_gate"]), f64(w["W_up"]), f64(w["W_down"])), shared,
                                   residual=f64(res))
    assert frob_rel(f64(y), y_ref) < MOE_FROB_REL


# ----------------------------------------------------------------------------- full-size MoE

def _run_moe(dev, w, x, idx, wt, residual=None, prefetch=False):
    M = x.shape[0]
    Hd, I, E, k, ns = FULL["Hd"], FULL["I"], FULL["E"], FULL["k"], FULL["n_shared"]
    y = torch.empty(M, Hd, dtype=torch.bfloat16, device=dev)
    nb = hla.moe_expert_forward_workspace_size(M, Hd, I, E, k, ns)
    ws = _ws(nb, dev)
    side = torch.cuda.Stream() if prefetch else 0
    hla.moe_expert_forward(M, Hd, I, E, k, ns, x, idx, wt, w["W_gate"], w["W_up"], w["W_down"],
                           w["Ws_gate"], w["Ws_up"], w["Ws_down"], residual, y, ws, nb,
                           prefetch_stream=side)
    return y


@pytest.mark.parametrize("M", [1, 2, 8, 32, 64])
def test_full_moe(dev, full_moe, M):
    Hd, E, k = FULL["Hd"], FULL["E"], FULL["k"]
    x, _ = tie_free_activations(M, Hd, full_moe["W_r64"], k, 3 + M)
    xd = x.to(dev)
    idx = torch.empty(M, k, dtype=torch.int32, device=dev)
    wt = torch.empty(M, k, device=dev)
    logits = torch.empty(M, E, device=dev)
    ws = _ws(hla.moe_route_topk_workspace_size(M, Hd, E), dev)
    hla.moe_route_topk(M, Hd, E, k, xd, full_moe["W_r"], idx, wt, logits, ws, ws.numel())
    res = inputs.activations(M, Hd, inputs.generator(55 + M)).to(dev)
    y = _run_moe(dev, full_moe, xd, idx, wt, residual=res)
    torch.cuda.synchronize()
    idx_ref, w_ref, lg_ref = oracle.moe.route_topk(f64(x), full_moe["W_r64"], k)
    assert np.array_equal(idx.cpu().numpy(), idx_ref)       # every token, bit-exact
    assert max_rel(f64(wt), w_ref) < ROUTER_W_REL
    assert frob_rel(f64(logits), lg_ref) < 1e-5
    cache = ExpertCache(full_moe)
    y_ref = oracle.moe.moe_forward(f64(x), idx_ref, w_ref, cache, cache.shared(), residual=f64(res))
    assert frob_rel(f64(y), y_ref) < MOE_FROB_REL        # every token of the batch
    for m in range(M):
        assert frob_rel(f64(y)[m], y_ref[m]) < MOE_FROB_REL, m


def test_skewed_routing_and_prefetch_bitwise(dev, full_moe):
    """All 64 tokens on the same 8 experts (64 tokens per expert: several token groups per
    weight row block); prefetch on and off must give bit-identical results."""
    M, Hd, k = 64, FULL["Hd"], FULL["k"]
    g = inputs.generator(99)
    x = inputs.activations(M, Hd, g)
    experts = torch.tensor([5, 17, 42, 99, 128, 200, 230, 255], dtype=torch.int32)
    idx = experts.repeat(M, 1)
    raw = torch.rand(M, k, generator=g) + 0.1
    wt = raw / raw.sum(1, keepdim=True)
    xd = x.to(dev)
    y1 = _run_moe(dev, full_moe, xd, idx.to(dev), wt.to(dev))
    y2 = _run_moe(dev, full_moe, xd, idx.to(dev), wt.to(dev), prefetch=True)
    y3 = _run_moe(dev, full_moe, xd, idx.to(dev), wt.to(dev))
    torch.cuda.synchronize()
    assert torch.equal(y1, y2) and torch.equal(y1, y3)
    cache = ExpertCache(full_moe)
    y_ref = oracle.moe.moe_forward(f64(x), idx.numpy(), f64(wt), cache, cache.shared())
    assert frob_rel(f64(y1), y_ref) < MOE_FROB_REL
    for m in range(M):
        assert frob_rel(f64(y1)[m], y_ref[m]) < MOE_FROB_REL, m


@pytest.mark.parametrize("M", [1, 8, 64])
def test_full_moe_shared_on_side_stream(dev, full_moe, M, monkeypatch):
    """Full-size MoE with the shared expert on the side stream: close to the default placement
    (grouped work unit; the two differ only in the order of the shared expert's fp32 sums) and
    within tolerance of the oracle on every token."""
    Hd, E, k = FULL["Hd"], FULL["E"], FULL["k"]
    x, _ = tie_free_activations(M, Hd, full_moe["W_r64"], k, 300 + M)
    xd = x.to(dev)
    idx_ref, w_ref, _ = oracle.moe.route_topk(f64(x), full_moe["W_r64"], k)
    idx = torch.from_numpy(idx_ref.astype("int32")).to(dev)
    wt = torch.from_numpy(w_ref.astype("float32")).to(dev)
    res = inputs.activations(M, Hd, inputs.generator(301 + M)).to(dev)
    y0 = _run_moe(dev, full_moe, xd, idx, wt, residual=res, prefetch=True)
    monkeypatch.setenv("HLA_SHARED_STREAM", "1")
    y1 = _run_moe(dev, full_moe, xd, idx, wt, residual=res, prefetch=True)
    assert "shared_side" in hla.hla_last_variant()
    y2 = _run_moe(dev, full_moe, xd, idx, wt, residual=res, prefetch=True)
    torch.cuda.synchronize()
    assert torch.equal(y1, y2)                      # deterministic across calls
    assert frob_rel(f64(y1), f64(y0)) < 2e-3
    cache = ExpertCache(full_moe)
    y_ref = oracle.moe.moe_forward(f64(x), idx_ref, w_ref, cache, cache.shared(), residual=f64(res))
    assert frob_rel(f64(y1), y_ref) < MOE_FROB_REL
    for m in range(M):
        assert frob_rel(f64(y1)[m], y_ref[m]) < MOE_FROB_REL, m



# ----------------------------------------------------------------------------- cross-item pipeline

def _skewed_routing(M, E, k, seed):
    """Distinct top-k experts per token drawn with weights 1/(e+1), so the first experts collect
    many tokens (several token groups) and the last few, one or none; normalised positive weights."""
    rng = np.random.default_rng(seed)
    p = 1.0 / np.arange(1, E + 1)
    p /= p.sum()
    idx = np.stack([rng.choice(E, size=k, replace=False, p=p) for _ in range(M)]).astype(np.int32)
    raw = rng.random((M, k)) + 0.1
    return idx, raw / raw.sum(1, keepdims=True)


@pytest.mark.parametrize("M,ks,ksd", [(3, "1", "1"), (3, "2", "2"), (12, "1", "1"), (12, "3", "2"),
                                      (40, "1", "1"), (40, "2", "2"), (64, "3", "1")])
def test_cross_item_pipeline_bitwise(dev, M, ks, ksd, monkeypatch):
    """The expert kernels whose load ring runs across work-item boundaries give the same bits
    as the kernels whose loads stop at each item (same products, same summation order), and
    match the oracle.  Hidden 544 (17 K steps) and intermediate 320 (10 K steps) with forced
    K splits make item lengths that are not multiples of the ring depth, so the ring's phase
    moves at every boundary; 8- and 16-token tiles, the 2-step gate/up ring from 32 tokens."""
    Hd, I, E, k, ns = 544, 320, 16, 4, 1
    monkeypatch.setenv("HLA_MOE_SPLIT", ks)
    monkeypatch.setenv("HLA_MOE_DOWN_SPLIT", ksd)
    g = inputs.generator(600 + M)
    w = inputs.moe_weights(E, Hd, I, ns, g)
    x = inputs.activations(M, Hd, g)
    res = inputs.activations(M, Hd, g)
    idx_np, wt_np = _skewed_routing(M, E, k, 600 + M)
    wd = {kk: vv.to(dev) for kk, vv in w.items()}
    xd, rd = x.to(dev), res.to(dev)
    idx = torch.from_numpy(idx_np).to(dev)
    wt = torch.from_numpy(wt_np.astype(np.float32)).to(dev)
    nb = hla.moe_expert_forward_workspace_size(M, Hd, I, E, k, ns)
    ws = _ws(nb, dev)
    out = {}
    for xi in ("1", "0"):
        monkeypatch.setenv("HLA_MOE_XITEM", xi)
        y = torch.empty(M, Hd, dtype=torch.bfloat16, device=dev)
        hla.moe_expert_forward(M, Hd, I, E, k, ns, xd, idx, wt, wd["W_gate"], wd["W_up"],
                               wd["W_down"], wd["Ws_gate"], wd["Ws_up"], wd["Ws_down"], rd, y, ws, nb)
        out[xi] = (y, hla.hla_last_variant())
    torch.cuda.synchronize()
    assert hla.hla_device_status() == 0
    v1, v0 = out["1"][1], out["0"][1]
    assert ",xgu" in v1 and ",xdn" in v1 and f"ks{ks}," in v1 and f"ksd{ksd}" in v1, v1
    assert ",xgu" not in v0 and ",xdn" not in v0, v0
    assert torch.equal(out["1"][0], out["0"][0])
    shared = [(f64(w["Ws_gate"][0]), f64(w["Ws_up"][0]), f64(w["Ws_down"][0]))]
    y_ref = oracle.moe.moe_forward(f64(x), idx_np, wt_np.astype(np.float64),
                                   (f64(w["W_gate"]), f64(w["W_up"]), f64(w["W_down"])), shared,
                                   residual=f64(res))
    assert frob_rel(f64(out["1"][0]), y_ref) < MOE_FROB_REL
