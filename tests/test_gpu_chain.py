"""Launch chains (hla_chain_begin / hla_chain_end): library calls queued back to back on one
stream, every kernel after the first a programmatic dependent of the one before it, must give
the bits of plain launches."""

import pytest
import torch

from hybrid_linear_attention_gated_gb300 import hla, inputs
from tests.gpu_common import require_gpu, warm_states

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def dev():
    return require_gpu()


def _to(d, dev):
    return {k: v.to(dev) for k, v in d.items()}


def _spec_window(B, T, H, d, S, win, dr, tg, acc, com, o):
    hla.kda_spec_verify_replay(hla.HLA_SPEC_VERIFY, B, T, H, d, d, S, None, win["q"], win["k"],
                               win["v"], win["alpha"], win["beta"], None, o)
    hla.spec_accept_prefix(B, T, dr, tg, acc, com)
    hla.kda_spec_verify_replay(hla.HLA_SPEC_REPLAY, B, T, H, d, d, S, None, win["q"], win["k"],
                               win["v"], win["alpha"], win["beta"], acc, None)


@pytest.mark.parametrize("B", [16, 64])
def test_launch_chain_is_bitwise_neutral(dev, B):
    """verify -> accept -> replay queued as one launch chain (each kernel a programmatic
    dependent of the one before it) gives the bits of plain launches, eager and in a CUDA graph,
    two windows in a row."""
    T, H, d = 4, 32, 128
    S0 = warm_states(8, B, H, d).to(dev)
    g = inputs.generator(4700 + B)
    wins = [_to(inputs.kda_inputs((B, T), H, d, d, g), dev) for _ in range(2)]
    ids = [inputs.accept_ids(B, T, g) for _ in range(2)]
    ids = [(dr.to(dev), tg.to(dev)) for dr, tg, _ in ids]

    def run(chain, graph=False):
        S = S0.clone()
        acc = torch.zeros(B, dtype=torch.int32, device=dev)
        com = torch.zeros(B, dtype=torch.int32, device=dev)
        os_ = [torch.empty(B, T, H, d, device=dev) for _ in range(2)]

        def body():
            for w, (dr, tg), o in zip(wins, ids, os_):
                if chain:
                    hla.hla_chain_begin()
                try:
                    _spec_window(B, T, H, d, S, w, dr, tg, acc, com, o)
                finally:
                    if chain:
                        hla.hla_chain_end()
        if graph:
            body()  # warm-up outside the capture
            S.copy_(S0)
            com.zero_()
            torch.cuda.synchronize()
            gr = torch.cuda.CUDAGraph()
            s = torch.cuda.Stream()
            with torch.cuda.stream(s):
                with torch.cuda.graph(gr, stream=s):
                    body()
            S.copy_(S0)
            com.zero_()
            gr.replay()
        else:
            body()
        torch.cuda.synchronize()
        return S, os_, acc, com

    ref = run(False)
    for got in (run(True), run(True, graph=True)):
        assert torch.equal(got[0], ref[0]) and torch.equal(got[2], ref[2]) and torch.equal(got[3], ref[3])
        assert all(torch.equal(a, b) for a, b in zip(got[1], ref[1]))


def test_chain_of_calls_on_the_same_state(dev):
    """Chained calls where a kernel's predecessor writes the very state it reads: two decode steps
    in a row, and the replay of one window followed by the verify of the next.  A kernel must not
    read its state before its wait here; the results are the bits of plain launches."""
    B, T, H, d = 8, 4, 32, 128
    S0 = warm_states(9, B, H, d).to(dev)
    g = inputs.generator(4900)
    steps = [_to(inputs.kda_inputs((B,), H, d, d, g), dev) for _ in range(3)]
    wins = [_to(inputs.kda_inputs((B, T), H, d, d, g), dev) for _ in range(2)]
    acc = torch.tensor([0, 1, 2, 3, 4, 4, 1, 2], dtype=torch.int32, device=dev)

    def run(chain):
        S = S0.clone()
        outs = []
        if chain:
            hla.hla_chain_begin()
        try:
            for u in steps:
                o = torch.empty(B, H, d, device=dev)
                hla.kda_decode_step(B, H, d, d, S, None, u["q"], u["k"], u["v"], u["alpha"], u["beta"], o)
                outs.append(o)
            w0, w1 = wins
            hla.kda_spec_verify_replay(hla.HLA_SPEC_REPLAY, B, T, H, d, d, S, None, w0["q"], w0["k"], w0["v"],
                                       w0["alpha"], w0["beta"], acc, None)
            o = torch.empty(B, T, H, d, device=dev)
            hla.kda_spec_verify_replay(hla.HLA_SPEC_VERIFY, B, T, H, d, d, S, None, w1["q"], w1["k"], w1["v"],
                                       w1["alpha"], w1["beta"], None, o)
            outs.append(o)
        finally:
            if chain:
                hla.hla_chain_end()
        torch.cuda.synchronize()
        return S, outs

    S_ref, o_ref = run(False)
    for _ in range(3):
        S_c, o_c = run(True)
        assert torch.equal(S_c, S_ref)
        assert all(torch.equal(a, b) for a, b in zip(o_c, o_ref))


@pytest.mark.parametrize("M", [1, 8, 32])
def test_entry_points_chain_their_own_kernels_bitwise(dev, M, monkeypatch):
    """The multi-kernel entry points (projections with their epilogues or split reductions, the
    router, the expert pipeline) chain their own kernels up to 32 tokens; HLA_PDL=0 launches them
    plain.  Both give the same bits, with the expert weights' shapes of the model at a reduced
    expert count."""
    Hd, I, E, k, ns, H, d = 7168, 2048, 24, 8, 1, 32, 128
    g = inputs.generator(5100 + M, dev)
    w = inputs.moe_weights(E, Hd, I, ns, g, device=dev)
    Wq = inputs.weight((4 * H * d + H, Hd), g, dev)
    Wo = inputs.weight((Hd, H * d), g, dev)
    gamma = inputs.gains(Hd, g, dev)
    x = inputs.activations(M, Hd, g, dev)
    o_in = inputs.activations(M, H * d, g, dev)
    res = inputs.activations(M, Hd, g, dev)

    def ws(n):
        return torch.empty(max(n, 256), dtype=torch.uint8, device=dev)

    def run():
        out = {}
        q, kk_, v = (torch.empty(M, H, d, dtype=torch.bfloat16, device=dev) for _ in range(3))
        al, be = torch.empty(M, H, d, device=dev), torch.empty(M, H, device=dev)
        nb = hla.kda_qkvg_proj_workspace_size(M, Hd, H, d, d, 0)
        hla.kda_qkvg_proj(M, Hd, H, d, d, x, Wq, q, kk_, v, al, be, 0, ws(nb), nb)
        out.update(q=q, k=kk_, v=v, alpha=al, beta=be)
        y = torch.empty(M, Hd, device=dev)
        nb = hla.skinny_proj_splitk_workspace_size(M, Hd, H * d, 4)
        hla.skinny_proj_splitk(M, Hd, H * d, o_in, Wo, res, y, hla.HLA_F32, 4, ws(nb), nb)
        out["proj"] = y
        r = torch.empty(M, Hd, dtype=torch.bfloat16, device=dev)
        xn = torch.empty(M, Hd, dtype=torch.bfloat16, device=dev)
        nb = hla.skinny_proj_residual_rmsnorm_workspace_size(M, Hd, H * d, 0)
        hla.skinny_proj_residual_rmsnorm(M, Hd, H * d, o_in, Wo, res, gamma, 1e-6, r, xn, 0, ws(nb), nb)
        out.update(r=r, xn=xn)
        idx = torch.empty(M, k, dtype=torch.int32, device=dev)
        wt = torch.empty(M, k, device=dev)
        nb = hla.moe_route_topk_workspace_size(M, Hd, E)
        hla.moe_route_topk(M, Hd, E, k, xn, w["W_r"], idx, wt, None, ws(nb), nb)
        out.update(idx=idx, wt=wt)
        ym = torch.empty(M, Hd, dtype=torch.bfloat16, device=dev)
        nb = hla.moe_expert_forward_workspace_size(M, Hd, I, E, k, ns)
        hla.moe_expert_forward(M, Hd, I, E, k, ns, xn, idx, wt, w["W_gate"], w["W_up"], w["W_down"],
                               w["Ws_gate"], w["Ws_up"], w["Ws_down"], r, ym, ws(nb), nb)
        out["moe"] = ym
        torch.cuda.synchronize()
        return {kk: vv.cpu() for kk, vv in out.items()}

    monkeypatch.setenv("HLA_PDL", "0")
    plain = run()
    monkeypatch.setenv("HLA_PDL", "1")
    chained = run()
    assert hla.hla_device_status() == 0
    for key in plain:
        assert torch.equal(plain[key], chained[key]), key
