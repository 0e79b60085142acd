"""Plant plausible mistakes in copies of the oracle (CPU only) and check the pins catch each.

A pin suite that a dropped term, a flipped sign, a transposed operand or a
wrong axis could slip past would not be evidence that the oracle is right.
"""

import numpy as np
import pytest

from oracle import kda, moe, layer, numerics
from oracle.numerics import f64, sigmoid, silu
from tests.oracle_pins import (kda_pin_failures, spec_pin_failures, moe_pin_failures,
                               layer_pin_failures, fused_pin_failures,
                               extend_pin_failures)


def _caught(fn, *args):
    try:
        return len(fn(*args)) > 0
    except Exception:  # a mutant that crashes on a pin is caught too
        return True


def _step_variant(kind):
    def step(S, q, k, v, alpha, beta):
        S, q, k, v, alpha, beta = (f64(a) for a in (S, q, k, v, alpha, beta))
        b = beta[..., None, None]
        if kind == "alpha_on_columns":
            decayed = alpha[..., None, :] * S
        elif kind == "q_scaled":
            decayed = alpha[..., :, None] * S
            q = q / np.sqrt(q.shape[-1])
        else:
            decayed = alpha[..., :, None] * S
        src = S if kind == "erase_undecayed" else decayed
        kT = np.einsum("...i,...ij->...j", k, src)
        erase = b * k[..., :, None] * kT[..., None, :]
        write = b * k[..., :, None] * v[..., None, :]
        if kind == "no_beta_erase":
            erase = k[..., :, None] * kT[..., None, :]
        if kind == "erase_sign":
            erase = -erase
        if kind == "no_write":
            write = 0.0 * write
        if kind == "write_v_k_swapped":
            write = b * np.swapaxes(v[..., :, None] * k[..., None, :], -1, -2) if v.shape[-1] == k.shape[-1] else write * 2
        S_t = decayed - erase + write
        if kind == "output_old_state":
            o = np.einsum("...ij,...i->...j", S, q)
        elif kind == "output_transposed":
            o = np.einsum("...ij,...j->...i", S_t, q)
        else:
            o = np.einsum("...ij,...i->...j", S_t, q)
        return S_t, o
    return step


@pytest.mark.parametrize("kind", ["alpha_on_columns", "q_scaled", "erase_undecayed", "no_beta_erase",
                                  "erase_sign", "no_write", "output_old_state", "output_transposed"])
def test_kda_mutants_are_caught(kind):
    assert _caught(kda_pin_failures, _step_variant(kind))


def test_unmutated_variant_passes():
    assert kda_pin_failures(_step_variant("none")) == []


def _verify_in_place(S_c, q, k, v, alpha, beta):
    S = S_c  # forgets to copy: the committed state gets overwritten
    outs = []
    for t in range(q.shape[1]):
        S_new, o = kda.kda_step(S, q[:, t], k[:, t], v[:, t], alpha[:, t], beta[:, t])
        S[...] = S_new
        outs.append(o)
    return np.stack(outs, axis=1)


def _replay_off_by_one(S_c, q, k, v, alpha, beta, acc):
    return kda.spec_replay(S_c, q, k, v, alpha, beta, np.minimum(np.asarray(acc) + 1, q.shape[1]))


def _accept_counts_all_matches(d, t, c):
    a = np.sum(np.asarray(d) == np.asarray(t), axis=1)
    return a, np.asarray(c) + a


def _accept_forgets_commit(d, t, c):
    a, _ = kda.accept_prefix(d, t, c)
    return a, np.asarray(c)


@pytest.mark.parametrize("which", ["verify_in_place", "replay_off_by_one", "accept_all_matches",
                                   "accept_no_commit"])
def test_spec_mutants_are_caught(which):
    verify, accept, replay = kda.spec_verify, kda.accept_prefix, kda.spec_replay
    if which == "verify_in_place":
        verify = _verify_in_place
    elif which == "replay_off_by_one":
        replay = _replay_off_by_one
    elif which == "accept_all_matches":
        accept = _accept_counts_all_matches
    else:
        accept = _accept_forgets_commit
    assert _caught(spec_pin_failures, kda.kda_step, verify, accept, replay)


def _route_variant(kind):
    def route(x, W_r, k):
        logits = moe.linear(x, W_r)
        s = sigmoid(logits)
        M, E = s.shape
        idx = np.zeros((M, k), dtype=np.int64)
        w = np.zeros((M, k))
        for m in range(M):
            if kind == "ascending":
                order = sorted(range(E), key=lambda e: (s[m, e], e))
            elif kind == "tie_high_index":
                order = sorted(range(E), key=lambda e: (-s[m, e], -e))
            else:
                order = sorted(range(E), key=lambda e: (-s[m, e], e))
            ch = order[:k]
            idx[m] = ch
            if kind == "softmax_weights":
                ex = np.exp(logits[m, ch])
                w[m] = ex / ex.sum()
            elif kind == "no_renorm":
                w[m] = s[m, ch]
            else:
                w[m] = s[m, ch] / s[m, ch].sum()
        return idx, w, logits
    return route


def _expert_variant(kind):
    def expert(x, Wg, Wu, Wd):
        g, u = f64(Wg) @ f64(x), f64(Wu) @ f64(x)
        if kind == "silu_on_up":
            h = g * silu(u)
        elif kind == "sigmoid_not_silu":
            h = sigmoid(g) * u
        else:
            h = silu(g) * u
        return f64(Wd) @ h
    return expert


def _moe_with_expert(expert_fn, drop_shared=False, drop_residual=False, unweighted=False):
    def fwd(x, idx, w, experts, shared=(), residual=None):
        if not callable(experts):
            Wg, Wu, Wd = experts
            get = lambda e: (Wg[e], Wu[e], Wd[e])  # noqa: E731
        else:
            get = experts
        ys = []
        for m in range(x.shape[0]):
            acc = np.zeros(np.asarray(x).shape[1])
            for j in range(idx.shape[1]):
                wt = 1.0 if unweighted else float(w[m, j])
                acc = acc + wt * expert_fn(x[m], *get(int(idx[m, j])))
            if not drop_shared:
                for sh in shared:
                    acc = acc + expert_fn(x[m], *sh)
            if residual is not None and not drop_residual:
                acc = acc + f64(residual[m])
            ys.append(acc)
        return np.stack(ys)
    return fwd


def _rms_variant(kind):
    def rms(x, gamma, eps=1e-6):
        x = f64(x)
        if kind == "sum_not_mean":
            return x * f64(gamma) / np.sqrt(np.sum(x * x, -1, keepdims=True) + eps)
        return x * f64(gamma) / (np.sqrt(np.mean(x * x, -1, keepdims=True)) + eps) * 1.001
    return rms


def _bf16_truncate(x):
    f = np.asarray(x, dtype=np.float64).astype(np.float32)
    b = f.view(np.uint32) & np.uint32(0xFFFF0000)
    return b.view(np.float32).astype(np.float64)


MOE_MUTANTS = {
    "router_ascending": dict(route_topk=_route_variant("ascending")),
    "router_tie_high": dict(route_topk=_route_variant("tie_high_index")),
    "router_softmax": dict(route_topk=_route_variant("softmax_weights")),
    "router_no_renorm": dict(route_topk=_route_variant("no_renorm")),
    "silu_on_up": dict(moe_forward=_moe_with_expert(_expert_variant("silu_on_up"))),
    "sigmoid_not_silu": dict(moe_forward=_moe_with_expert(_expert_variant("sigmoid_not_silu"))),
    "drop_shared": dict(moe_forward=_moe_with_expert(_expert_variant("ok"), drop_shared=True)),
    "drop_residual": dict(moe_forward=_moe_with_expert(_expert_variant("ok"), drop_residual=True)),
    "unweighted": dict(moe_forward=_moe_with_expert(_expert_variant("ok"), unweighted=True)),
    "rms_sum": dict(rmsnorm=_rms_variant("sum_not_mean")),
    "rms_eps_outside": dict(rmsnorm=_rms_variant("eps_outside")),
    "linear_no_transpose": dict(linear=lambda x, W: f64(x) @ f64(W)),
    "bf16_truncates": dict(round_bf16=_bf16_truncate),
}


@pytest.mark.parametrize("name", sorted(MOE_MUTANTS))
def test_moe_mutants_are_caught(name):
    fns = dict(route_topk=moe.route_topk, moe_forward=moe.moe_forward,
               swiglu_expert=moe.swiglu_expert, rmsnorm=moe.rmsnorm, linear=moe.linear,
               round_bf16=numerics.round_bf16, silu=numerics.silu)
    fns.update(MOE_MUTANTS[name])
    assert _caught(moe_pin_failures, fns["route_topk"], fns["moe_forward"], fns["swiglu_expert"],
                   fns["rmsnorm"], fns["linear"], fns["round_bf16"], fns["silu"])


def _epilogue_variant(kind):
    def epi(z, H, dk, dv):
        q, k, v, g, b = layer.qkvgb_split(f64(z), H, dk, dv)
        if kind == "q_not_normalised":
            qn = q
        else:
            qn = layer.l2_normalise(q)
        kn = layer.l2_normalise(k)
        alpha = np.exp(-numerics.softplus(g)) if kind != "alpha_softplus" else numerics.softplus(g)
        if kind == "alpha_sigmoid_g":
            alpha = sigmoid(g)
        beta = sigmoid(b)
        return (numerics.round_bf16(qn), numerics.round_bf16(kn), numerics.round_bf16(v),
                numerics.round_f32(alpha), numerics.round_f32(beta))
    return epi


@pytest.mark.parametrize("kind", ["q_not_normalised", "alpha_softplus", "alpha_sigmoid_g"])
def test_layer_epilogue_mutants_are_caught(kind):
    assert _caught(layer_pin_failures, _epilogue_variant(kind), layer.decode_layer, kda.kda_step,
                   moe.rmsnorm, numerics.round_bf16)


def _layer_variant(kind):
    """A copy of the oracle's decode_layer with one plausible wiring mistake in its second half."""
    rb = numerics.round_bf16

    def decode_layer(x, S, p, experts, shared=()):
        H, dk, dv, eps = p["H"], p["dk"], p["dv"], p.get("eps", 1e-6)
        x = f64(x)
        M = x.shape[0]
        x1 = rb(moe.rmsnorm(x, p["gamma_attn"], eps))
        q, k, v, alpha, beta = layer.qkvg_epilogue(moe.linear(x1, p["W_qkvgb"]), H, dk, dv)
        S_new, o = kda.kda_step(S, q, k, v, alpha, beta)
        o_b = (o if kind == "o_unrounded" else rb(o)).reshape(M, H * dv)
        proj = f64(o_b) @ f64(p["W_o"]) if kind == "W_o_transposed" else moe.linear(o_b, p["W_o"])
        r = rb(x + proj)
        x2 = rb(moe.rmsnorm(r, p["gamma_moe"], eps))
        idx, w, logits = moe.route_topk(x2, p["W_r"], p["top_k"])
        moe_in = {"moe_fed_x1": x1, "moe_fed_x": x}.get(kind, x2)
        res = x if kind == "residual_from_x" else r
        y = rb(moe.moe_forward(moe_in, idx, w, experts, shared, residual=res))
        aux = dict(x1=x1, q=q, k=k, v=v, alpha=alpha, beta=beta, o=o, r=r, x2=x2,
                   topk_idx=idx, topk_w=w, logits=logits)
        return y, S_new, aux
    return decode_layer


def test_layer_variant_without_mistake_passes():
    assert layer_pin_failures(layer.qkvg_epilogue, _layer_variant("none"), kda.kda_step,
                              moe.rmsnorm, numerics.round_bf16) == []


@pytest.mark.parametrize("kind", ["W_o_transposed", "residual_from_x", "moe_fed_x1", "moe_fed_x",
                                  "o_unrounded"])
def test_layer_wiring_mutants_are_caught(kind):
    assert _caught(layer_pin_failures, layer.qkvg_epilogue, _layer_variant(kind), kda.kda_step,
                   moe.rmsnorm, numerics.round_bf16)


def _fused_verifies_stale_state(S_c, prev, acc, new):
    S = kda.spec_replay(S_c, prev["q"], prev["k"], prev["v"], prev["alpha"], prev["beta"], acc)
    o = kda.spec_verify(S_c, new["q"], new["k"], new["v"], new["alpha"], new["beta"])
    return S, o


def _fused_replays_all(S_c, prev, acc, new):
    full = np.full_like(np.asarray(acc), prev["q"].shape[1])
    return kda.spec_replay_verify(S_c, prev, full, new)


@pytest.mark.parametrize("mutant", [_fused_verifies_stale_state, _fused_replays_all])
def test_fused_mutants_are_caught(mutant):
    assert _caught(fused_pin_failures, kda.kda_step, mutant)


def _extend_off_by_one_offsets(S, cu, q, k, v, alpha, beta):
    cu = np.asarray(cu).copy()
    cu[1:-1] += 1  # sequences take one token of their successor
    return kda.extend(S, cu, q, k, v, alpha, beta)


def _extend_reversed(S, cu, q, k, v, alpha, beta):
    S = np.asarray(S, float).copy()
    o = np.zeros((q.shape[0],) + tuple(np.shape(v)[1:]))
    for b in range(S.shape[0]):
        for n in reversed(range(int(cu[b]), int(cu[b + 1]))):
            S[b], o[n] = kda.kda_step(S[b], q[n], k[n], v[n], alpha[n], beta[n])
    return S, o


@pytest.mark.parametrize("mutant", [_extend_off_by_one_offsets, _extend_reversed])
def test_extend_mutants_are_caught(mutant):
    assert _caught(extend_pin_failures, kda.kda_step, mutant)
