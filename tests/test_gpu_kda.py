"""KDA decode step, speculative verify / accept / replay on the GPU against the oracle."""

import os

import numpy as np
import pytest
import torch

import oracle
from hybrid_linear_attention_gated_gb300 import hla, inputs
from tests.gpu_common import KDA_MAX_REL, f64, max_rel, require_gpu, warm_states

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def dev():
    return require_gpu()


def _to(d, dev):
    return {k: v.to(dev) for k, v in d.items()}


def _decode(dev, S, inp, o_dtype=hla.HLA_F32, state_idx=None):
    B, H, d = inp["q"].shape
    o = torch.empty(B, H, d, device=dev, dtype=torch.float32 if o_dtype == hla.HLA_F32 else torch.bfloat16)
    hla.kda_decode_step(B, H, d, d, S, state_idx, inp["q"], inp["k"], inp["v"], inp["alpha"],
                        inp["beta"], o, o_dtype)
    return o


def _np(inp):
    return {k: f64(v) for k, v in inp.items()}


def test_tiny_case_steps_verify_accept_replay(dev):
    """Batch 1, 4 heads, d=64: 8 steps from S0 ~ N(0,0.02), a 4-token draft, 2 accepted."""
    g = inputs.generator(0)
    B, H, d, T = 1, 4, 64, 4
    S0 = inputs.small_state(B, H, d, d, g)
    steps = [inputs.kda_inputs((B,), H, d, d, g) for _ in range(8)]
    win = inputs.kda_inputs((B, T), H, d, d, g)
    draft, target, a_int = inputs.accept_ids(B, T, g)
    # the tiny case fixes 2 accepted tokens
    target = draft.clone()
    target[:, 2] = draft[:, 2] + 1

    S = S0.to(dev)
    S_ref = f64(S0)
    for st in steps:
        o = _decode(dev, S, _to(st, dev))
        n = _np(st)
        S_ref, o_ref = oracle.kda.kda_step(S_ref, n["q"], n["k"], n["v"], n["alpha"], n["beta"])
        assert max_rel(f64(o), o_ref) < KDA_MAX_REL
    assert max_rel(f64(S), S_ref) < KDA_MAX_REL

    wd, wn = _to(win, dev), _np(win)
    S_before = S.clone()
    ov = torch.empty(B, T, H, d, device=dev)
    hla.kda_spec_verify_replay(hla.HLA_SPEC_VERIFY, B, T, H, d, d, S, None, wd["q"], wd["k"], wd["v"],
                               wd["alpha"], wd["beta"], None, ov)
    acc = torch.zeros(B, dtype=torch.int32, device=dev)
    com = torch.full((B,), 9, dtype=torch.int32, device=dev)
    hla.spec_accept_prefix(B, T, draft.to(dev), target.to(dev), acc, com)
    hla.kda_spec_verify_replay(hla.HLA_SPEC_REPLAY, B, T, H, d, d, S, None, wd["q"], wd["k"],
                               wd["v"], wd["alpha"], wd["beta"], acc, None)
    torch.cuda.synchronize()
    ov_ref = oracle.kda.spec_verify(S_ref, wn["q"], wn["k"], wn["v"], wn["alpha"], wn["beta"])
    a_ref, com_ref = oracle.kda.accept_prefix(draft.numpy(), target.numpy(), np.array([9]))
    S_new_ref = oracle.kda.spec_replay(S_ref, wn["q"], wn["k"], wn["v"], wn["alpha"], wn["beta"], a_ref)
    assert int(a_ref[0]) == 2
    assert np.array_equal(acc.cpu().numpy(), a_ref) and np.array_equal(com.cpu().numpy(), com_ref)
    assert max_rel(f64(ov), ov_ref) < KDA_MAX_REL
    assert max_rel(f64(S), S_new_ref) < KDA_MAX_REL
    assert not torch.equal(S, S_before)


@pytest.mark.parametrize("B", [1, 2, 8, 32, 64])
def test_decode_step_sweep(dev, B):
    """Batch sweep at H=32, d=128 from warm committed states (256 prior updates)."""
    H, d = 32, 128
    S0 = warm_states(1, B, H, d)
    inp = inputs.kda_inputs((B,), H, d, d, inputs.generator(1000 + B))
    S = S0.to(dev)
    o = _decode(dev, S, _to(inp, dev))
    torch.cuda.synchronize()
    n = _np(inp)
    S_ref, o_ref = oracle.kda.kda_step(f64(S0), n["q"], n["k"], n["v"], n["alpha"], n["beta"])
    assert max_rel(f64(o), o_ref) < KDA_MAX_REL
    assert max_rel(f64(S), S_ref) < KDA_MAX_REL
    assert hla.hla_last_variant().startswith("kda_recur<dk128")


@pytest.mark.parametrize("B,cw", [(1, "0"), (8, "0"), (64, "0"), (8, "32"), (8, "64")])
def test_decode_step_d64(dev, B, cw, monkeypatch):
    """d_k = d_v = 64 (the other supported head size) against the oracle, at the default slice
    width and forced wider ones (whole heads at 64), with bits equal across widths."""
    H, d = 16, 64
    monkeypatch.setenv("HLA_KDA_CW", cw)
    S0 = warm_states(3, B, H, d)
    inp = inputs.kda_inputs((B,), H, d, d, inputs.generator(1200 + B))
    S = S0.to(dev)
    o = _decode(dev, S, _to(inp, dev))
    torch.cuda.synchronize()
    assert hla.hla_last_variant().startswith("kda_recur<dk64")
    n = _np(inp)
    S_ref, o_ref = oracle.kda.kda_step(f64(S0), n["q"], n["k"], n["v"], n["alpha"], n["beta"])
    assert max_rel(f64(o), o_ref) < KDA_MAX_REL
    assert max_rel(f64(S), S_ref) < KDA_MAX_REL
    monkeypatch.setenv("HLA_KDA_CW", "16")
    S16 = S0.to(dev)
    o16 = _decode(dev, S16, _to(inp, dev))
    torch.cuda.synchronize()
    assert torch.equal(S16, S) and torch.equal(o16, o)


def test_decode_bf16_output_and_state_idx(dev):
    B, H, d = 8, 32, 128
    S0 = warm_states(1, B, H, d)
    inp = inputs.kda_inputs((B,), H, d, d, inputs.generator(77))
    perm = torch.randperm(12, generator=inputs.generator(78))[:B].to(torch.int32)
    pool = torch.zeros(12, H, d, d)
    pool[perm.long()] = S0
    Sd = pool.to(dev)
    o = _decode(dev, Sd, _to(inp, dev), hla.HLA_BF16, perm.to(dev))
    torch.cuda.synchronize()
    n = _np(inp)
    S_ref, o_ref = oracle.kda.kda_step(f64(S0), n["q"], n["k"], n["v"], n["alpha"], n["beta"])
    # bf16 output: rounding of 2^-9 relative on top of the fp32 path
    assert max_rel(f64(o), o_ref) < 5e-3
    got = Sd.cpu()
    assert max_rel(got[perm.long()].double().numpy(), S_ref) < KDA_MAX_REL
    untouched = torch.ones(12, dtype=torch.bool)
    untouched[perm.long()] = False
    assert torch.count_nonzero(got[untouched]) == 0


def test_spec_window_config(dev):
    """B=16, T=4, H=32, d=128, accepted length uniform in {0..4}."""
    B, T, H, d = 16, 4, 32, 128
    S0 = warm_states(2, B, H, d)
    g = inputs.generator(2)
    win = inputs.kda_inputs((B, T), H, d, d, g)
    draft, target, a_int = inputs.accept_ids(B, T, g)
    S = S0.to(dev)
    wd, wn = _to(win, dev), _np(win)
    ov = torch.empty(B, T, H, d, device=dev)
    hla.kda_spec_verify_replay(hla.HLA_SPEC_VERIFY, B, T, H, d, d, S, None, wd["q"], wd["k"], wd["v"],
                               wd["alpha"], wd["beta"], None, ov)
    torch.cuda.synchronize()
    assert torch.equal(S.cpu(), S0), "verify must not write the committed state"
    acc = torch.zeros(B, dtype=torch.int32, device=dev)
    com = torch.arange(B, dtype=torch.int32, device=dev)
    hla.spec_accept_prefix(B, T, draft.to(dev), target.to(dev), acc, com)
    hla.kda_spec_verify_replay(hla.HLA_SPEC_REPLAY, B, T, H, d, d, S, None, wd["q"], wd["k"],
                               wd["v"], wd["alpha"], wd["beta"], acc, None)
    torch.cuda.synchronize()
    a_ref, com_ref = oracle.kda.accept_prefix(draft.numpy(), target.numpy(), np.arange(B))
    assert np.array_equal(a_ref, a_int.numpy())
    assert np.array_equal(acc.cpu().numpy(), a_ref)
    assert np.array_equal(com.cpu().numpy(), com_ref)
    ov_ref = oracle.kda.spec_verify(f64(S0), wn["q"], wn["k"], wn["v"], wn["alpha"], wn["beta"])
    S_ref = oracle.kda.spec_replay(f64(S0), wn["q"], wn["k"], wn["v"], wn["alpha"], wn["beta"], a_ref)
    assert max_rel(f64(ov), ov_ref) < KDA_MAX_REL
    Sg = S.cpu()
    assert max_rel(Sg.double().numpy(), S_ref) < KDA_MAX_REL
    for b in range(B):  # nothing accepted -> state bitwise untouched
        if a_ref[b] == 0:
            assert torch.equal(Sg[b], S0[b])


@pytest.mark.parametrize("B,H,T,d,o_bf16", [(5, 8, 1, 128, False), (5, 8, 3, 64, True), (5, 8, 7, 128, True),
                                            (5, 8, 8, 64, False), (64, 32, 4, 128, False)])
def test_spec_window_draft_lengths(dev, B, H, T, d, o_bf16):
    """Verify and replay at other draft lengths, head sizes and batch 64 (the sweep's larger window),
    states in a slot pool, against the oracle's sequential steps."""
    S0 = warm_states(11, B, H, d)
    g = inputs.generator(1100 + T + d)
    win = inputs.kda_inputs((B, T), H, d, d, g)
    draft, target, a = inputs.accept_ids(B, T, g)
    perm = torch.randperm(B + 2, generator=inputs.generator(1101))[:B].to(torch.int32)
    pool = torch.zeros(B + 2, H, d, d)
    pool[perm.long()] = S0
    S = pool.to(dev)
    wd, wn = _to(win, dev), _np(win)
    o = torch.empty(B, T, H, d, device=dev, dtype=torch.bfloat16 if o_bf16 else torch.float32)
    hla.kda_spec_verify_replay(hla.HLA_SPEC_VERIFY, B, T, H, d, d, S, perm.to(dev), wd["q"], wd["k"], wd["v"],
                               wd["alpha"], wd["beta"], None, o, hla.HLA_BF16 if o_bf16 else hla.HLA_F32)
    acc = torch.zeros(B, dtype=torch.int32, device=dev)
    com = torch.zeros(B, dtype=torch.int32, device=dev)
    hla.spec_accept_prefix(B, T, draft.to(dev), target.to(dev), acc, com)
    hla.kda_spec_verify_replay(hla.HLA_SPEC_REPLAY, B, T, H, d, d, S, perm.to(dev), wd["q"], wd["k"], wd["v"],
                               wd["alpha"], wd["beta"], acc, None)
    torch.cuda.synchronize()
    assert np.array_equal(acc.cpu().numpy(), a.numpy())
    o_ref = oracle.kda.spec_verify(f64(S0), wn["q"], wn["k"], wn["v"], wn["alpha"], wn["beta"])
    S_ref = oracle.kda.spec_replay(f64(S0), wn["q"], wn["k"], wn["v"], wn["alpha"], wn["beta"], a.numpy())
    # bf16 output: rounding of 2^-9 relative on top of the fp32 path
    assert max_rel(f64(o), o_ref) < (5e-3 if o_bf16 else KDA_MAX_REL)
    assert max_rel(S.cpu()[perm.long()].double().numpy(), S_ref) < KDA_MAX_REL


def test_verify_with_vanishing_decays(dev):
    """Verify where some rows' decays vanish (exact zeros, and tiny values whose products underflow)
    next to ordinary ones, against the oracle; a fused replay-and-verify of the same window (nothing
    replayed) gives the same bits as the separate call."""
    B, T, H, d = 4, 4, 8, 128
    S0 = warm_states(13, B, H, d)
    g = inputs.generator(1400)
    win = inputs.kda_inputs((B, T), H, d, d, g)
    al = win["alpha"]
    al[0, 1, 2, 5] = 0.0          # one row of one head of sequence 0 forgets everything at token 1
    al[1, :, 3, 7:9] = 1e-30      # two rows of a head of sequence 1 underflow over the window
    al[2, 0, :, 64] = 1e-12       # one row of every head of sequence 2 (products reach 1e-48)
    wd, wn = _to(win, dev), _np(win)
    S = S0.to(dev)
    o = torch.empty(B, T, H, d, device=dev)
    hla.kda_spec_verify_replay(hla.HLA_SPEC_VERIFY, B, T, H, d, d, S, None, wd["q"], wd["k"], wd["v"],
                               wd["alpha"], wd["beta"], None, o)
    torch.cuda.synchronize()
    o_ref = oracle.kda.spec_verify(f64(S0), wn["q"], wn["k"], wn["v"], wn["alpha"], wn["beta"])
    assert torch.isfinite(o).all()
    assert max_rel(f64(o), o_ref) < KDA_MAX_REL
    # fused: replay nothing of a previous window (accepted 0), then verify this one
    acc0 = torch.zeros(B, dtype=torch.int32, device=dev)
    o2 = torch.empty_like(o)
    S2 = S0.to(dev)
    hla.kda_spec_replay_verify(B, T, T, H, d, d, S2, None, wd["q"], wd["k"], wd["v"], wd["alpha"], wd["beta"],
                               acc0, wd["q"], wd["k"], wd["v"], wd["alpha"], wd["beta"], o2)
    torch.cuda.synchronize()
    assert torch.equal(o2, o) and torch.equal(S2, S)


def test_replay_all_equals_decode_steps_bitwise(dev):
    B, T, H, d = 4, 4, 32, 128
    S0 = warm_states(3, B, H, d)
    win = inputs.kda_inputs((B, T), H, d, d, inputs.generator(31))
    wd = _to(win, dev)
    S1 = S0.to(dev)
    acc = torch.full((B,), T, dtype=torch.int32, device=dev)
    hla.kda_spec_verify_replay(hla.HLA_SPEC_REPLAY, B, T, H, d, d, S1, None, wd["q"], wd["k"], wd["v"],
                               wd["alpha"], wd["beta"], acc, None)
    S2 = S0.to(dev)
    for t in range(T):
        step = {k: v[:, t].contiguous() for k, v in wd.items()}
        _decode(dev, S2, step)
    torch.cuda.synchronize()
    assert torch.equal(S1, S2)


@pytest.mark.parametrize("cw", ["16", "32", "64", "128"])
def test_slice_width_variants_bitwise_equal(dev, cw, monkeypatch):
    B, H, d = 2, 32, 128
    S0 = warm_states(1, B, H, d)
    inp = _to(inputs.kda_inputs((B,), H, d, d, inputs.generator(5)), dev)
    S_ref = S0.to(dev)
    o_ref = _decode(dev, S_ref, inp)
    monkeypatch.setenv("HLA_KDA_CW", cw)
    S = S0.to(dev)
    o = _decode(dev, S, inp)
    torch.cuda.synchronize()
    assert hla.hla_last_variant() == f"kda_recur<dk128,cw{cw},decode>"
    assert torch.equal(S, S_ref) and torch.equal(o, o_ref)


def test_run_to_run_determinism(dev):
    B, H, d = 16, 32, 128
    S0 = warm_states(2, B, H, d)
    win = _to(inputs.kda_inputs((B, 4), H, d, d, inputs.generator(9)), dev)
    outs = []
    for _ in range(2):
        S = S0.to(dev)
        ov = torch.empty(B, 4, H, d, device=dev)
        hla.kda_spec_verify_replay(hla.HLA_SPEC_VERIFY, B, 4, H, d, d, S, None, win["q"], win["k"],
                                   win["v"], win["alpha"], win["beta"], None, ov)
        outs.append(ov)
    torch.cuda.synchronize()
    assert torch.equal(outs[0], outs[1])


@pytest.mark.parametrize("B,Tp,T,d,acc_kind", [(16, 4, 4, 128, "uniform"), (4, 3, 5, 128, "zero"),
                                                (4, 8, 8, 128, "all"), (2, 4, 2, 64, "uniform"),
                                                (64, 4, 4, 128, "uniform")])
def test_fused_replay_verify(dev, B, Tp, T, d, acc_kind):
    """Replay of the previous window + verify of the next in one pass over the state:
    bit-identical to the two separate calls, and within tolerance of the oracle."""
    H = 32 if d == 128 else 4
    S0 = warm_states(6, B, H, d)
    g = inputs.generator(600 + B + Tp + T)
    prev = inputs.kda_inputs((B, Tp), H, d, d, g)
    new = inputs.kda_inputs((B, T), H, d, d, g)
    if acc_kind == "uniform":
        _, _, acc = inputs.accept_ids(B, Tp, g)
    elif acc_kind == "zero":
        acc = torch.zeros(B, dtype=torch.int64)
    else:
        acc = torch.full((B,), Tp, dtype=torch.int64)
    accd = acc.to(torch.int32).to(dev)
    pd, nd = _to(prev, dev), _to(new, dev)
    # fused
    S1 = S0.to(dev)
    o1 = torch.empty(B, T, H, d, device=dev)
    hla.kda_spec_replay_verify(B, Tp, T, H, d, d, S1, None, pd["q"], pd["k"], pd["v"], pd["alpha"],
                               pd["beta"], accd, nd["q"], nd["k"], nd["v"], nd["alpha"], nd["beta"], o1)
    assert "replay_verify" in hla.hla_last_variant()
    # separate
    S2 = S0.to(dev)
    o2 = torch.empty(B, T, H, d, device=dev)
    hla.kda_spec_verify_replay(hla.HLA_SPEC_REPLAY, B, Tp, H, d, d, S2, None, pd["q"], pd["k"], pd["v"],
                               pd["alpha"], pd["beta"], accd, None)
    hla.kda_spec_verify_replay(hla.HLA_SPEC_VERIFY, B, T, H, d, d, S2, None, nd["q"], nd["k"], nd["v"],
                               nd["alpha"], nd["beta"], None, o2)
    torch.cuda.synchronize()
    assert torch.equal(S1, S2) and torch.equal(o1, o2)
    S_ref, o_ref = oracle.kda.spec_replay_verify(f64(S0), _np(prev), acc.numpy(), _np(new))
    assert max_rel(f64(S1), S_ref) < KDA_MAX_REL
    assert max_rel(f64(o1), o_ref) < KDA_MAX_REL
    for b in range(B):
        if int(acc[b]) == 0:
            assert torch.equal(S1[b].cpu(), S0[b])


def test_extend_bf16_output_is_the_rounded_fp32_output(dev):
    """kda_extend with bf16 outputs: the same fp32 arithmetic, rounded to nearest even at the store,
    so each output equals the fp32 run's output rounded to bf16; the states are bitwise equal."""
    lens = [3, 1, 20, 0, 9]
    B, H, d = len(lens), 8, 128
    cu = torch.tensor(np.concatenate([[0], np.cumsum(lens)]).astype(np.int32), device=dev)
    N = int(sum(lens))
    S0 = warm_states(12, B, H, d)
    tok = _to(inputs.kda_inputs((N,), H, d, d, inputs.generator(1300)), dev)
    out = {}
    for dt, tdt in ((hla.HLA_F32, torch.float32), (hla.HLA_BF16, torch.bfloat16)):
        S = S0.to(dev)
        o = torch.empty(N, H, d, device=dev, dtype=tdt)
        hla.kda_extend(B, cu, H, d, d, S, None, tok["q"], tok["k"], tok["v"], tok["alpha"], tok["beta"], o, dt)
        torch.cuda.synchronize()
        out[dt] = (S, o)
    assert torch.equal(out[hla.HLA_F32][0], out[hla.HLA_BF16][0])
    assert torch.equal(out[hla.HLA_F32][1].to(torch.bfloat16), out[hla.HLA_BF16][1])


def test_extend_single_tokens_equal_decode_bitwise(dev):
    B, H, d = 8, 32, 128
    S0 = warm_states(1, B, H, d)
    inp = _to(inputs.kda_inputs((B,), H, d, d, inputs.generator(81)), dev)
    S1, S2 = S0.to(dev), S0.to(dev)
    o1 = _decode(dev, S1, inp)
    o2 = torch.empty(B, H, d, device=dev)
    cu = torch.arange(B + 1, dtype=torch.int32, device=dev)
    hla.kda_extend(B, cu, H, d, d, S2, None, inp["q"], inp["k"], inp["v"], inp["alpha"], inp["beta"], o2)
    torch.cuda.synchronize()
    assert "extend" in hla.hla_last_variant()
    assert torch.equal(S1, S2) and torch.equal(o1, o2)


@pytest.mark.parametrize("lens,d", [([0, 1, 5, 17, 3, 40, 8, 1], 128), ([2, 0, 9], 64),
                                    ([int(n) for n in np.random.default_rng(5).choice([0, 1, 1, 1, 2, 9, 20], 300)], 64)])
def test_extend_ragged_mixed_batch(dev, lens, d):
    """Ragged sequences (empty, single-token decode, multi-block prefill chunks) in one call:
    against the oracle, and bitwise against one decode call per token.  The kernel schedules the
    multi-block chains first; 300 sequences take the schedule through several rounds of its
    block-wide count (128 threads per CTA)."""
    B = len(lens)
    H = 32 if d == 128 else 4
    cu = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
    N = int(cu[-1])
    S0 = warm_states(8, B, H, d)
    tok = inputs.kda_inputs((N,), H, d, d, inputs.generator(82 + N))
    perm = torch.randperm(B + 3, generator=inputs.generator(83))[:B].to(torch.int32)
    pool = torch.zeros(B + 3, H, d, d)
    pool[perm.long()] = S0
    S = pool.to(dev)
    td = _to(tok, dev)
    o = torch.empty(N, H, d, device=dev)
    hla.kda_extend(B, torch.from_numpy(cu).to(dev), H, d, d, S, perm.to(dev), td["q"], td["k"], td["v"],
                   td["alpha"], td["beta"], o)
    torch.cuda.synchronize()
    S_ref, o_ref = oracle.kda.extend(f64(S0), cu, *(f64(tok[key]) for key in ("q", "k", "v", "alpha", "beta")))
    got = S.cpu()[perm.long()]
    assert max_rel(got.double().numpy(), S_ref) < KDA_MAX_REL
    assert max_rel(f64(o), o_ref) < KDA_MAX_REL
    for b in range(B):
        if lens[b] == 0:
            assert torch.equal(got[b], S0[b])
    # bitwise against single decode steps, one sequence at a time
    S2 = pool.to(dev)
    o2 = torch.empty(N, H, d, device=dev)
    for b in range(B):
        for n in range(cu[b], cu[b + 1]):
            step = {key: val[n:n + 1].contiguous() for key, val in td.items()}
            ob = torch.empty(1, H, d, device=dev)
            hla.kda_decode_step(1, H, d, d, S2, perm[b:b + 1].to(dev), step["q"], step["k"], step["v"],
                                step["alpha"], step["beta"], ob)
            o2[n] = ob[0]
    torch.cuda.synchronize()
    assert torch.equal(S2, S) and torch.equal(o2, o)
