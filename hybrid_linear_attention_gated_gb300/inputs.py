"""Seeded synthetic inputs for the KDA decode / speculative window / routed-MoE workloads.

This module only draws random tensors in the shapes, dtypes and value
distributions of the workloads; it computes none of the operations the library
implements.  Tests feed the same tensors to the CUDA library and to the oracle;
the benchmark uses them for timing.  Draws happen in a fixed order per call, so
a (seed, device) pair always yields the same tensors on that device.

Distributions (per the workload descriptions):
  q, k   ~ N(0,1), L2-normalised per (token, head), stored bf16
  v      ~ N(0,1), bf16
  alpha  = exp(-softplus(z)), z ~ N(0,1), per key channel, fp32, in (0,1)
  beta   = sigmoid(z), z ~ N(0,1), per (token, head), fp32
  tiny-case state S_0 ~ N(0, 0.02^2) fp32
  weights ~ N(0, 0.02^2) bf16; activations ~ N(0,1) bf16
  RMSNorm gains = 1 + 0.1 N(0,1), bf16
"""

import torch

BF16 = torch.bfloat16
F32 = torch.float32


def generator(seed, device="cpu"):
    g = torch.Generator(device=device)
    g.manual_seed(int(seed))
    return g


def _randn(shape, g, device, std=1.0, dtype=F32):
    t = torch.randn(tuple(shape), generator=g, device=device, dtype=F32)
    if std != 1.0:
        t.mul_(std)
    return t.to(dtype)


def _unit_rows_bf16(t):
    """Scale each last-axis vector of a fresh N(0,1) draw to unit length, store bf16."""
    return (t / t.norm(dim=-1, keepdim=True).clamp_min(1e-30)).to(BF16)


def kda_inputs(lead, H, dk, dv, g, device="cpu"):
    """Per-token KDA inputs with leading shape `lead` (e.g. (B,) or (B, T)).

    Returns dict q, k [*lead, H, dk] bf16; v [*lead, H, dv] bf16;
    alpha [*lead, H, dk] fp32; beta [*lead, H] fp32.
    """
    lead = tuple(lead)
    q = _unit_rows_bf16(_randn(lead + (H, dk), g, device))
    k = _unit_rows_bf16(_randn(lead + (H, dk), g, device))
    v = _randn(lead + (H, dv), g, device, dtype=BF16)
    alpha = torch.exp(-torch.nn.functional.softplus(_randn(lead + (H, dk), g, device)))
    beta = torch.sigmoid(_randn(lead + (H,), g, device))
    return dict(q=q, k=k, v=v, alpha=alpha.contiguous(), beta=beta.contiguous())


def small_state(B, H, dk, dv, g, device="cpu", std=0.02):
    """S_0 ~ N(0, std^2), fp32 [B, H, dk, dv] (tiny oracle case)."""
    return _randn((B, H, dk, dv), g, device, std=std)


def warm_update_inputs(n_updates, P, dk, dv, g, device="cpu"):
    """Inputs for `n_updates` prior updates of P independent states (one head each).

    Shapes [n_updates, P, d]; a committed state is the result of applying them in
    order from S = 0 (done by whoever consumes them).
    """
    d = kda_inputs((n_updates, P), 1, dk, dv, g, device)
    return {key: val.squeeze(2) for key, val in d.items()}


def pool_assignment(n_heads, P, g, device="cpu"):
    """Which of P pooled warm states each of n_heads (sequence, head) slots starts from."""
    if n_heads <= P:
        return torch.randperm(P, generator=g, device=device)[:n_heads]
    return torch.randint(0, P, (n_heads,), generator=g, device=device)


def accept_ids(B, T, g, device="cpu", vocab=163840):
    """Drafted and target token ids with accepted length uniform in {0..T}.

    Returns (draft_ids, target_ids) int32 [B, T] and the intended accepted
    lengths int64 [B]: targets equal drafts before position a_b, differ at a_b
    (when a_b < T), and are random after it.
    """
    a = torch.randint(0, T + 1, (B,), generator=g, device=device)
    draft = torch.randint(0, vocab, (B, T), generator=g, device=device, dtype=torch.int64)
    later = torch.randint(0, vocab, (B, T), generator=g, device=device, dtype=torch.int64)
    bump = torch.randint(1, vocab, (B, T), generator=g, device=device, dtype=torch.int64)
    pos = torch.arange(T, device=device)[None, :]
    target = torch.where(pos < a[:, None], draft,
                         torch.where(pos == a[:, None], (draft + bump) % vocab, later))
    return draft.to(torch.int32), target.to(torch.int32), a


def activations(M, Hd, g, device="cpu"):
    """Token activations x ~ N(0,1), bf16 [M, Hd]."""
    return _randn((M, Hd), g, device, dtype=BF16)


def gains(Hd, g, device="cpu"):
    """RMSNorm gains 1 + 0.1 N(0,1), bf16 [Hd]."""
    return (1.0 + 0.1 * _randn((Hd,), g, device)).to(BF16)


def weight(shape, g, device="cpu", std=0.02):
    """A bf16 weight matrix ~ N(0, std^2), drawn in fp32 one leading slice at a time."""
    shape = tuple(shape)
    out = torch.empty(shape, dtype=BF16, device=device)
    if len(shape) == 3:
        for i in range(shape[0]):
            out[i] = _randn(shape[1:], g, device, std=std, dtype=BF16)
    else:
        out.copy_(_randn(shape, g, device, std=std, dtype=BF16))
    return out


def moe_weights(E, Hd, I, n_shared, g, device="cpu", std=0.02):
    """Router and expert weights.

    W_r [E, Hd]; W_gate, W_up [E, I, Hd]; W_down [E, Hd, I]; shared expert
    stacks Ws_gate, Ws_up [n_shared, I, Hd], Ws_down [n_shared, Hd, I].
    """
    W_r = weight((E, Hd), g, device, std)
    W_gate = weight((E, I, Hd), g, device, std)
    W_up = weight((E, I, Hd), g, device, std)
    W_down = weight((E, Hd, I), g, device, std)
    if n_shared:
        Ws_gate = weight((n_shared, I, Hd), g, device, std)
        Ws_up = weight((n_shared, I, Hd), g, device, std)
        Ws_down = weight((n_shared, Hd, I), g, device, std)
    else:
        Ws_gate = Ws_up = Ws_down = None
    return dict(W_r=W_r, W_gate=W_gate, W_up=W_up, W_down=W_down,
                Ws_gate=Ws_gate, Ws_up=Ws_up, Ws_down=Ws_down)


def layer_weights(Hd, H, dk, dv, g, device="cpu", std=0.02):
    """Attention-side weights of one hybrid decode layer.

    gamma_attn, gamma_moe [Hd]; W_qkvgb [(3*dk + dv)*H + H, Hd] whose rows are
    [q | k | v | gate | beta]; W_o [Hd, H*dv].
    """
    gamma_attn = gains(Hd, g, device)
    gamma_moe = gains(Hd, g, device)
    W_qkvgb = weight(((3 * dk + dv) * H + H, Hd), g, device, std)
    W_o = weight((Hd, H * dv), g, device, std)
    return dict(gamma_attn=gamma_attn, gamma_moe=gamma_moe, W_qkvgb=W_qkvgb, W_o=W_o)
