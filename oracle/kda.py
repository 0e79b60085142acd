"""KDA recurrent-state decode, speculative verify, accepted-prefix bookkeeping and replay.

Test infrastructure only (see ``oracle/__init__``).  float64 throughout.

Sources
-------
* "Kimi K3: From Day-0 Availability to Optimized Inference" (webinar summary),
  opening paragraph: Kimi Delta Attention (KDA) keeps a *fixed-size recurrent
  state* per sequence that every generated token updates.  The page names the
  state but not its update rule; the rule used here is the gated delta rule

      S_t = (I - beta_t k_t k_t^T) diag(alpha_t) S_{t-1} + beta_t k_t v_t^T
      o_t = S_t^T q_t

  with S a d_k x d_v matrix per (sequence, head), alpha_t in (0,1)^{d_k} a
  per-key-channel decay (so diag(alpha) scales the *rows* of S), beta_t a scalar
  write strength, and the output read from the *updated* state.  No 1/sqrt(d_k)
  scaling of q is applied: none appears in the rule.
* Same page, paragraphs on speculative decoding: a drafter proposes several
  tokens, the target verifies them, and because KDA's state is recurrent a
  partial rejection is handled by *storing the drafted tokens' recurrent inputs*
  and *replaying only the accepted portion from the last committed state*.

Array conventions (leading batch axes are free):
  S      [..., d_k, d_v]
  q, k   [..., d_k]      v [..., d_v]
  alpha  [..., d_k]      beta [...]
Windowed inputs carry the draft position as axis 1: q is [B, T, H, d_k] etc.
"""

import numpy as np

from .numerics import f64


def kda_step(S, q, k, v, alpha, beta):
    """One gated-delta-rule update of the state and the output read from it.

    The matrix products of the rule are written out term by term:
      diag(alpha) S                     -> row i of S multiplied by alpha_i
      (I - beta k k^T) X = X - beta k (k^T X)
      + beta k v^T                      -> outer product
      o = S_t^T q                       -> o_j = sum_i S_t[i, j] q_i
    Returns (S_t, o_t); the input S is not modified.
    """
    S, q, k, v, alpha, beta = (f64(a) for a in (S, q, k, v, alpha, beta))
    decayed = alpha[..., :, None] * S                        # diag(alpha) S
    kT_decayed = np.einsum("...i,...ij->...j", k, decayed)   # k^T diag(alpha) S
    b = beta[..., None, None]
    S_t = (decayed
           - b * k[..., :, None] * kT_decayed[..., None, :]  # - beta k k^T diag(alpha) S
           + b * k[..., :, None] * v[..., None, :])          # + beta k v^T
    o_t = np.einsum("...ij,...i->...j", S_t, q)              # S_t^T q
    return S_t, o_t


def kda_run(S0, q, k, v, alpha, beta):
    """Apply T steps in order; inputs are [T, ...].  Returns (S_T, o[T, ...])."""
    S = f64(S0)
    outs = []
    for t in range(len(q)):
        S, o = kda_step(S, q[t], k[t], v[t], alpha[t], beta[t])
        outs.append(o)
    return S, np.stack(outs) if outs else np.zeros((0,) + S.shape[:-2] + S.shape[-1:])


def warm_state(shape_dk_dv, q, k, v, alpha, beta):
    """State after len(q) updates starting from S_0 = 0 (used to build realistic
    committed states).  shape_dk_dv is the leading shape + (d_k, d_v)."""
    S, _ = kda_run(np.zeros(shape_dk_dv), q, k, v, alpha, beta)
    return S


def spec_verify(S_c, q, k, v, alpha, beta):
    """Score a drafted window from the committed state without committing it.

    S_c [B, H, d_k, d_v]; q, k, alpha [B, T, H, d_k]; v [B, T, H, d_v];
    beta [B, T, H].  The T drafted tokens are applied one after another to a
    private copy of S_c and the output of every position is kept.
    Returns o [B, T, H, d_v]; S_c is left as it was.
    """
    S = f64(S_c).copy()
    T = q.shape[1]
    outs = []
    for t in range(T):
        S, o = kda_step(S, q[:, t], k[:, t], v[:, t], alpha[:, t], beta[:, t])
        outs.append(o)
    return np.stack(outs, axis=1)


def accept_prefix(draft_ids, target_ids, committed_len):
    """Greedy acceptance of a drafted window.

    accepted_len[b] = number of leading positions t at which the drafter's token
    equals the target's token (the first mismatch ends acceptance);
    committed_len[b] grows by accepted_len[b].
    Returns (accepted_len, new_committed_len) as int64 arrays.
    """
    draft_ids = np.asarray(draft_ids)
    target_ids = np.asarray(target_ids)
    B, T = draft_ids.shape
    accepted = np.zeros(B, dtype=np.int64)
    for b in range(B):
        n = 0
        while n < T and draft_ids[b, n] == target_ids[b, n]:
            n += 1
        accepted[b] = n
    return accepted, np.asarray(committed_len, dtype=np.int64) + accepted


def spec_replay(S_c, q, k, v, alpha, beta, accepted_len):
    """Rebuild each sequence's committed state from the stored window inputs.

    Sequence b replays only its first accepted_len[b] drafted tokens, in order,
    starting from its last committed state S_c[b]; a sequence with nothing
    accepted keeps S_c[b].  Returns the new committed states [B, H, d_k, d_v].
    """
    S = f64(S_c).copy()
    for b in range(S.shape[0]):
        for t in range(int(accepted_len[b])):
            S[b], _ = kda_step(S[b], q[b, t], k[b, t], v[b, t], alpha[b, t], beta[b, t])
    return S


def spec_replay_verify(S_c, prev, accepted_prev, new):
    """One speculative step in fused form: commit the accepted prefix of the previous window,
    then verify the new window from the new committed state.

    prev / new: dicts of q, k, v, alpha, beta with the draft axis at 1.  Returns
    (new committed states [B, H, d_k, d_v], outputs of the new window [B, T, H, d_v]).
    """
    S = spec_replay(S_c, prev["q"], prev["k"], prev["v"], prev["alpha"], prev["beta"], accepted_prev)
    o = spec_verify(S, new["q"], new["k"], new["v"], new["alpha"], new["beta"])
    return S, o


def extend(S, cu_seqlens, q, k, v, alpha, beta):
    """Mixed batch: sequence b applies its packed tokens cu_seqlens[b]..cu_seqlens[b+1]-1 in
    order.  q, k, alpha [N, H, d_k]; v [N, H, d_v]; beta [N, H]; S [B, H, d_k, d_v].
    Returns (new states, o [N, H, d_v])."""
    S = f64(S).copy()
    N = q.shape[0]
    o = np.zeros((N,) + tuple(np.shape(v)[1:]))
    for b in range(S.shape[0]):
        for n in range(int(cu_seqlens[b]), int(cu_seqlens[b + 1])):
            S[b], o[n] = kda_step(S[b], q[n], k[n], v[n], alpha[n], beta[n])
    return S, o
