"""RMSNorm, dense projections, sigmoid top-k router and SwiGLU experts.

Test infrastructure only (see ``oracle/__init__``).  float64 throughout.

Sources
-------
* "Kimi K3: From Day-0 Availability to Optimized Inference", paragraph on
  profiling: at low batch the cost is moving *expert weights* through GPU
  memory; paragraph on optimisations: residual additions and normalisation sit
  next to the projections.
* "Hyper-optimizing Kimi K3 in vLLM", Part 1 section 3 ("Improve MoE
  scheduling and overlap"): router scores feed routed experts, and a *shared
  expert* runs for every token beside them.  Section 1 ("Tune shapes for the
  workload"): the projections are skinny matrix products x W^T.
* "Kimi-K3 release on HuggingFace", section "Decoding the Model Configuration":
  rms_norm_eps = 1e-6 (the only constant taken from that page).

The pages give no router formula.  The reading used: per-expert score
s_e = sigmoid(x . w_e) computed from float32-or-better logits, the k experts
with the largest scores (ties broken towards the lower expert index, listed in
descending score), mixing weights s / sum(s over the chosen k); no score bias,
no expert groups, no extra scaling.  Experts are SwiGLU MLPs
y = W_down (SiLU(W_gate x) * (W_up x)); shared experts have weight 1 and are
not part of the renormalisation.
"""

import numpy as np

from .numerics import f64, sigmoid, silu

RMS_NORM_EPS = 1e-6


def rmsnorm(x, gamma, eps=RMS_NORM_EPS):
    """y = x * gamma / sqrt(mean(x^2) + eps), over the last axis."""
    x = f64(x)
    ms = np.mean(x * x, axis=-1, keepdims=True)
    return x * f64(gamma) / np.sqrt(ms + eps)


def linear(x, W):
    """y = x W^T for x [M, K], W [N, K]."""
    return f64(x) @ f64(W).T


def router_logits(x, W_r):
    """Router logits x W_r^T, [M, E]."""
    return linear(x, W_r)


def route_topk(x, W_r, k):
    """Sigmoid top-k routing.  Returns (idx [M,k] int64, w [M,k], logits [M,E]).

    The order among the chosen experts is by descending score, then ascending
    expert index; the full list of E experts is sorted for every token.
    """
    logits = router_logits(x, W_r)
    scores = sigmoid(logits)
    M, E = scores.shape
    idx = np.zeros((M, k), dtype=np.int64)
    w = np.zeros((M, k))
    for m in range(M):
        order = sorted(range(E), key=lambda e: (-scores[m, e], e))
        chosen = order[:k]
        idx[m] = chosen
        w[m] = scores[m, chosen] / scores[m, chosen].sum()
    return idx, w, logits


def swiglu_expert(x, W_gate, W_up, W_down):
    """One SwiGLU expert on one token x [Hd]: W_down (SiLU(W_gate x) * (W_up x))."""
    x = f64(x)
    g = f64(W_gate) @ x
    u = f64(W_up) @ x
    h = silu(g) * u
    return f64(W_down) @ h


def moe_forward(x, topk_idx, topk_w, experts, shared=(), residual=None):
    """Routed + shared expert output for tokens x [M, Hd].

    experts : callable e -> (W_gate [I,Hd], W_up [I,Hd], W_down [Hd,I]) or a
              tuple of stacked arrays (W_gate [E,I,Hd], W_up, W_down [E,Hd,I]).
    shared  : sequence of (W_gate, W_up, W_down) for the always-on experts.
    y[m] = sum_j topk_w[m,j] * expert_{topk_idx[m,j]}(x[m]) + sum_s shared_s(x[m])
           (+ residual[m]).
    """
    if not callable(experts):
        Wg_all, Wu_all, Wd_all = experts

        def experts(e):  # noqa: F811  (stacked arrays -> accessor)
            return Wg_all[e], Wu_all[e], Wd_all[e]

    x = f64(x)
    M = x.shape[0]
    y = []
    for m in range(M):
        acc = None
        for j in range(topk_idx.shape[1]):
            e = int(topk_idx[m, j])
            ye = float(topk_w[m, j]) * swiglu_expert(x[m], *experts(e))
            acc = ye if acc is None else acc + ye
        for (Wg, Wu, Wd) in shared:
            ys = swiglu_expert(x[m], Wg, Wu, Wd)
            acc = ys if acc is None else acc + ys
        if residual is not None:
            acc = acc + f64(residual[m])
        y.append(acc)
    return np.stack(y)
