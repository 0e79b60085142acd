"""The q/k/v/gate/beta projection epilogue and the composed hybrid decode layer.

Test infrastructure only (see ``oracle/__init__``).  float64 arithmetic; values
are rounded to bfloat16 / float32 only where the kernels hand a stored tensor
of that type from one operation to the next, so both sides consume inputs of
the same precision at every operation boundary.

Sources
-------
* "Hyper-optimizing Kimi K3 in vLLM", Part 1 section 1: attention input
  projections (small-matrix at batch 1-2, split-K above), then the KDA decode
  kernel; section 2: the attention output projection is followed by the
  attention-residual computation; section 3: router, routed and shared experts.
* "Kimi K3: From Day-0 Availability to Optimized Inference": residual additions
  and normalisation around the projections; KDA's fixed-size recurrent state.

Readings where the pages are silent (the plainest ones):
* one input projection x W^T yields q, k, v (H x d each), a gate g (H x d_k)
  and one beta logit per head; q and k are L2-normalised per head; the decay is
  alpha = exp(-softplus(g)) per key channel; beta = sigmoid(beta logit);
* no short convolution, output gate, positional rotation or output norm;
* residual adds after the output projection and after the MoE block;
* RMSNorm eps = 1e-6.
"""

import numpy as np

from .numerics import f64, round_bf16, round_f32, sigmoid, softplus
from .kda import kda_step
from .moe import rmsnorm, linear, route_topk, moe_forward


def l2_normalise(t):
    """t / ||t||_2 over the last axis (a zero vector stays zero)."""
    t = f64(t)
    n = np.sqrt(np.sum(t * t, axis=-1, keepdims=True))
    return np.where(n > 0, t / np.where(n > 0, n, 1.0), 0.0)


def qkvgb_split(z, H, dk, dv):
    """Split projection rows [q | k | v | g | beta] of z [M, 2*H*dk + H*dv + H*dk + H]."""
    M = z.shape[0]
    o = 0
    q = z[:, o:o + H * dk].reshape(M, H, dk); o += H * dk
    k = z[:, o:o + H * dk].reshape(M, H, dk); o += H * dk
    v = z[:, o:o + H * dv].reshape(M, H, dv); o += H * dv
    g = z[:, o:o + H * dk].reshape(M, H, dk); o += H * dk
    b = z[:, o:o + H]
    return q, k, v, g, b


def qkvg_epilogue(z, H, dk, dv):
    """Projection output -> KDA step inputs, rounded to the stored types.

    q, k: per-head L2 normalisation, stored bf16; v stored bf16;
    alpha = exp(-softplus(g)) stored fp32; beta = sigmoid(b) stored fp32.
    """
    q, k, v, g, b = qkvgb_split(f64(z), H, dk, dv)
    q = round_bf16(l2_normalise(q))
    k = round_bf16(l2_normalise(k))
    v = round_bf16(v)
    alpha = round_f32(np.exp(-softplus(g)))
    beta = round_f32(sigmoid(b))
    return q, k, v, alpha, beta


def decode_layer(x, S, p, experts, shared=()):
    """One hybrid decode layer for M sequences, one token each.

    x [M, Hd] (bf16 values), S [M, H, d_k, d_v] committed states.  p holds
    gamma_attn, gamma_moe [Hd], W_qkvgb, W_o [Hd, H*d_v], W_r [E, Hd], H, dk,
    dv, top_k and eps.  Returns (y [M, Hd] bf16 values, S_new, aux dict).
    """
    H, dk, dv = p["H"], p["dk"], p["dv"]
    eps = p.get("eps", 1e-6)
    x = f64(x)
    M = x.shape[0]
    x1 = round_bf16(rmsnorm(x, p["gamma_attn"], eps))
    z = linear(x1, p["W_qkvgb"])
    q, k, v, alpha, beta = qkvg_epilogue(z, H, dk, dv)
    S_new, o = kda_step(S, q, k, v, alpha, beta)
    o_b = round_bf16(o).reshape(M, H * dv)
    r = round_bf16(x + linear(o_b, p["W_o"]))
    x2 = round_bf16(rmsnorm(r, p["gamma_moe"], eps))
    idx, w, logits = route_topk(x2, p["W_r"], p["top_k"])
    y = round_bf16(moe_forward(x2, idx, w, experts, shared, residual=r))
    aux = dict(x1=x1, q=q, k=k, v=v, alpha=alpha, beta=beta, o=o, r=r, x2=x2,
               topk_idx=idx, topk_w=w, logits=logits)
    return y, S_new, aux
