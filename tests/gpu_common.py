"""Helpers shared by the GPU parity tests (comparison metrics, oracle-built warm states)."""

import collections
import functools

import numpy as np
import pytest
import torch

import oracle
from hybrid_linear_attention_gated_gb300 import build, hla, inputs

# Tolerances (stated by the workload definition):
KDA_MAX_REL = 2e-3        # KDA outputs and states: max relative error (floored, see max_rel)
MOE_FROB_REL = 1e-2       # bf16-weight MoE outputs: relative Frobenius error
ROUTER_W_REL = 1e-5       # router mixing weights (fp32 level)
PROJ_FROB_REL_BF16 = 1e-2
PROJ_FROB_REL_F32 = 1e-3
LAYER_FROB_REL = 1e-2


def require_gpu():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    build.build()
    hla.load()
    return torch.device("cuda:0")


def f64(t):
    return t.detach().to("cpu").double().numpy()


def max_rel(got, ref):
    """max_i |g_i - r_i| / max(|r_i|, 1e-3 * max|r|)  (the floor keeps near-zero entries
    from dominating a tensor whose scale is set by its large entries)."""
    got = np.asarray(got, np.float64)
    ref = np.asarray(ref, np.float64)
    floor = 1e-3 * float(np.max(np.abs(ref))) if ref.size else 1.0
    return float(np.max(np.abs(got - ref) / np.maximum(np.abs(ref), max(floor, 1e-300)))) if ref.size else 0.0


def frob_rel(got, ref):
    got = np.asarray(got, np.float64)
    ref = np.asarray(ref, np.float64)
    return float(np.linalg.norm(got - ref) / max(np.linalg.norm(ref), 1e-300))


@functools.lru_cache(maxsize=4)
def warm_pool(seed, P, d, n_updates=256):
    """P committed states, each the oracle's result of n_updates random updates from 0."""
    g = inputs.generator(seed)
    u = inputs.warm_update_inputs(n_updates, P, d, d, g)
    f = lambda t: t.double().numpy()  # noqa: E731
    return oracle.kda.warm_state((P, d, d), f(u["q"]), f(u["k"]), f(u["v"]), f(u["alpha"]),
                                 f(u["beta"]))


def warm_states(seed, B, H, d, P=64):
    """fp32 states [B, H, d, d] drawn from the warm pool by a seeded assignment."""
    pool = warm_pool(seed, P, d).astype(np.float32)
    assign = inputs.pool_assignment(B * H, P, inputs.generator(seed + 7)).numpy()
    return torch.from_numpy(pool[assign].reshape(B, H, d, d).copy())


FULL = dict(Hd=7168, I=2048, E=256, k=8, n_shared=1)


def f64_big(t):
    """Exact fp64 host copy of a large device tensor (widened on the device, then copied)."""
    return t.detach().to(torch.float64).to("cpu").numpy()


class ExpertCache:
    """An expert's three matrices as fp64 host arrays, fetched when the oracle asks for them.
    At most ``capacity`` experts are kept (least recently used dropped first), so that
    comparing every token of a 64-token batch does not hold ~220 experts (~77 GB in fp64)."""

    def __init__(self, w, capacity=16):
        self.w, self.capacity = w, capacity
        self.cache = collections.OrderedDict()

    def __call__(self, e):
        e = int(e)
        if e in self.cache:
            self.cache.move_to_end(e)
        else:
            while len(self.cache) >= self.capacity:
                self.cache.popitem(last=False)
            self.cache[e] = (f64_big(self.w["W_gate"][e]), f64_big(self.w["W_up"][e]),
                             f64_big(self.w["W_down"][e]))
        return self.cache[e]

    def shared(self):
        return [(f64_big(self.w["Ws_gate"][s]), f64_big(self.w["Ws_up"][s]), f64_big(self.w["Ws_down"][s]))
                for s in range(self.w["Ws_gate"].shape[0])]
