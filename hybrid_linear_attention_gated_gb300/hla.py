"""ctypes binding of the C ABI in include/hla.h (argument marshalling only).

Every function here has the name and argument order of the C entry point.  A
tensor argument may be a torch tensor (its data_ptr() is passed), a plain
integer address, or None (NULL).  ``stream`` defaults to torch's current CUDA
stream.  A non-zero status raises HlaError.  Nothing here computes: every step
of the path runs in the CUDA library, and the library must be built
(``build.build()``) -- there is no fallback.
"""

import ctypes
import os

from . import build as _build

HLA_OK = 0
HLA_F32 = 0
HLA_BF16 = 1
HLA_SPEC_VERIFY = 1
HLA_SPEC_REPLAY = 2
HLA_SPEC_BOTH = 3  # named by the ABI, answered with HLA_ERR_UNSUPPORTED (see include/hla.h)

_lib = None

c_int, c_size_t, c_float, c_void_p, c_char_p = (ctypes.c_int, ctypes.c_size_t, ctypes.c_float,
                                                ctypes.c_void_p, ctypes.c_char_p)
P = c_void_p  # every tensor / stream argument is an address


class HlaError(RuntimeError):
    def __init__(self, fn, status):
        super().__init__(f"{fn}: status {status} ({status_string(status)})")
        self.status = status


class hla_layer(ctypes.Structure):
    _fields_ = [("hidden", c_int), ("heads", c_int), ("dk", c_int), ("dv", c_int),
                ("n_experts", c_int), ("top_k", c_int), ("inter", c_int), ("n_shared", c_int),
                ("eps", c_float),
                ("gamma_attn", P), ("gamma_moe", P), ("W_qkvgb", P), ("W_o", P),
                ("W_router", P), ("W_gate", P), ("W_up", P), ("W_down", P),
                ("Ws_gate", P), ("Ws_up", P), ("Ws_down", P)]


SIGNATURES = {
    "hla_status_string": (c_char_p, [c_int]),
    "hla_last_variant": (c_char_p, []),
    "hla_version": (c_int, []),
    "hla_chain_begin": (c_int, [P]),
    "hla_chain_end": (c_int, []),
    "kda_decode_step": (c_int, [c_int] * 4 + [P] * 8 + [c_int, P]),
    "kda_spec_verify_replay": (c_int, [c_int] * 6 + [P] * 9 + [c_int, P]),
    "spec_accept_prefix": (c_int, [c_int, c_int] + [P] * 4 + [P]),
    "kda_spec_replay_verify": (c_int, [c_int] * 6 + [P] * 14 + [c_int, P]),
    "kda_extend": (c_int, [c_int, P, c_int, c_int, c_int] + [P] * 8 + [c_int, P]),
    "skinny_proj_splitk_workspace_size": (c_size_t, [c_int] * 4),
    "skinny_proj_splitk": (c_int, [c_int] * 3 + [P] * 4 + [c_int, c_int, P, c_size_t, P]),
    "skinny_proj_residual_rmsnorm_workspace_size": (c_size_t, [c_int] * 4),
    "skinny_proj_residual_rmsnorm": (c_int, [c_int] * 3 + [P] * 4 + [c_float, P, P, c_int, P,
                                                                      c_size_t, P]),
    "kda_qkvg_proj_workspace_size": (c_size_t, [c_int] * 6),
    "kda_qkvg_proj": (c_int, [c_int] * 5 + [P] * 7 + [c_int, P, c_size_t, P]),
    "hla_rmsnorm": (c_int, [c_int, c_int, P, P, c_float, P, P]),
    "moe_route_topk_workspace_size": (c_size_t, [c_int] * 3),
    "moe_route_topk": (c_int, [c_int] * 4 + [P] * 6 + [c_size_t, P]),
    "moe_expert_forward_workspace_size": (c_size_t, [c_int] * 6),
    "moe_expert_forward": (c_int, [c_int] * 6 + [P] * 12 + [c_size_t, P, P]),
    "hla_l2_prefetch": (c_int, [P, c_size_t, P]),
    "hla_decode_layer_workspace_size": (c_size_t, [ctypes.POINTER(hla_layer), c_int]),
    "hla_decode_layer": (c_int, [ctypes.POINTER(hla_layer), c_int] + [P] * 4 + [P, c_size_t, P, P]),
    "hla_decode_layer_routing": (c_int, [ctypes.POINTER(hla_layer), c_int, P,
                                         ctypes.POINTER(c_void_p), ctypes.POINTER(c_void_p)]),
    "skinny_proj_splitk_noalloc": (c_int, [c_int] * 3 + [P] * 4 + [c_int, c_int, P]),
    "hla_launch_count": (ctypes.c_ulonglong, []),
    "hla_device_status": (c_int, []),
    "hla_test_force_wait_timeout": (c_int, [c_int]),
    "hla_trace_enable": (c_int, [c_char_p, c_int]),
    "hla_trace_read": (c_int, [ctypes.POINTER(c_float), c_int]),
}


def library_path():
    return _build.LIB


def load(path=None):
    """Load (once) and return the CUDA library; raises if it has not been built."""
    global _lib
    if _lib is None:
        path = path or library_path()
        if not os.path.exists(path):
            raise RuntimeError(f"CUDA library {path} is missing: build it with "
                               "hybrid_linear_attention_gated_gb300.build.build()")
        lib = ctypes.CDLL(path)
        for name, (res, args) in SIGNATURES.items():
            fn = getattr(lib, name)
            fn.restype = res
            fn.argtypes = args
        _lib = lib
    return _lib


def _p(t):
    if t is None:
        return None
    if isinstance(t, int):
        return t
    return t.data_ptr()


def _stream(s):
    if s is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    if isinstance(s, int):
        return s
    return s.cuda_stream


def _check(fn, status):
    if status != HLA_OK:
        raise HlaError(fn, status)
    return status


def status_string(status):
    return load().hla_status_string(status).decode()


def hla_status_string(status):
    return status_string(status)


def hla_last_variant():
    return load().hla_last_variant().decode()


def hla_version():
    return load().hla_version()


def hla_chain_begin(stream=None):
    return _check("hla_chain_begin", load().hla_chain_begin(_stream(stream)))


def hla_chain_end():
    return _check("hla_chain_end", load().hla_chain_end())


def kda_decode_step(B, H, dk, dv, S, state_idx, q, k, v, alpha, beta, o, o_dtype=HLA_F32,
                    stream=None):
    return _check("kda_decode_step", load().kda_decode_step(
        B, H, dk, dv, _p(S), _p(state_idx), _p(q), _p(k), _p(v), _p(alpha), _p(beta), _p(o),
        o_dtype, _stream(stream)))


def kda_spec_verify_replay(phase, B, T, H, dk, dv, S, state_idx, q, k, v, alpha, beta,
                           accepted_len, o, o_dtype=HLA_F32, stream=None):
    return _check("kda_spec_verify_replay", load().kda_spec_verify_replay(
        phase, B, T, H, dk, dv, _p(S), _p(state_idx), _p(q), _p(k), _p(v), _p(alpha), _p(beta),
        _p(accepted_len), _p(o), o_dtype, _stream(stream)))


def kda_spec_replay_verify(B, T_prev, T, H, dk, dv, S, state_idx, q_prev, k_prev, v_prev,
                           alpha_prev, beta_prev, accepted_prev, q, k, v, alpha, beta, o,
                           o_dtype=HLA_F32, stream=None):
    return _check("kda_spec_replay_verify", load().kda_spec_replay_verify(
        B, T_prev, T, H, dk, dv, _p(S), _p(state_idx), _p(q_prev), _p(k_prev), _p(v_prev),
        _p(alpha_prev), _p(beta_prev), _p(accepted_prev), _p(q), _p(k), _p(v), _p(alpha), _p(beta),
        _p(o), o_dtype, _stream(stream)))


def kda_extend(B, cu_seqlens, H, dk, dv, S, state_idx, q, k, v, alpha, beta, o, o_dtype=HLA_F32,
               stream=None):
    return _check("kda_extend", load().kda_extend(
        B, _p(cu_seqlens), H, dk, dv, _p(S), _p(state_idx), _p(q), _p(k), _p(v), _p(alpha),
        _p(beta), _p(o), o_dtype, _stream(stream)))


def spec_accept_prefix(B, T, draft_ids, target_ids, accepted_len, committed_len, stream=None):
    return _check("spec_accept_prefix", load().spec_accept_prefix(
        B, T, _p(draft_ids), _p(target_ids), _p(accepted_len), _p(committed_len),
        _stream(stream)))


def skinny_proj_splitk_workspace_size(M, N, K, split=0):
    return load().skinny_proj_splitk_workspace_size(M, N, K, split)


def skinny_proj_splitk(M, N, K, x, W, residual, y, y_dtype, split, ws, ws_bytes, stream=None):
    return _check("skinny_proj_splitk", load().skinny_proj_splitk(
        M, N, K, _p(x), _p(W), _p(residual), _p(y), y_dtype, split, _p(ws), ws_bytes,
        _stream(stream)))


def skinny_proj_residual_rmsnorm_workspace_size(M, N, K, split=0):
    return load().skinny_proj_residual_rmsnorm_workspace_size(M, N, K, split)


def skinny_proj_residual_rmsnorm(M, N, K, x, W, residual, gamma, eps, r, xn, split, ws, ws_bytes,
                                 stream=None):
    return _check("skinny_proj_residual_rmsnorm", load().skinny_proj_residual_rmsnorm(
        M, N, K, _p(x), _p(W), _p(residual), _p(gamma), eps, _p(r), _p(xn), split, _p(ws), ws_bytes,
        _stream(stream)))


def kda_qkvg_proj_workspace_size(M, Hd, H, dk, dv, split=0):
    return load().kda_qkvg_proj_workspace_size(M, Hd, H, dk, dv, split)


def kda_qkvg_proj(M, Hd, H, dk, dv, x, W, q, k, v, alpha, beta, split, ws, ws_bytes, stream=None):
    return _check("kda_qkvg_proj", load().kda_qkvg_proj(
        M, Hd, H, dk, dv, _p(x), _p(W), _p(q), _p(k), _p(v), _p(alpha), _p(beta), split, _p(ws),
        ws_bytes, _stream(stream)))


def hla_rmsnorm(M, Hd, x, gamma, eps, y, stream=None):
    return _check("hla_rmsnorm", load().hla_rmsnorm(M, Hd, _p(x), _p(gamma), eps, _p(y),
                                                    _stream(stream)))


def moe_route_topk_workspace_size(M, Hd, E):
    return load().moe_route_topk_workspace_size(M, Hd, E)


def moe_route_topk(M, Hd, E, k, x, W_r, topk_idx, topk_w, logits, ws, ws_bytes, stream=None):
    return _check("moe_route_topk", load().moe_route_topk(
        M, Hd, E, k, _p(x), _p(W_r), _p(topk_idx), _p(topk_w), _p(logits), _p(ws), ws_bytes,
        _stream(stream)))


def moe_expert_forward_workspace_size(M, Hd, I, E, k, n_shared):
    return load().moe_expert_forward_workspace_size(M, Hd, I, E, k, n_shared)


def moe_expert_forward(M, Hd, I, E, k, n_shared, x, topk_idx, topk_w, W_gate, W_up, W_down,
                       Ws_gate, Ws_up, Ws_down, residual, y, ws, ws_bytes, stream=None,
                       prefetch_stream=0):
    return _check("moe_expert_forward", load().moe_expert_forward(
        M, Hd, I, E, k, n_shared, _p(x), _p(topk_idx), _p(topk_w), _p(W_gate), _p(W_up),
        _p(W_down), _p(Ws_gate), _p(Ws_up), _p(Ws_down), _p(residual), _p(y), _p(ws), ws_bytes,
        _stream(stream), prefetch_stream and _stream(prefetch_stream) or None))


def hla_l2_prefetch(ptr, nbytes, stream=None):
    return _check("hla_l2_prefetch", load().hla_l2_prefetch(_p(ptr), nbytes, _stream(stream)))


def make_layer(hidden, heads, dk, dv, n_experts, top_k, inter, n_shared, eps, weights):
    """Build an hla_layer descriptor from a dict of device tensors (keeps no references)."""
    L = hla_layer(hidden, heads, dk, dv, n_experts, top_k, inter, n_shared, eps)
    for name in ("gamma_attn", "gamma_moe", "W_qkvgb", "W_o"):
        setattr(L, name, _p(weights[name]))
    L.W_router = _p(weights["W_r"])
    for name in ("W_gate", "W_up", "W_down", "Ws_gate", "Ws_up", "Ws_down"):
        setattr(L, name, _p(weights.get(name)))
    return L


def hla_decode_layer_workspace_size(L, M):
    return load().hla_decode_layer_workspace_size(ctypes.byref(L), M)


def hla_decode_layer(L, M, x, S, state_idx, y, ws, ws_bytes, stream=None, prefetch_stream=0):
    return _check("hla_decode_layer", load().hla_decode_layer(
        ctypes.byref(L), M, _p(x), _p(S), _p(state_idx), _p(y), _p(ws), ws_bytes,
        _stream(stream), prefetch_stream and _stream(prefetch_stream) or None))


def hla_decode_layer_routing(L, M, ws):
    """(topk_idx address, topk_w address) inside a layer workspace."""
    a, b = c_void_p(), c_void_p()
    _check("hla_decode_layer_routing", load().hla_decode_layer_routing(ctypes.byref(L), M, _p(ws),
                                                                      ctypes.byref(a), ctypes.byref(b)))
    return a.value, b.value


def hla_launch_count():
    return load().hla_launch_count()


def hla_trace_enable(kernel, capacity):
    return _check("hla_trace_enable", load().hla_trace_enable(
        kernel.encode() if kernel else None, capacity))


def hla_trace_read(max_n=4096):
    buf = (c_float * max_n)()
    n = load().hla_trace_read(buf, max_n)
    if n < 0:
        raise HlaError("hla_trace_read", -n)
    return [buf[i] for i in range(min(n, max_n))]


HLA_NOALLOC_SCRATCH_BYTES = 16 << 20


def skinny_proj_splitk_noalloc(M, N, K, x, W, residual, y, y_dtype, split, stream=None):
    """skinny_proj_splitk with its split-K partials in the library's fixed device array
    (for callers that cannot allocate a workspace); see include/hla.h."""
    return _check("skinny_proj_splitk_noalloc", load().skinny_proj_splitk_noalloc(
        M, N, K, _p(x), _p(W), _p(residual), _p(y), y_dtype, split, _stream(stream)))


def hla_device_status():
    return load().hla_device_status()


def hla_test_force_wait_timeout(on):
    return _check("hla_test_force_wait_timeout", load().hla_test_force_wait_timeout(int(on)))
