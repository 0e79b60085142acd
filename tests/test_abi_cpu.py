"""The C-ABI library without a GPU: it loads, exports every symbol include/hla.h declares,
answers workspace queries, and rejects bad arguments on the host before any launch."""

import ctypes
import os
import re

import pytest

from hybrid_linear_attention_gated_gb300 import build, hla

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    build.build()
    return hla.load()


def declared_functions():
    src = open(os.path.join(ROOT, "include", "hla.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    names = re.findall(r"^[A-Za-z_][\w \*]*?\b([a-z_][a-z0-9_]*)\s*\(", src, flags=re.M)
    return sorted(set(n for n in names if n not in ("if", "while", "sizeof")))


def test_header_declares_the_entry_points():
    names = declared_functions()
    for n in ["kda_decode_step", "kda_spec_verify_replay", "spec_accept_prefix",
              "skinny_proj_splitk", "moe_route_topk", "moe_expert_forward"]:
        assert n in names


def test_every_declared_symbol_is_exported(lib):
    missing = [n for n in declared_functions() if not hasattr(lib, n)]
    assert missing == []
    assert set(hla.SIGNATURES) == set(declared_functions())


def declared_signatures():
    """name -> list of parameter type strings, parsed from include/hla.h."""
    src = open(os.path.join(ROOT, "include", "hla.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    src = re.sub(r"#.*", "", src)
    out = {}
    for m in re.finditer(r"([A-Za-z_][\w \*]*?)\b([a-z_][a-z0-9_]*)\s*\(([^;{]*?)\)\s*;", src, flags=re.S):
        params = [p.strip() for p in m.group(3).split(",")]
        out[m.group(2)] = [] if params == ["void"] or params == [""] else params
    return out


def test_binding_signatures_match_the_header(lib):
    """Every ctypes signature has the header's parameter count, and pointer parameters are
    marshalled as pointers (a pointer passed as int would be truncated)."""
    sigs = declared_signatures()
    assert set(sigs) == set(hla.SIGNATURES)
    for name, params in sigs.items():
        _, argtypes = hla.SIGNATURES[name]
        assert len(argtypes) == len(params), name
        for decl, at in zip(params, argtypes):
            is_ptr = "*" in decl or decl.startswith("hla_stream")
            assert is_ptr == (at is not ctypes.c_int and at is not ctypes.c_float and
                              at is not ctypes.c_size_t), (name, decl, at)


def test_built_for_sm103a_only(lib):
    assert "arch=compute_103a,code=sm_103a" in " ".join(build.ARCH)


def test_status_strings_and_version(lib):
    assert hla.status_string(0) == "ok"
    assert "workspace" in hla.status_string(4)
    assert hla.hla_version() >= 100


def test_workspace_queries(lib):
    assert hla.skinny_proj_splitk_workspace_size(64, 7168, 4096, 1) == 0
    assert hla.skinny_proj_splitk_workspace_size(64, 7168, 4096, 4) == 4 * 64 * 7168 * 4
    assert hla.kda_qkvg_proj_workspace_size(1, 7168, 32, 128, 128, 2) == 2 * (4 * 32 * 128 + 32) * 4
    assert hla.moe_route_topk_workspace_size(8, 7168, 256) > 0
    w1 = hla.moe_expert_forward_workspace_size(1, 7168, 2048, 256, 8, 1)
    w64 = hla.moe_expert_forward_workspace_size(64, 7168, 2048, 256, 8, 1)
    assert 0 < w1 < w64
    assert hla.moe_expert_forward_workspace_size(0, 7168, 2048, 256, 8, 1) == 0


FAKE = 0x10000  # never dereferenced: validation fails before any launch


@pytest.mark.parametrize("args,status", [
    ((0, 32, 128, 128), 1),     # B = 0
    ((1, 32, 96, 96), 2),       # unsupported head dim
    ((1, 32, 128, 64), 2),      # dk != dv
])
def test_kda_decode_rejects_bad_shapes(lib, args, status):
    r = lib.kda_decode_step(*args, FAKE, None, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, 0, None)
    assert r == status


def test_kda_rejects_null_and_misaligned(lib):
    assert lib.kda_decode_step(1, 4, 64, 64, None, None, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, 0, None) == 1
    assert lib.kda_decode_step(1, 4, 64, 64, FAKE + 4, None, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, 0, None) == 3


def test_spec_window_rejects_bad_phase_and_long_window(lib):
    # BOTH is a named phase that no single call can serve (a window's acceptance depends on its
    # own verify outputs): unsupported, not an invalid argument
    assert lib.kda_spec_verify_replay(hla.HLA_SPEC_BOTH, 1, 4, 4, 64, 64, FAKE, None, FAKE, FAKE,
                                      FAKE, FAKE, FAKE, FAKE, FAKE, 0, None) == 2
    assert lib.kda_spec_verify_replay(4, 1, 4, 4, 64, 64, FAKE, None, FAKE, FAKE, FAKE, FAKE, FAKE,
                                      FAKE, FAKE, 0, None) == 1
    assert lib.kda_spec_verify_replay(0, 1, 4, 4, 64, 64, FAKE, None, FAKE, FAKE, FAKE, FAKE, FAKE,
                                      FAKE, FAKE, 0, None) == 1
    assert lib.kda_spec_verify_replay(1, 1, 9, 4, 64, 64, FAKE, None, FAKE, FAKE, FAKE, FAKE, FAKE,
                                      None, FAKE, 0, None) == 2
    # replay needs accepted_len
    assert lib.kda_spec_verify_replay(2, 1, 4, 4, 64, 64, FAKE, None, FAKE, FAKE, FAKE, FAKE, FAKE,
                                      None, None, 0, None) == 1


def test_short_workspace_is_rejected(lib):
    need = hla.moe_expert_forward_workspace_size(4, 256, 128, 16, 2, 1)
    r = lib.moe_expert_forward(4, 256, 128, 16, 2, 1, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE,
                               FAKE, None, FAKE, FAKE, need - 16, None, None)
    assert r == 4
    assert lib.skinny_proj_splitk(4, 256, 256, FAKE, FAKE, None, FAKE, 0, 4, None, 0, None) == 4
    assert lib.moe_route_topk(2, 256, 16, 2, FAKE, FAKE, FAKE, FAKE, None, None, 0, None) == 4


def test_router_and_moe_shape_limits(lib):
    assert lib.moe_route_topk(1, 256, 16, 17, FAKE, FAKE, FAKE, FAKE, None, FAKE, 1 << 30, None) == 2
    assert lib.moe_route_topk(1, 250, 16, 2, FAKE, FAKE, FAKE, FAKE, None, FAKE, 1 << 30, None) == 2
    assert lib.moe_expert_forward(1, 256, 128, 1020, 2, 8, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE,
                                  FAKE, FAKE, None, FAKE, FAKE, 1 << 30, None, None) == 2


def test_layer_rejects_aliasing_and_bad_descriptor(lib):
    L = hla.hla_layer(7168, 32, 128, 128, 256, 8, 2048, 1, 1e-6)
    assert lib.hla_decode_layer(ctypes.byref(L), 1, FAKE, FAKE, None, FAKE, FAKE, 1 << 30, None, None) == 1
    assert hla.hla_decode_layer_workspace_size(L, 1) == 0


def test_oracle_is_not_on_the_product_path():
    """The package and the CUDA sources never import or mention the oracle."""
    pkg = os.path.join(ROOT, "hybrid_linear_attention_gated_gb300")
    for dirpath, _, files in os.walk(pkg):
        for f in files:
            if f.endswith((".py", ".cu", ".cuh", ".h")):
                src = open(os.path.join(dirpath, f)).read()
                assert "import oracle" not in src and "from oracle" not in src, f


def test_launch_chain_rules(lib):
    """One chain per host thread; hla_chain_end needs an open chain (no CUDA call is made)."""
    assert lib.hla_chain_end() == 1
    assert lib.hla_chain_begin(None) == 0
    assert lib.hla_chain_begin(None) == 1
    assert lib.hla_chain_end() == 0
    assert lib.hla_chain_end() == 1
