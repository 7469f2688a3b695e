"""Host-side checks of libmoe_expand.so that need no GPU: it builds, loads,
exports every function include/moe_expand.h declares, and its host helpers
(capacity bound, workspace size, argument validation) behave."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def capi():
    from expanded_layout_expert_gb300 import build, _capi
    build.build()
    return _capi


def _declared_functions():
    text = open(os.path.join(ROOT, "include", "moe_expand.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(moe_[a-z0-9_]+)\s*\(", text)))


def test_header_and_binding_agree(capi):
    declared = _declared_functions()
    assert len(declared) >= 10
    assert set(declared) == set(capi.SIGNATURES), set(declared) ^ set(capi.SIGNATURES)


def test_library_exports_every_declared_symbol(capi):
    lib = ctypes.CDLL(capi.library_path())
    for name in _declared_functions():
        assert hasattr(lib, name), name


def test_capacity_matches_oracle(capi, orc):
    lib = capi.load()
    for T, K, E, a in [(64, 2, 8, 32), (4096, 8, 32, 128), (16384, 8, 32, 128), (8192, 8, 64, 128),
                       (32768, 8, 32, 128), (0, 4, 8, 128), (3, 1, 16, 4), (5, 3, 2, 1)]:
        assert lib.moe_expanded_capacity(T, K, E, a) == orc.expanded_capacity(T * K, E, a)
    assert lib.moe_expanded_capacity(-1, 2, 8, 32) == -1
    assert lib.moe_expanded_capacity(4, 2, 0, 32) == -1


def test_workspace_size(capi):
    lib = capi.load()
    assert lib.moe_workspace_size(16384, 8, 32) >= 2 * 32 * 64 * 4 + 4
    assert lib.moe_workspace_size(16384, 8, 32) % 256 == 0
    assert lib.moe_workspace_size(0, 8, 32) > 0
    assert lib.moe_workspace_size(-1, 8, 32) == 0


def test_argument_validation_without_a_device(capi):
    lib = capi.load()
    # null outputs and bad shapes are rejected before any CUDA call
    assert lib.moe_expand_layout(None, 4, 2, 8, 32, None, 64, None, None, None, None, None, None,
                                 None, 0, None, None) == capi.MOE_ERR_INVALID_ARG
    assert b"null" in lib.moe_last_error_string()
    assert lib.moe_grouped_gemm(None, None, 0, 0, None, None, None, None, None, None, 0, 8, 256,
                                512, 128, None, None, None) == capi.MOE_ERR_INVALID_ARG
    assert lib.moe_combine(None, None, None, None, 4, 100, 2, None, None) == capi.MOE_ERR_INVALID_ARG
    assert lib.moe_act_quant(None, 256, None, 0, 0, None, 16, None, None, 2, None,
                             None) == capi.MOE_ERR_INVALID_ARG
    # the fused layout + scatter: null outputs, then H not a multiple of 128
    assert lib.moe_expand_layout_scatter(None, None, None, None, 0, 4, 4, 512, 2, 8, 32, None, 64,
                                         None, None, None, None, None, None, None, None, 4, None,
                                         None, 0, None, None) == capi.MOE_ERR_INVALID_ARG
    buf = (ctypes.c_int32 * 4096)()
    p = ctypes.cast(buf, ctypes.c_void_p).value
    assert lib.moe_expand_layout_scatter(p, p, p, p, 0, 4, 4, 500, 2, 8, 32, None, 64, p, p, p, p,
                                         p, p, p, p, 4, p, p, 4096, None,
                                         None) == capi.MOE_ERR_INVALID_ARG
    assert b"multiple of 128" in lib.moe_last_error_string()


def test_product_package_does_not_import_the_oracle():
    pkg = os.path.join(ROOT, "expanded_layout_expert_gb300")
    for dirpath, _, files in os.walk(pkg):
        for f in files:
            if f.endswith((".py", ".cu", ".cuh", ".h")):
                src = open(os.path.join(dirpath, f)).read()
                assert "import oracle" not in src and "from oracle" not in src, f
                assert "moe_oracle" not in src, f


def test_noalloc_scratch_limit(capi):
    """moe_expand_layout_noalloc's fixed array holds floor((2^20 - 256) / 8E)
    chunks of 2048 pairs; one pair more is refused before any device work."""
    lib = capi.load()
    cap = lib.moe_expand_layout_noalloc_max_scratch()
    assert cap == 1 << 20
    buf = (ctypes.c_int32 * 16)()
    p = ctypes.cast(buf, ctypes.c_void_p).value
    for E, nb_max in ((32, 4095), (1024, 127)):
        assert nb_max == (cap - 256) // (8 * E)
        assert lib.moe_workspace_size(nb_max * 2048, 1, E) <= cap
        assert lib.moe_workspace_size(nb_max * 2048 + 1, 1, E) > cap
        rc = lib.moe_expand_layout_noalloc(p, nb_max * 2048 + 1, 1, E, 128, None, 64, p, p, p, p,
                                           p, p, None, None)
        assert rc == capi.MOE_ERR_INVALID_ARG
        assert b"scratch" in lib.moe_last_error_string()
