"""The C ABI without a GPU: the library loads, exports every symbol include/mla.h
declares, and rejects bad configurations / arguments on the host before any CUDA call."""
import ctypes
import os
import re
import subprocess

import pytest

from mla_absorbed_latent_decode_gb300 import binding as B
from mla_absorbed_latent_decode_gb300 import build
from tests.conftest import ROOT

HEADER = os.path.join(ROOT, "include", "mla.h")


@pytest.fixture(scope="module")
def lib():
    build.build()
    return B.load()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(mla_[a-z_]+)\s*\(", text)))


def test_header_declares_the_boundary():
    names = declared_functions()
    for n in ("mla_create", "mla_destroy", "mla_kv_append", "mla_decode_workspace_size", "mla_decode",
              "mla_get_status", "mla_last_error"):
        assert n in names
    assert sorted(B.EXPORTED) == names


def test_library_exports_every_declared_symbol(lib):
    out = subprocess.run(["nm", "-D", "--defined-only", build.LIB], capture_output=True, text=True, check=True).stdout
    exported = set(re.findall(r"\bT (mla_\w+)", out))
    for n in declared_functions():
        assert n in exported, n
        assert getattr(lib, n)


def _cfg(**kw):
    base = dict(n_h=16, cache_dtype=B.MLA_CACHE_BF16, max_position=4096)
    base.update(kw)
    return B.make_config(**base)


@pytest.mark.parametrize("field", ["d_c", "d_rope", "n_h", "d_nope", "d_v", "page_size", "cache_dtype",
                                   "max_position", "rope_base"])
def test_missing_field_is_named(lib, field):
    cfg = _cfg()
    setattr(cfg, field, 0)
    h = ctypes.c_void_p()
    s = lib.mla_create(ctypes.byref(cfg), 1, 1, None, ctypes.byref(h))
    assert s == B.MLA_ERR_MISSING_FIELD
    msg = lib.mla_last_error().decode()
    assert field in msg and "mla_config_t" in msg
    assert not h.value


def test_fp8_scale_mandatory_only_for_fp8(lib):
    h = ctypes.c_void_p()
    cfg = _cfg(cache_dtype=B.MLA_CACHE_FP8_E4M3)
    assert lib.mla_create(ctypes.byref(cfg), 1, 1, None, ctypes.byref(h)) == B.MLA_ERR_MISSING_FIELD
    assert "fp8_scale" in lib.mla_last_error().decode()


@pytest.mark.parametrize("kw", [dict(d_c=256), dict(d_rope=32), dict(n_h=129), dict(page_size=32),
                                dict(d_v=64), dict(max_position=(1 << 20) + 1)])
def test_unsupported_shapes(lib, kw):
    cfg = _cfg(**kw)
    h = ctypes.c_void_p()
    assert lib.mla_create(ctypes.byref(cfg), 1, 1, None, ctypes.byref(h)) == B.MLA_ERR_UNSUPPORTED


@pytest.mark.parametrize("kw", [dict(n_h=-4), dict(cache_dtype=7), dict(softmax_scale=-1.0),
                                dict(rope_base=float("inf"))])
def test_invalid_values(lib, kw):
    cfg = _cfg(**kw)
    h = ctypes.c_void_p()
    assert lib.mla_create(ctypes.byref(cfg), 1, 1, None, ctypes.byref(h)) == B.MLA_ERR_INVALID_ARG


def test_null_arguments(lib):
    h = ctypes.c_void_p()
    cfg = _cfg()
    assert lib.mla_create(None, 1, 1, None, ctypes.byref(h)) == B.MLA_ERR_INVALID_ARG
    assert lib.mla_create(ctypes.byref(cfg), 0, 1, None, ctypes.byref(h)) == B.MLA_ERR_INVALID_ARG
    assert lib.mla_create(ctypes.byref(cfg), 1, 1, None, None) == B.MLA_ERR_INVALID_ARG
    assert lib.mla_destroy(None) == B.MLA_OK
    sz = ctypes.c_size_t()
    assert lib.mla_decode_workspace_size(None, 1, 1, ctypes.byref(sz)) == B.MLA_ERR_INVALID_ARG
    assert lib.mla_kv_append(None, 1, 1, 1, 1, 1, 1, 1, 1, 1, None) == B.MLA_ERR_INVALID_ARG
    assert lib.mla_decode(None, 1, 1, 1, 1, 1, 1, 1, 1, 1, 1, 1, None) == B.MLA_ERR_INVALID_ARG
    assert lib.mla_decode_fixed_scratch(None, 1, 1, 1, 1, 1, 1, 1, 1, 1, None) == B.MLA_ERR_INVALID_ARG
    assert lib.mla_get_status(None, None, None) == B.MLA_ERR_INVALID_ARG
    assert lib.mla_set_option(None, 1, 0) == B.MLA_ERR_INVALID_ARG
    n = ctypes.c_int32()
    assert lib.mla_profile_read(None, None, 0, ctypes.byref(n)) == B.MLA_ERR_INVALID_ARG
    assert lib.mla_status_string(B.MLA_ERR_WORKSPACE) == b"MLA_ERR_WORKSPACE"
    assert lib.mla_profile_kernel_name(1) == b"mla_decode_splitkv"
    assert lib.mla_profile_kernel_name(0) == b"mla_q_absorb_plan"
    assert lib.mla_profile_kernel_name(3) == b""
    # the entry points beyond the decode step
    assert lib.mla_kv_project_append(None, 1, 256, 1, 1, 1, 1, 1, 1, 1, 1, 1, None) == B.MLA_ERR_INVALID_ARG
    assert lib.mla_project(None, 1, 1, 256, 1, 16, 1, None) == B.MLA_ERR_INVALID_ARG
    assert lib.mla_rmsnorm(None, 1, 1, 8, 8, 1, 1e-6, 1, 8, None) == B.MLA_ERR_INVALID_ARG
    assert lib.mla_expand_kv(None, 1, 1, 1, None) == B.MLA_ERR_INVALID_ARG
    assert lib.mla_decode_naive_workspace_size(None, 1, 1, ctypes.byref(sz)) == B.MLA_ERR_INVALID_ARG
    assert lib.mla_decode_naive(None, 1, 1, 1, 1, 1, 1, 1, 1, 1, 1, 1, None) == B.MLA_ERR_INVALID_ARG
    assert lib.mla_prefill_workspace_size(None, 1, 1, ctypes.byref(sz)) == B.MLA_ERR_INVALID_ARG
    assert lib.mla_prefill(None, 1, 1, 1, 1, 1, 1, 1, 1, 1, 1, 1, 1, 1, 1, 1, None) == B.MLA_ERR_INVALID_ARG
    assert lib.mla_profile_last_name(None, 0) == b""


def test_valid_config_without_gpu_fails_cleanly(lib):
    """A valid configuration reaches the CUDA calls; with no GPU they fail with MLA_ERR_CUDA."""
    import torch
    if torch.cuda.is_available():
        pytest.skip("a GPU is present")
    cfg = _cfg()
    h = ctypes.c_void_p()
    s = lib.mla_create(ctypes.byref(cfg), 1, 1, None, ctypes.byref(h))
    assert s in (B.MLA_ERR_CUDA, B.MLA_ERR_UNSUPPORTED)
    assert not h.value


def test_header_constants_match_the_binding():
    """Every integer #define of include/mla.h that the binding also names has the same value."""
    import re
    text = open(HEADER).read()
    found = 0
    for name, val in re.findall(r"#define\s+(MLA_\w+)\s+(0x[0-9a-fA-F]+|\d+)u?\b", text):
        if hasattr(B, name):
            assert getattr(B, name) == int(val, 0), name
            found += 1
    assert found >= 7          # the check bits and the options
