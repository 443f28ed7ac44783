"""The C-ABI library builds, loads without a GPU and exports every entry point
that include/dflash.h declares. No compute calls are made here."""
import ctypes
import os
import re

import pytest

import block_diffusion_drafter_pass_gb300 as dfl
from block_diffusion_drafter_pass_gb300 import _build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "dflash.h")


def declared_symbols():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(dflash_[a-z0-9_]+)\s*\(", text)))


@pytest.fixture(scope="module")
def lib():
    _build.build()
    return dfl.load_library()


def test_header_declares_the_hot_path():
    syms = declared_symbols()
    for name in ("dflash_create", "dflash_fuse_ctx", "dflash_draft", "dflash_verify", "dflash_destroy"):
        assert name in syms


def test_library_exports_every_declared_symbol(lib):
    missing = [s for s in declared_symbols() if not hasattr(lib, s)]
    assert not missing, missing
    assert sorted(dfl.EXPORTED) == declared_symbols()


def test_struct_layouts_match_the_header(lib):
    # 16 ints + 2 floats; 9 pointers; 5 pointers + 1 pointer
    assert ctypes.sizeof(dfl.dflash_config) == 18 * 4
    assert ctypes.sizeof(dfl.dflash_layer_weights) == 9 * ctypes.sizeof(ctypes.c_void_p)
    assert ctypes.sizeof(dfl.dflash_weights) == 6 * ctypes.sizeof(ctypes.c_void_p)


def test_library_is_built_for_sm103a():
    # nvcc was asked for sm_103a only; the flags are part of the build recipe
    assert "arch=compute_103a,code=sm_103a" in " ".join(_build.ARCH)


def test_create_rejects_bad_config_without_touching_the_gpu(lib):
    cfg = dfl.dflash_config()
    w = dfl.dflash_weights()
    out = ctypes.c_void_p()
    # null layer array: rejected before any CUDA call
    assert lib.dflash_create(ctypes.byref(cfg), ctypes.byref(w), ctypes.byref(out)) == dfl.DFLASH_EINVAL
    assert out.value is None
    assert lib.dflash_last_error(None)


def test_stateless_calls_validate_arguments(lib):
    assert lib.dflash_rows_argmax_bf16(None, 4, 0, None, None) == dfl.DFLASH_EINVAL
    assert lib.dflash_rows_argmax_bf16(None, -1, 8, None, None) == dfl.DFLASH_EINVAL
    assert lib.dflash_debug_gemm(None, None, None, 1, 1, 8, 0, None) == dfl.DFLASH_EINVAL


def test_target_feature_layers_follow_the_oracle(lib):
    """The library's default feature layers (host code) are the oracle's
    reading of the setup table for every depth and count it accepts."""
    from oracle import target_pass
    for L in (5, 8, 12, 28, 36, 40, 64):
        for n in range(1, min(16, L - 3) + 1):
            assert dfl.target_feature_layers(L, n) == target_pass.feature_layers(L, n), (L, n)
    out = (ctypes.c_int32 * 5)()
    assert lib.dflash_target_feature_layers(4, 5, out) == dfl.DFLASH_EINVAL
