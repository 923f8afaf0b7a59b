"""The C ABI without a GPU: the library loads, exports every symbol include/svd.h declares,
names its error codes, sizes the native layout and rejects bad arguments before touching CUDA.
Also checks that the product package never reaches into the oracle."""
import ctypes
import os
import re

import pytest

from speculative_decoding_verify_06_gb300 import build, svd

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "svd.h")


@pytest.fixture(scope="module")
def lib():
    build.build_library()
    return svd.load()


def declared_functions():
    src = open(HEADER).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(svd_[a-z_0-9]+)\s*\(", src)))


def test_header_and_binding_agree():
    assert declared_functions() == sorted(svd.EXPORTS)


def test_library_exports_every_declared_symbol(lib):
    for name in declared_functions():
        assert hasattr(lib, name), name


def test_error_strings(lib):
    for code in (0, -1, -2, -3, -4):
        assert svd.svd_error_string(code).startswith("SVD_")
    assert "unknown" in svd.svd_error_string(7)


def test_native_sizes(lib):
    cb, sb = svd.svd_native_sizes(5120, 7168)
    assert cb == 7168 * 5120 // 2 and sb == 7168 * 5120 // 32 * 2
    cb, sb = svd.svd_native_sizes(96, 40)  # rows padded to 64, inputs to 64
    assert cb == 64 * 128 // 2 and sb == 64 * 128 // 32 * 2
    with pytest.raises(svd.SvdError):
        svd.svd_native_sizes(100, 64)


def test_q4k_native_sizes(lib):
    # 7168 x 5120: 112 row blocks x 20 super-block columns, 8192 + 1024 bytes each -- the
    # format's own 144 bytes per 256 weights
    cb, hb = svd.svd_q4k_native_sizes(5120, 7168)
    assert (cb, hb) == (112 * 20 * 8192, 112 * 20 * 1024)
    assert cb + hb == 7168 * 5120 // 256 * 144
    cb, hb = svd.svd_q4k_native_sizes(512, 40)  # rows padded to 64
    assert (cb, hb) == (2 * 8192, 2 * 1024)
    for bad in ((480, 64), (0, 64), (256, 0)):
        with pytest.raises(svd.SvdError):
            svd.svd_q4k_native_sizes(*bad)


def test_q4k_arguments_rejected_on_the_host(lib):
    L = lib
    # raw Q4_K: scales must be NULL, in_features % 256 == 0; Q4_K native: headers required
    w = svd._QWeight(16, 16, 512, 64, svd.SVD_LAYOUT_Q4K, 0)
    assert L.svd_verify_linear(ctypes.byref(w), 16, 4, 16, None, 0, 0, None) == svd.SVD_ERR_INVALID_ARG
    w = svd._QWeight(16, None, 480, 64, svd.SVD_LAYOUT_Q4K, 0)
    assert L.svd_verify_linear(ctypes.byref(w), 16, 4, 16, None, 0, 0, None) == svd.SVD_ERR_INVALID_ARG
    w = svd._QWeight(16, None, 512, 64, svd.SVD_LAYOUT_Q4K_NATIVE, 0)
    assert L.svd_verify_linear(ctypes.byref(w), 16, 4, 16, None, 0, 0, None) == svd.SVD_ERR_INVALID_ARG
    w = svd._QWeight(16, 16, 480, 64, svd.SVD_LAYOUT_Q4K_NATIVE, 0)
    assert L.svd_verify_linear(ctypes.byref(w), 16, 4, 16, None, 0, 0, None) == svd.SVD_ERR_INVALID_ARG
    # repack: a Q4_K source with scales, or misaligned destinations
    src = svd._QWeight(16, 16, 512, 64, svd.SVD_LAYOUT_Q4K, 0)
    assert L.svd_repack_weights(ctypes.byref(src), 16, 16, None) == svd.SVD_ERR_INVALID_ARG
    src = svd._QWeight(16, None, 512, 64, svd.SVD_LAYOUT_Q4K, 0)
    assert L.svd_repack_weights(ctypes.byref(src), 8, 16, None) == svd.SVD_ERR_INVALID_ARG


def test_bad_arguments_rejected_on_the_host(lib):
    L = lib
    assert L.svd_verify_linear(None, None, 4, None, None, 0, 0, None) == svd.SVD_ERR_INVALID_ARG
    w = svd._QWeight(16, 16, 64, 64, svd.SVD_LAYOUT_NATIVE, 0)
    assert L.svd_verify_linear(ctypes.byref(w), 16, 0, 16, None, 0, 0, None) == svd.SVD_ERR_INVALID_ARG
    assert L.svd_verify_linear(ctypes.byref(w), 16, 33, 16, None, 0, 0, None) == svd.SVD_ERR_INVALID_ARG
    w_odd = svd._QWeight(16, 16, 48, 64, svd.SVD_LAYOUT_NATIVE, 0)
    assert L.svd_verify_linear(ctypes.byref(w_odd), 16, 4, 16, None, 0, 0, None) == svd.SVD_ERR_INVALID_ARG
    w_mis = svd._QWeight(8, 16, 64, 64, svd.SVD_LAYOUT_NATIVE, 0)
    assert L.svd_verify_linear(ctypes.byref(w_mis), 16, 4, 16, None, 0, 0, None) == svd.SVD_ERR_INVALID_ARG
    # acceptance: k out of range, V out of range; zero windows is a no-op
    args = (16, None, 16, None, None, 16)
    assert L.svd_accept(*args, 10, 0, 100, 0, 0, None, 16, 16, 16, None) == svd.SVD_ERR_INVALID_ARG
    assert L.svd_accept(*args, 10, 33, 100, 0, 0, None, 16, 16, 16, None) == svd.SVD_ERR_INVALID_ARG
    assert L.svd_accept(*args, 10, 3, 0, 0, 0, None, 16, 16, 16, None) == svd.SVD_ERR_INVALID_ARG
    assert L.svd_accept(*args, 0, 3, 100, 0, 0, None, 16, 16, 16, None) == svd.SVD_OK
    # sampler: bad temperature, bad top_p, aliasing
    bad = svd._Sampler(0.0, 0.9, 0.05, 0)
    assert L.svd_sampler_probs(16, 2, 100, ctypes.byref(bad), 32, None, 64, 1 << 20, None) == svd.SVD_ERR_INVALID_ARG
    bad = svd._Sampler(0.6, 1.5, 0.05, 0)
    assert L.svd_sampler_probs(16, 2, 100, ctypes.byref(bad), 32, None, 64, 1 << 20, None) == svd.SVD_ERR_INVALID_ARG
    ok = svd._Sampler(0.6, 0.9, 0.05, 0)
    assert L.svd_sampler_probs(16, 2, 100, ctypes.byref(ok), 16, None, 64, 1 << 20, None) == svd.SVD_ERR_INVALID_ARG
    assert L.svd_sampler_probs(16, 2, 100, ctypes.byref(ok), 32, None, None, 0, None) == svd.SVD_ERR_WORKSPACE
    assert L.svd_graph_begin(None) == svd.SVD_ERR_INVALID_ARG


def test_product_never_imports_the_oracle():
    pkg = os.path.join(ROOT, "speculative_decoding_verify_06_gb300")
    for dirpath, _, files in os.walk(pkg):
        for f in files:
            if f.endswith((".py", ".cu", ".cuh", ".h")):
                src = open(os.path.join(dirpath, f)).read()
                assert not re.search(r"^\s*(import|from)\s+oracle\b", src, re.M), f
                assert "orc.c" not in src and "liborc" not in src, f
