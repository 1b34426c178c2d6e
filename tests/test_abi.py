"""The C-ABI library builds, loads and exports every declared entry point.
Host-side argument checks that return before any CUDA call are exercised
too; nothing here launches a kernel (CPU only)."""
import ctypes
import os
import re

import pytest

import speculative_decoding_verification_49_gb300 as sv
from speculative_decoding_verification_49_gb300 import build as svbuild

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "spec_verify.h")


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    names = re.findall(r"\b(spec_verify_\w+)\s*\(", text)
    return sorted(set(names))


@pytest.fixture(scope="module")
def lib():
    svbuild.build()
    return sv.load()


def test_header_declares_the_boundary():
    names = declared_functions()
    for want in ("spec_verify_create", "spec_verify_run", "spec_verify_destroy",
                 "spec_verify_run_debug", "spec_verify_get_status", "spec_verify_error_string"):
        assert want in names


def test_every_declared_symbol_is_exported(lib):
    for name in declared_functions():
        assert hasattr(lib, name), name
    assert sorted(sv.exported_names()) == declared_functions()


def test_error_strings(lib):
    for code in range(11):
        s = sv.spec_verify_error_string(code)
        assert s.startswith("SV_")
    assert "unknown" in sv.spec_verify_error_string(99)


def test_host_validation_without_gpu(lib):
    ctx = ctypes.c_void_p(123)
    # unsupported vocabulary: 1001 bf16 logits are not a whole number of 16-byte vectors
    assert lib.spec_verify_create(ctypes.byref(ctx), 0, 4, 3, 1001, sv.SV_BF16) == sv.SV_ERR_SHAPE
    assert ctx.value is None
    assert lib.spec_verify_create(ctypes.byref(ctx), 0, 4, 3, 1002, sv.SV_F32) == sv.SV_ERR_SHAPE
    assert lib.spec_verify_create(ctypes.byref(ctx), 0, 4, 3, 0, sv.SV_F32) == sv.SV_ERR_SHAPE
    assert lib.spec_verify_create(ctypes.byref(ctx), 0, 4, 3, 1024, 7) == sv.SV_ERR_DTYPE
    assert lib.spec_verify_create(ctypes.byref(ctx), 0, -1, 3, 1024, sv.SV_F32) == sv.SV_ERR_INVALID_ARG
    assert lib.spec_verify_create(None, 0, 4, 3, 1024, sv.SV_F32) == sv.SV_ERR_INVALID_ARG
    # a NULL context is rejected before anything is enqueued
    assert sv.spec_verify_run(None, 16, 16, 16, 16, 16, 0, 1, 1, 16, 16, None) == sv.SV_ERR_INVALID_ARG
    assert sv.spec_verify_get_status(None) == sv.SV_ERR_INVALID_ARG
    assert sv.spec_verify_set_cluster_size(None, 2) == sv.SV_ERR_INVALID_ARG
    st, _ = sv.spec_verify_acceptance_counts(None, 8)
    assert st == sv.SV_ERR_INVALID_ARG
    sv.spec_verify_destroy(None)


def test_tree_run_host_validation_without_gpu(lib):
    tr = sv.spec_verify_tree_run
    args = (16, 16, 16, 16, 16, 16, 0, 2, 3, 16, 16, 16, None, None, None, None)
    assert tr(None, *args) == sv.SV_ERR_INVALID_ARG  # no context: rejected before any CUDA call


def test_fused_and_lm_head_host_validation_without_gpu(lib):
    fr = lib.spec_verify_run_fused
    args = (16, 16, 64, 16, 16, 64, 16, 16, 16, 0, 2, 3, 16, 16, None, None, None, None)
    assert fr(None, *args) == sv.SV_ERR_INVALID_ARG  # no context
    lm = lib.spec_verify_lm_head_logits
    assert lm(16, 16, 4, 8, 12, 16, None) == sv.SV_ERR_INVALID_ARG   # K not a multiple of 8
    assert lm(16, 16, -1, 8, 16, 16, None) == sv.SV_ERR_INVALID_ARG  # negative rows
    assert lm(24, 16, 4, 8, 16, 16, None) == sv.SV_ERR_INVALID_ARG   # misaligned hidden states
    assert lm(16, 16, 0, 8, 16, 16, None) == sv.SV_OK                # nothing to do


def test_selftest_timeout_host_validation_without_gpu(lib):
    flag = ctypes.c_int(7)
    assert lib.spec_verify_selftest_timeout(0, ctypes.byref(flag), None) == sv.SV_ERR_INVALID_ARG
    assert lib.spec_verify_selftest_timeout(10 ** 8, ctypes.byref(flag), None) == sv.SV_ERR_INVALID_ARG
    assert lib.spec_verify_selftest_timeout(1000, None, None) == sv.SV_ERR_INVALID_ARG


def test_kv_commit_host_validation_without_gpu(lib):
    kv = sv.spec_verify_kv_commit
    ok = (256, 512, 1024, 2048, None)  # scratch, cache, cache_len, num_accepted, status
    assert kv(*ok, 2, 4, 5, 16, 0, None) == sv.SV_ERR_INVALID_ARG      # row_bytes 0
    assert kv(*ok, 2, 4, 5, 16, 24, None) == sv.SV_ERR_INVALID_ARG     # not a multiple of 16
    assert kv(*ok, 0, 4, 5, 16, 32, None) == sv.SV_ERR_INVALID_ARG     # no planes
    assert kv(*ok, 2, -1, 5, 16, 32, None) == sv.SV_ERR_INVALID_ARG
    assert kv(*ok, 2, 4, -1, 16, 32, None) == sv.SV_ERR_INVALID_ARG
    assert kv(*ok, 2, 4, 5, -1, 32, None) == sv.SV_ERR_INVALID_ARG
    assert kv(264, 512, 1024, 2048, None, 2, 4, 5, 16, 32, None) == sv.SV_ERR_INVALID_ARG  # misaligned
    assert kv(256, 520, 1024, 2048, None, 2, 4, 5, 16, 32, None) == sv.SV_ERR_INVALID_ARG
    assert kv(None, 512, 1024, 2048, None, 2, 4, 5, 16, 32, None) == sv.SV_ERR_INVALID_ARG
    assert kv(256, 512, None, 2048, None, 2, 4, 5, 16, 32, None) == sv.SV_ERR_INVALID_ARG
    assert kv(*ok, 1 << 20, 1 << 20, 5, 1 << 20, 1 << 20, None) == sv.SV_ERR_TOO_LARGE
    assert kv(*ok, 2, 0, 5, 16, 32, None) == sv.SV_OK                  # no sequences: nothing to do


def test_library_is_built_for_sm_103a():
    assert "arch=compute_103a,code=sm_103a" in svbuild.NVCC_FLAGS


def test_header_is_plain_c(tmp_path):
    """A C99 caller of every entry point compiles against the header (gcc)."""
    import shutil
    import subprocess
    gcc = shutil.which("gcc")
    if gcc is None:
        pytest.skip("gcc not available")
    here = os.path.dirname(os.path.abspath(__file__))
    root = os.path.dirname(here)
    src = os.path.join(here, "c", "abi_usage.c")
    r = subprocess.run([gcc, "-std=c99", "-Wall", "-Wextra", "-Werror", "-pedantic", "-c", src,
                        "-I", os.path.join(root, "include"), "-o", str(tmp_path / "abi_usage.o")],
                       capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
    # every declared function is called by the example
    text = open(src).read()
    for name in declared_functions():
        assert name + "(" in text, name
