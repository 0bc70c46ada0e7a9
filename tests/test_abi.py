"""The C ABI without a GPU: the library builds, loads, exports every symbol
include/fa.h declares, and rejects bad arguments before touching the device."""
from __future__ import annotations

import os
import re
import subprocess

import pytest

import exact_attention_gb300 as fa
from exact_attention_gb300 import _binding, build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "fa.h")


@pytest.fixture(scope="module")
def lib():
    build.build()
    return fa.lib()


def declared_functions():
    src = open(HEADER).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(fa_[a-z_0-9]+)\s*\(", src)))


def test_header_declares_the_binding_exports():
    assert declared_functions() == sorted(_binding.EXPORTS)


def test_library_exports_every_declared_symbol(lib):
    out = subprocess.run(["nm", "-D", "--defined-only", build.LIB], capture_output=True, text=True, check=True).stdout
    exported = set(re.findall(r"\bT (fa_[a-z_0-9]+)\b", out))
    missing = [f for f in declared_functions() if f not in exported]
    assert not missing, f"declared but not exported: {missing}"
    for f in declared_functions():
        assert hasattr(lib, f)


def test_library_has_no_link_time_driver_dependency(lib):
    out = subprocess.run(["ldd", build.LIB], capture_output=True, text=True).stdout
    assert "libcuda.so" not in out and "libtorch" not in out


def test_status_strings(lib):
    for s in range(5):
        assert fa.fa_status_string(s).startswith("FA_")


def test_workspace_sizes(lib):
    assert fa.fa_decode_workspace_bytes(8, 32, 128, 16) == 8 * 32 * 16 * 130 * 4
    assert fa.fa_decode_workspace_bytes(0, 32, 128, 16) == 0
    assert fa.fa_bwd_workspace_bytes(1, 2, 1024) == 2 * 1024 * 4


FAKE = 1 << 20  # a 16-byte aligned non-null address; never dereferenced: validation fails first


@pytest.mark.parametrize("D", [32, 96, 256])
def test_unsupported_head_dim_rejected_before_launch(lib, D):
    s = fa.fa_fwd(FAKE, FAKE, FAKE, FAKE, None, 1, 1, 128, 128, D, 0.1, 0, fa.FA_F16, 0)
    assert s == fa.FA_ERR_UNSUPPORTED
    assert "D=" in fa.fa_last_error_message()
    assert fa.fa_decode(FAKE, FAKE, FAKE, FAKE, FAKE, 1, 1, 128, D, 0.1, 1, fa.FA_BF16, 0) == fa.FA_ERR_UNSUPPORTED


def test_invalid_arguments_rejected_before_launch(lib):
    assert fa.fa_fwd(None, FAKE, FAKE, FAKE, None, 1, 1, 8, 8, 64, 0.1, 0, fa.FA_F16, 0) == fa.FA_ERR_INVALID
    assert "Q is NULL" in fa.fa_last_error_message()
    assert fa.fa_fwd(FAKE + 2, FAKE, FAKE, FAKE, None, 1, 1, 8, 8, 64, 0.1, 0, fa.FA_F16, 0) == fa.FA_ERR_INVALID
    assert fa.fa_fwd(FAKE, FAKE, FAKE, FAKE, None, 1, 1, 8, 0, 64, 0.1, 0, fa.FA_F16, 0) == fa.FA_ERR_INVALID
    assert fa.fa_fwd(FAKE, FAKE, FAKE, FAKE, None, -1, 1, 8, 8, 64, 0.1, 0, fa.FA_F16, 0) == fa.FA_ERR_INVALID
    assert fa.fa_fwd(FAKE, FAKE, FAKE, FAKE, None, 1, 1, 8, 8, 64, 0.1, 0, 7, 0) == fa.FA_ERR_INVALID
    assert fa.fa_fwd(FAKE, FAKE, FAKE, FAKE, None, 1, 1, 8, 8, 64, float("-inf"), 0, fa.FA_F16, 0) == fa.FA_ERR_INVALID
    assert "finite" in fa.fa_last_error_message()
    assert fa.fa_fwd(FAKE, FAKE, FAKE, FAKE, None, 1, 1, 8, 8, 64, float("nan"), 0, fa.FA_F16, 0) == fa.FA_ERR_INVALID
    # B*H*max(M,N) overflowing a 32-bit row index
    assert fa.fa_fwd(FAKE, FAKE, FAKE, FAKE, None, 1 << 16, 1 << 10, 1 << 10, 8, 64, 0.1, 0, fa.FA_F16, 0) == \
        fa.FA_ERR_INVALID
    # decode: n_splits outside [1, N]
    assert fa.fa_decode(FAKE, FAKE, FAKE, FAKE, FAKE, 1, 1, 100, 128, 0.1, 0, fa.FA_BF16, 0) == fa.FA_ERR_INVALID
    assert fa.fa_decode(FAKE, FAKE, FAKE, FAKE, FAKE, 1, 1, 100, 128, 0.1, 101, fa.FA_BF16, 0) == fa.FA_ERR_INVALID
    assert fa.fa_decode(FAKE, FAKE, FAKE, FAKE, None, 1, 1, 100, 128, 0.1, 4, fa.FA_BF16, 0) == fa.FA_ERR_INVALID
    # backward: f32 not supported, missing LSE invalid
    assert fa.fa_bwd(*([FAKE] * 10), 1, 1, 8, 8, 64, 0.1, 0, fa.FA_F32, 0) == fa.FA_ERR_UNSUPPORTED
    args = [FAKE] * 10
    args[5] = None
    assert fa.fa_bwd(*args, 1, 1, 8, 8, 64, 0.1, 0, fa.FA_F16, 0) == fa.FA_ERR_INVALID
    assert fa.fa_set_wait_budget_ns(10) == fa.FA_ERR_INVALID
    assert fa.fa_debug_inject(5) == fa.FA_ERR_INVALID
    assert fa.fa_debug_inject(7) == fa.FA_ERR_INVALID
    assert fa.fa_debug_inject(0) == fa.FA_OK  # cancels nothing pending; host-only
    # host-buffer forward: NULL host buffers, a head dimension it cannot run, bad scale
    assert fa.fa_fwd_host(None, FAKE, FAKE, FAKE, None, FAKE, 1 << 20, 1, 1, 8, 8, 64, 0.1, 0, fa.FA_F16, 0) == \
        fa.FA_ERR_INVALID
    assert fa.fa_fwd_host(FAKE, FAKE, FAKE, FAKE, None, FAKE, 1 << 20, 1, 1, 8, 8, 96, 0.1, 0, fa.FA_F16, 0) == \
        fa.FA_ERR_UNSUPPORTED
    assert fa.fa_fwd_host(FAKE, FAKE, FAKE, FAKE, None, FAKE, 1 << 20, 1, 1, 8, 8, 128, 0.1, 0, fa.FA_F32, 0) == \
        fa.FA_ERR_UNSUPPORTED
    assert fa.fa_fwd_host(FAKE, FAKE, FAKE, FAKE, None, FAKE, 1 << 20, 1, 1, 8, 8, 64, float("inf"), 0, fa.FA_F16,
                          0) == fa.FA_ERR_INVALID
    # FP8 forward: the signs are read 16 bytes at a time, so a misaligned or NULL pointer is refused
    assert fa.fa_fwd_fp8(FAKE, FAKE, FAKE, FAKE, None, FAKE + 1, FAKE, 1 << 24, 1, 1, 8, 8, 64, 0.1, 0, fa.FA_F16,
                         0) == fa.FA_ERR_INVALID
    assert fa.fa_fwd_fp8(FAKE, FAKE, FAKE, FAKE, None, None, FAKE, 1 << 24, 1, 1, 8, 8, 64, 0.1, 0, fa.FA_F16,
                         0) == fa.FA_ERR_INVALID
    # decode with rows: R = 0 invalid, R = 5 unsupported
    assert fa.fa_decode_ex(FAKE, FAKE, FAKE, FAKE, None, FAKE, 1, 1, 0, 100, 128, 0.1, 4, fa.FA_BF16, 0) == \
        fa.FA_ERR_INVALID
    assert fa.fa_decode_ex(FAKE, FAKE, FAKE, FAKE, None, FAKE, 1, 1, 5, 100, 128, 0.1, 4, fa.FA_BF16, 0) == \
        fa.FA_ERR_UNSUPPORTED


def test_empty_problems_are_no_ops(lib):
    # B*H == 0 or M == 0: nothing to compute, nothing launched, pointers unused
    assert fa.fa_fwd(None, None, None, None, None, 0, 4, 8, 8, 64, 0.1, 0, fa.FA_F16, 0) == fa.FA_OK
    assert fa.fa_fwd(None, None, None, None, None, 2, 4, 0, 8, 64, 0.1, 0, fa.FA_F16, 0) == fa.FA_OK
    assert fa.fa_decode(None, None, None, None, None, 0, 4, 8, 64, 0.1, 1, fa.FA_F16, 0) == fa.FA_OK
    assert fa.fa_fwd_host(None, None, None, None, None, None, 0, 0, 4, 8, 8, 64, 0.1, 0, fa.FA_F16, 0) == fa.FA_OK


def test_schedule_controls(lib):
    """fa_set_schedule: valid keys and values are accepted (and reset to automatic), others refused."""
    for key in (fa.FA_SCHED_FWD_SPLIT, fa.FA_SCHED_BWD_SPLIT, fa.FA_SCHED_BWD_PAIR):
        for v in (0, 1, -1):
            assert fa.fa_set_schedule(key, v) == fa.FA_OK
        assert fa.fa_set_schedule(key, 2) == fa.FA_ERR_INVALID
    for v in (1, 8, -1):
        assert fa.fa_set_schedule(fa.FA_SCHED_HOST_CHUNKS, v) == fa.FA_OK
    for v in (0, 9, -2):
        assert fa.fa_set_schedule(fa.FA_SCHED_HOST_CHUNKS, v) == fa.FA_ERR_INVALID
    assert fa.fa_set_schedule(0, 1) == fa.FA_ERR_INVALID
    assert fa.fa_set_schedule(5, 1) == fa.FA_ERR_INVALID
    with fa.schedule(fa.FA_SCHED_FWD_SPLIT, 1):
        pass
