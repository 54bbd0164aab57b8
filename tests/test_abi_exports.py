"""The C-ABI library loads and exports every function include/pagedattn.h and
include/pagedattn_test.h declare; host-only entry points answer without a
GPU; the test hooks stay out of the production header."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "pagedattn.h")
TEST_HEADER = os.path.join(ROOT, "include", "pagedattn_test.h")


def _declared(path=HEADER):
    text = open(path).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(pa_[a-z_0-9]+)\s*\(", text)))


@pytest.fixture(scope="module")
def lib():
    from paged_kv_attention_06_gb300 import build
    path = build.build()
    return ctypes.CDLL(path)


def test_header_declares_the_entry_points():
    names = _declared()
    for must in ("pa_append_kv", "pa_decode", "pa_prefill", "pa_attention",
                 "pa_decode_workspace_bytes", "pa_get_device_error", "pa_status_string"):
        assert must in names


def test_every_declared_symbol_is_exported(lib):
    for name in _declared() + _declared(TEST_HEADER):
        assert hasattr(lib, name), f"{name} declared but not exported"


def test_test_hooks_only_in_the_test_header():
    """Production callers see no kernel-selection switch or injected wait."""
    hooks = _declared(TEST_HEADER)
    assert hooks == ["pa_debug_arm_wait_timeout", "pa_debug_prefill_variant"]
    assert not [n for n in _declared() if n.startswith("pa_debug")]


def test_status_strings(lib):
    lib.pa_status_string.restype = ctypes.c_char_p
    lib.pa_status_string.argtypes = [ctypes.c_int]
    for code in range(7):
        assert lib.pa_status_string(code).decode().startswith("PA_")
    lib.pa_version.restype = ctypes.c_char_p
    assert lib.pa_version().decode().count(".") == 2


class Shape(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int32) for n in
                ("batch", "num_q_heads", "num_kv_heads", "head_dim", "q_len", "num_pages",
                 "max_pages")]


def test_dispatch_route_rule(lib):
    """Short queries take the decode schedule, long ones the prefill one
    (Week 3 Day 4, "Choose a Schedule for Each Query Shape"), with the
    GB300 thresholds: L <= 24, or L <= 32 when max_context_len >= 3072,
    whatever the group size."""
    lib.pa_attention_route.argtypes = [Shape, ctypes.c_int32]
    lib.pa_attention_route.restype = ctypes.c_int32
    for H_kv in (2, 4, 8):     # G = 4, 2, 1
        for L in range(1, 25):
            assert lib.pa_attention_route(Shape(2, 8, H_kv, 128, L, 16, 4), 1024) == 0
        for L in range(25, 33):
            assert lib.pa_attention_route(Shape(2, 8, H_kv, 128, L, 16, 4), 4096) == 0
            assert lib.pa_attention_route(Shape(2, 8, H_kv, 128, L, 16, 4), 3072) == 0
            assert lib.pa_attention_route(Shape(2, 8, H_kv, 128, L, 16, 4), 3071) == 1
            assert lib.pa_attention_route(Shape(2, 8, H_kv, 128, L, 16, 4), 0) == 1
        for L in (33, 48, 64, 512):
            assert lib.pa_attention_route(Shape(2, 8, H_kv, 128, L, 16, 4), 1 << 20) == 1
    assert lib.pa_attention_route(Shape(2, 8, 2, 128, 0, 16, 4), 0) == -1
    assert lib.pa_attention_route(Shape(2, 8, 0, 128, 4, 16, 4), 0) == -1
