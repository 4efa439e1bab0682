"""The C-ABI library builds, loads and exports every symbol include/marble.h declares; its
argument checks that need no GPU reject bad calls.  No compute call is made here."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _declared():
    src = open(os.path.join(ROOT, "include", "marble.h")).read()
    return sorted(set(re.findall(r"^(?:marble_status_t|const char \*)\s*(marble_\w+)\s*\(", src,
                                 re.M)))


@pytest.fixture(scope="module")
def libm():
    from context_attention_metadata_gb300 import _build
    _build.build()
    import context_attention_metadata_gb300 as M
    return M.lib()


def test_header_declares_the_boundary_calls():
    names = _declared()
    for want in ("marble_plan", "marble_attn_step", "marble_attn_finalize", "marble_attn_bwd",
                 "marble_attn_bwd_prep", "marble_plan_stats", "marble_plan_export",
                 "marble_permute", "marble_check", "marble_last_error"):
        assert want in names


def test_library_exports_every_declared_symbol(libm):
    for name in _declared():
        assert hasattr(libm, name), name


def test_binding_covers_every_declared_symbol():
    import context_attention_metadata_gb300 as M
    assert set(_declared()) <= set(M._SIGS)


def test_host_side_argument_checks(libm):
    import context_attention_metadata_gb300 as M
    assert libm.marble_plan(None, None, None) == M.ERR_INVALID_ARG
    assert b"non-null" in libm.marble_last_error()
    assert libm.marble_set_wait_limit_ns(0) == M.ERR_INVALID_ARG
    assert libm.marble_plan_destroy(None) == M.OK
    assert libm.marble_check(None, None) == M.ERR_INVALID_ARG
    assert libm.marble_cast_bf16(None, None, 3, None) == M.ERR_INVALID_ARG
    d = M._PlanDesc(1000, 0, 0, 0, 0, 1, 0, 0)  # not a multiple of 128
    h = ctypes.c_void_p()
    assert libm.marble_plan(ctypes.byref(d), None, ctypes.byref(h)) == M.ERR_INVALID_ARG
    assert b"multiple of 128" in libm.marble_last_error()
    assert b"sm_103a" in libm.marble_version()
    # process-wide settings and host-only entry points
    assert libm.marble_set_side_streams(5) == M.ERR_INVALID_ARG
    assert libm.marble_set_side_streams(-1) == M.ERR_INVALID_ARG
    assert libm.marble_set_side_streams(4) == M.OK
    assert libm.marble_layout_vision_groups(None, None, 4, None) == M.ERR_INVALID_ARG
    assert libm.marble_chunk_layout_search(None, 4, 2, 0, None, None) == M.ERR_INVALID_ARG
    d = M._PlanDesc(1024, 0, 0, 0, 0, 2, 3, 0, -5)  # chunk search with a negative range cost
    assert libm.marble_plan(ctypes.byref(d), None, ctypes.byref(h)) == M.ERR_INVALID_ARG
    assert b"range_cost" in libm.marble_last_error()
    d = M._PlanDesc(1024, 0, 0, 0, 0, 2, 4, 0)      # unknown order
    assert libm.marble_plan(ctypes.byref(d), None, ctypes.byref(h)) == M.ERR_INVALID_ARG
