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
    assert libm.marble_permute_cast_bf16(None, None, None, 4, 1, None) == M.ERR_INVALID_ARG
    assert b"plan is null" in libm.marble_last_error()
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


def test_tile_map_static_argument_checks(libm):
    """marble_tile_map_static refuses bad arguments on the host, before any launch: sizes,
    the static scratch's limit, the window, the capacity, null pointers, and pointers that
    are not device memory (host buffers here; no GPU is needed to refuse them)."""
    import numpy as np
    import context_attention_metadata_gb300 as M
    n = 1024
    trk = [np.zeros(n, np.int32) for _ in range(3)]
    rp = np.zeros(n // 128 + 1, np.int64)
    col = np.zeros(64, np.int32)
    tag = np.zeros(64, np.uint8)
    ptr = lambda a: ctypes.c_void_p(a.ctypes.data)
    f = libm.marble_tile_map_static

    def call(n_=n, w=0, cap=64, c=col, t=tag, tracks=trk, r=rp):
        return f(n_, *[ptr(x) for x in tracks], w, ptr(r),
                 ptr(c) if c is not None else None, ptr(t) if t is not None else None, cap,
                 None)

    cases = [
        (dict(n_=1000), b"multiple of 128"),
        (dict(n_=0), b"multiple of 128"),
        (dict(n_=M.TILE_MAP_STATIC_MAX_TOKENS + 128), b"MAX_TOKENS"),
        (dict(w=-1), b"window"),
        (dict(cap=-1), b"capacity"),
        (dict(c=None), b"null"),
        (dict(t=None), b"null"),
        (dict(), b"device memory"),  # host buffers
    ]
    for kw, msg in cases:
        assert call(**kw) == M.ERR_INVALID_ARG, kw
        assert msg in libm.marble_last_error(), (kw, libm.marble_last_error())
    # null col / tag are allowed with capacity 0 (only the row pointers are written); the
    # host track buffers are then what is refused
    assert call(cap=0, c=None, t=None) == M.ERR_INVALID_ARG
    assert b"device memory" in libm.marble_last_error()
