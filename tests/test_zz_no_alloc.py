"""The tile map built without allocation (marble_tile_map_static) equals the one built by
marble_plan.

marble_tile_map_static is for callers that cannot call cudaMalloc.  One example is a
planner that runs for every packed batch on a side stream while the previous step still
trains, and cannot take the device-wide synchronisation cudaMalloc may cause.  Another is
a process whose device memory belongs to another allocator or a fixed budget.  The call
keeps its scratch in a fixed array inside the library, and writes only into the buffers
the caller passes.  These tests call it through the C ABI twice in a row (the second call
finds the first call's leftovers in the shared scratch) and compare its output with the
plan's exported tile map, which integer data must match exactly.  This file is named so
that pytest collects it last.
"""
import numpy as np
import pytest
import torch

import context_attention_metadata_gb300 as M
import workloads as wl
from marble_testlib import device_tracks, make_plan

pytestmark = pytest.mark.gpu
INF = wl.WINDOW_INF


def _static_map(tr, W, capacity=None):
    s, g, z = device_tracks(tr)
    n = s.shape[0]
    nb = n // M.BLOCK
    row_ptr = torch.full((nb + 1,), -7, dtype=torch.int64, device="cuda")
    cap = capacity if capacity is not None else nb * nb
    col = torch.full((cap,), -7, dtype=torch.int32, device="cuda")
    tag = torch.full((cap,), 99, dtype=torch.uint8, device="cuda")
    M.tile_map_static(s, g, z, W, row_ptr, col, tag)
    torch.cuda.synchronize()
    return row_ptr.cpu().numpy(), col.cpu().numpy(), tag.cpu().numpy()


def _plan_map(tr, W):
    pl = make_plan(tr, W, 1)
    out = (pl.export("tile_rowptr").cpu().numpy(), pl.export("tile_col").cpu().numpy(),
           pl.export("tile_tag").cpu().numpy())
    pl.close()
    return out


@pytest.mark.parametrize("case", ["config2", "config3", "random"])
def test_static_tile_map_matches_plan_twice(case):
    if case == "config2":
        tr, W = wl.config_tracks(2), INF
    elif case == "config3":
        tr, W = wl.config_tracks(3), 4096
    else:
        tr, W = wl.random_pack(np.random.default_rng(77), 128 * 40, max_samples=5), 300
    rp, col, tag = _plan_map(tr, W)
    nnz = int(rp[-1])
    for _ in range(2):
        srp, scol, stag = _static_map(tr, W)
        assert (srp == rp).all()
        assert (scol[:nnz] == col).all()
        assert (stag[:nnz] == tag).all()
        assert (scol[nnz:] == -7).all() and (stag[nnz:] == 99).all()


def test_static_tile_map_short_buffer_and_bad_metadata():
    tr = wl.config_tracks(1)
    rp, col, tag = _plan_map(tr, INF)
    srp, scol, stag = _static_map(tr, INF, capacity=50)
    assert (srp == rp).all() and int(srp[-1]) == 88
    assert (scol == col[:50]).all() and (stag == tag[:50]).all()
    bad = dict(tr)
    bad["sample"] = tr["sample"][::-1].copy()  # sample ids must not decrease
    srp, _, _ = _static_map(bad, INF)
    assert srp[0] == -1
    # a good call right after a bad one starts from a cleared validation word
    srp, scol, stag = _static_map(tr, INF)
    assert (srp == rp).all() and (scol[:88] == col).all()


def test_static_tile_map_allocates_nothing():
    """After a first call on the device (which loads the kernels and looks up the scratch
    array's address), repeated calls leave the device's free memory exactly unchanged: the
    entry point takes no memory from the driver, the library's pool or torch."""
    tr, W = wl.config_tracks(2), INF
    s, g, z = device_tracks(tr)
    nb = s.shape[0] // M.BLOCK
    row_ptr = torch.empty((nb + 1,), dtype=torch.int64, device="cuda")
    col = torch.empty((nb * 64,), dtype=torch.int32, device="cuda")
    tag = torch.empty((nb * 64,), dtype=torch.uint8, device="cuda")
    M.tile_map_static(s, g, z, W, row_ptr, col, tag)
    torch.cuda.synchronize()
    free0, _ = torch.cuda.mem_get_info()
    reserved0 = torch.cuda.memory_reserved()
    for _ in range(5):
        M.tile_map_static(s, g, z, W, row_ptr, col, tag)
    torch.cuda.synchronize()
    free1, _ = torch.cuda.mem_get_info()
    assert free1 == free0
    assert torch.cuda.memory_reserved() == reserved0


def test_static_tile_map_rejects_packs_beyond_its_scratch():
    n = M.TILE_MAP_STATIC_MAX_TOKENS + M.BLOCK
    z = torch.zeros(n, dtype=torch.int32, device="cuda")
    rp = torch.zeros(n // M.BLOCK + 1, dtype=torch.int64, device="cuda")
    col = torch.zeros(16, dtype=torch.int32, device="cuda")
    tag = torch.zeros(16, dtype=torch.uint8, device="cuda")
    with pytest.raises(M.MarbleError) as e:
        M.tile_map_static(z, z, z, INF, rp, col, tag)
    assert e.value.status == M.ERR_INVALID_ARG
    assert "MAX_TOKENS" in str(e.value)
