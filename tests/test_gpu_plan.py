"""Planner parity: the CUDA planner's tile map, token order, per-step lists and needed-KV
index are bit-exact against the oracle planner; legal-pair statistics match the oracle's
counters and closed forms."""
import numpy as np
import pytest
import torch

import workloads as wl
from oracle import counts, plan as oplan

pytestmark = pytest.mark.gpu

INF = wl.WINDOW_INF


def _compare(pl, opl):
    ex = lambda f: pl.export(f).cpu().numpy()
    assert (ex("tile_rowptr") == opl.row_ptr).all()
    assert (ex("tile_col") == opl.col).all()
    assert (ex("tile_tag") == opl.tag).all()
    assert (ex("block_perm") == opl.block_perm).all()
    assert (ex("perm") == opl.perm).all()
    trp = ex("tracks_perm").reshape(4, -1)
    for i, k in enumerate(("sample", "seg", "noise", "pos")):
        assert (trp[i] == opl.tracks_perm[k]).all(), k
    assert (ex("step_ptr") == opl.step_ptr).all()
    assert (ex("step_col") == opl.step_col).all()
    assert (ex("step_tag") == opl.step_tag).all()
    assert (ex("colT_ptr") == opl.colT_ptr).all()
    assert (ex("colT_row") == opl.colT_row).all()
    assert (ex("colT_tag") == opl.colT_tag).all()
    assert (ex("needed_ptr") == opl.needed_ptr).all()
    assert (ex("needed") == opl.needed).all()


def _check(tr, W, P, order, chunk=0):
    from marble_testlib import make_plan
    pl = make_plan(tr, W, P, order, chunk)
    opl = oplan.make_plan(tr, W, P, order, chunk)
    _compare(pl, opl)
    return pl, opl


@pytest.mark.parametrize("seed", range(6))
@pytest.mark.parametrize("order", ["contiguous", "ptrr_block", "ptrr_chunk"])
def test_random_packs(seed, order):
    rng = np.random.default_rng(1000 + seed)
    n = 128 * int(rng.choice([8, 16, 48, 96]))
    tr = wl.random_pack(rng, n, max_samples=int(rng.integers(2, 9)))
    P = int(rng.choice([1, 2, 4, 8]))
    W = int(rng.choice([INF, 1, 77, 300, 1000]))
    _check(tr, W, P, order, chunk=(n // (2 * P)) // 128 * 128 or 128)


def test_config1_plan_and_pairs():
    tr = wl.config_tracks(1)
    pl, opl = _check(tr, INF, 4, "contiguous")
    st = pl.stats()
    assert st["n_full"] == 80 and st["n_partial"] == 8 and st["nnz"] == 88
    assert st["legal_pairs"] == 1376768


@pytest.mark.parametrize("cid", [2, 3, 4, 5])
def test_mini_configs(cid):
    cfg = wl.mini_config(cid, 16384)
    tr = wl.config_tracks(cid, cfg.n)
    pl, _ = _check(tr, cfg.window, cfg.shards, cfg.order, cfg.chunk_tokens)
    assert pl.stats()["legal_pairs"] == counts.by_key_classes(tr, cfg.window)


@pytest.mark.parametrize("cid", [2, 3, 4, 5])
def test_full_configs(cid):
    cfg = wl.CONFIGS[cid]
    tr = wl.config_tracks(cid)
    pl, opl = _check(tr, cfg.window, cfg.shards, cfg.order, cfg.chunk_tokens)
    st = pl.stats()
    assert st["legal_pairs"] == counts.by_key_classes(tr, cfg.window)
    if cid == 3:
        assert st["legal_pairs"] == 1065355264
        sizes = np.diff(opl.needed_ptr)
        assert sizes[0] == 128 and (sizes[1:] == 160).all()
    # PTRR balances the q shards
    if cfg.order != "contiguous":
        assert st["shard_cost_max"] <= 1.05 * st["shard_cost_sum"] / cfg.shards


def test_bad_metadata_is_rejected():
    import context_attention_metadata_gb300 as M
    from marble_testlib import make_plan
    tr = wl.config_tracks(1)
    bad = dict(tr)
    bad["sample"] = tr["sample"][::-1].copy()  # decreasing sample ids
    with pytest.raises(M.MarbleError) as e:
        make_plan(bad, INF, 4)
    assert e.value.status == M.ERR_INVALID_ARG
    bad = dict(tr)
    bad["seg"] = tr["seg"].copy()
    bad["seg"][5] = -7
    with pytest.raises(M.MarbleError):
        make_plan(bad, INF, 4)
    with pytest.raises(M.MarbleError):
        make_plan(tr, INF, 3)  # 16 blocks not divisible by 3


def test_bounded_wait_reports_timeout_and_context_survives():
    import context_attention_metadata_gb300 as M
    from marble_testlib import make_plan
    pl = make_plan(wl.config_tracks(1), INF, 4)
    M.debug_wait_timeout(pl, 50_000_000)  # 50 ms, nothing ever arrives
    with pytest.raises(M.MarbleError) as e:
        pl.check()
    assert e.value.status == M.ERR_TIMEOUT
    pl.check()  # the error word was cleared and the context still works
    x = torch.ones(16, device="cuda")
    assert float(x.sum()) == 16.0
