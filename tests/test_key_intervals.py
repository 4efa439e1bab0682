"""Key intervals (MARBLE post, section 03: each key's visible queries form one range, so a
partial tile tests lo_k <= pos_q < hi_k): the planner's intervals and block flags against
the oracle, and attention with the interval test bit-identical to attention with the
four-track predicate."""
import numpy as np
import pytest
import torch

import workloads as wl
from oracle import plan as oplan

pytestmark = pytest.mark.gpu
INF = wl.WINDOW_INF


def _single_runs(tr):
    """True if every segment id and noise id forms one run of consecutive tokens."""
    for key in ("seg", "noise"):
        t = np.asarray(tr[key])
        starts = t[np.r_[True, t[1:] != t[:-1]]]
        starts = starts[starts >= 0]
        if len(np.unique(starts)) != len(starts):
            return False
    return True


def _check_intervals(tr, W, P, order, chunk=0):
    """The planner flags a block only when every key's segment and noise span are single
    runs, a sufficient condition for exactness: every flagged block must be exact in the
    oracle with the oracle's intervals (soundness), and without multi-run segments the flags
    must be the oracle's (completeness)."""
    from marble_testlib import make_plan
    pl = make_plan(tr, W, P, order, chunk)
    lo, hi, ex = oplan.key_intervals(tr, W)
    perm = pl.export("perm").cpu().numpy()
    kiv = pl.export("key_intervals").cpu().numpy().reshape(2, -1)
    ivb = pl.export("interval_blocks").cpu().numpy().astype(bool)
    bperm = pl.export("block_perm").cpu().numpy()
    oivb = oplan.interval_blocks(ex)[bperm]
    assert not (ivb & ~oivb).any()
    flagged = np.repeat(ivb, 128)          # tokens of flagged blocks, new order
    assert (kiv[0][flagged] == lo[perm][flagged]).all()
    assert (kiv[1][flagged] == hi[perm][flagged]).all()
    if _single_runs(tr):
        assert (ivb == oivb).all()
        e = ex[perm]
        assert (kiv[0][e] == lo[perm][e]).all() and (kiv[1][e] == hi[perm][e]).all()
    return pl, ivb


@pytest.mark.parametrize("seed", range(6))
def test_intervals_match_oracle_on_random_packs(seed):
    rng = np.random.default_rng(300 + seed)
    n = 128 * int(rng.choice([8, 16, 32]))
    tr = wl.random_pack(rng, n, max_samples=int(rng.integers(1, 6)))
    W = int(rng.choice([INF, 0, 1, 77, 400]))
    P = int(rng.choice([1, 2, 4]))
    order = ["contiguous", "ptrr_block", "ptrr_chunk"][seed % 3]
    _check_intervals(tr, W, P, order, chunk=(n // (2 * P)) // 128 * 128 or 128)


@pytest.mark.parametrize("cid", [2, 3, 5])
def test_intervals_match_oracle_on_configs(cid):
    cfg = wl.mini_config(cid, 8192)
    tr = wl.config_tracks(cid, cfg.n)
    _, ivb = _check_intervals(tr, cfg.window, cfg.shards, cfg.order, cfg.chunk_tokens)
    if cid in (2, 3):
        assert ivb.all()       # no image groups: every key's visible queries are one range


@pytest.mark.parametrize("cid", [2, 5])
def test_attention_with_intervals_equals_predicate(cid):
    from marble_testlib import device_tracks, run_backward, run_forward
    import context_attention_metadata_gb300 as M
    cfg = wl.mini_config(cid, 8192, hq=2)
    tr = wl.config_tracks(cid, cfg.n)
    q, k, v, do = wl.make_qkvdo(cfg.n, cfg.hq, cfg.hkv, cfg.d, device="cuda", seed=cid)
    s, g, z = device_tracks(tr)
    out = []
    for iv in (True, False):
        pl = M.Plan(s, g, z, cfg.window, cfg.shards, cfg.order, cfg.chunk_tokens,
                    key_intervals=iv)
        assert pl.export("interval_blocks").any().item() == iv
        O, L, _ = run_forward(pl, q, k, v)
        dq, dk, dv = run_backward(pl, q, k, v, do)
        out.append((O, L, dq, dk, dv))
    for a, b in zip(*out):
        assert torch.equal(a, b)


def _layout_tracks(cid, n):
    tr = wl.config_tracks(cid, n)
    perm = oplan.vision_group_layout(tr)
    return oplan.apply_layout(tr, perm)


@pytest.mark.parametrize("cid,n,order", [(7, 16384, "ptrr_block"), (5, 16384, "contiguous"),
                                         (2, 8192, "ptrr_block")])
def test_intervals_on_layout_packs(cid, n, order):
    """Packs in the vision-group layout, every token carrying its original position (MARBLE
    s04 "Layout transforms"): each flagged block's keys have exactly the oracle's intervals
    (indices of the given order) and are exact in the oracle; on the video-group pack, whose
    groups the layout turns into single ranges, almost every block is flagged."""
    from marble_testlib import device_tracks
    import context_attention_metadata_gb300 as M
    trp = _layout_tracks(cid, n)
    s_, g_, z_ = device_tracks(trp)
    pos = torch.as_tensor(np.asarray(trp["pos"], np.int32)).cuda()
    pl = M.Plan(s_, g_, z_, INF, 4, order, pos=pos)
    lo, hi, ex = oplan.key_intervals(trp, INF)
    perm = pl.export("perm").cpu().numpy()
    kiv = pl.export("key_intervals").cpu().numpy().reshape(2, -1)
    ivb = pl.export("interval_blocks").cpu().numpy().astype(bool)
    oivb = oplan.interval_blocks(ex)[pl.export("block_perm").cpu().numpy()]
    assert not (ivb & ~oivb).any()                      # sound
    flagged = np.repeat(ivb, 128)
    assert (kiv[0][flagged] == lo[perm][flagged]).all()
    assert (kiv[1][flagged] == hi[perm][flagged]).all()
    print(f"flagged {ivb.mean():.3f} of blocks, oracle-exact {oivb.mean():.3f}")
    if cid == 7:
        assert ivb.sum() >= 0.9 * oivb.sum()
    # with a window the position track switches the interval test off
    plw = M.Plan(s_, g_, z_, 300, 4, order, pos=pos)
    assert not plw.export("interval_blocks").any().item()


def test_intervals_reject_positions_that_are_not_a_permutation():
    """Duplicate positions (not a permutation of the indices): no block is flagged, the plan
    still works through the four-track predicate."""
    from marble_testlib import device_tracks
    import context_attention_metadata_gb300 as M
    trp = _layout_tracks(7, 4096)
    pos = np.asarray(trp["pos"], np.int32).copy()
    pos[10] = pos[11]
    s_, g_, z_ = device_tracks(trp)
    pl = M.Plan(s_, g_, z_, INF, 2, "contiguous", pos=torch.as_tensor(pos).cuda())
    assert not pl.export("interval_blocks").any().item()


@pytest.mark.parametrize("cid", [7, 5])
def test_attention_on_layout_with_intervals_equals_predicate(cid):
    """Attention on a layout pack with the interval test is bit-identical to attention with
    the four-track predicate on every partial tile (forward and backward)."""
    from marble_testlib import device_tracks, run_backward, run_forward
    import context_attention_metadata_gb300 as M
    n = 16384 if cid == 5 else 8192
    cfg = wl.mini_config(cid, n, hq=2)
    trp = _layout_tracks(cid, n)
    q, k, v, do = wl.make_qkvdo(n, cfg.hq, cfg.hkv, cfg.d, device="cuda", seed=cid)
    s_, g_, z_ = device_tracks(trp)
    pos = torch.as_tensor(np.asarray(trp["pos"], np.int32)).cuda()
    out = []
    for iv in (True, False):
        pl = M.Plan(s_, g_, z_, INF, cfg.shards, "ptrr_block", key_intervals=iv, pos=pos)
        assert pl.export("interval_blocks").any().item() == iv
        O, L, _ = run_forward(pl, q, k, v)
        dq, dk, dv = run_backward(pl, q, k, v, do)
        out.append((O, L, dq, dk, dv))
    for a, b in zip(*out):
        assert torch.equal(a, b)
