"""Backward parity: dQ, dK, dV from the CUDA backward ring steps (against the final LSE,
fp32 accumulation across steps) against the fp64 oracle's analytic gradients; relative
Frobenius error <= 1e-2.  Dense oracle on small packs, sampled rows/columns at full size."""
import numpy as np
import pytest
import torch

import workloads as wl
from marble_testlib import (TOL_GRAD_REL, make_plan, plan_for, rel_fro, run_backward,
                            spread_tokens, token_shards)
from oracle import attention, mask

pytestmark = pytest.mark.gpu
INF = wl.WINDOW_INF


def _check_dense(tr, W, q, k, v, do, dq, dk, dv):
    rq, rk, rv, _, _ = attention.backward(q, k, v, do, mask.dense_mask(tr, W))
    for name, got, ref in (("dq", dq, rq), ("dk", dk, rk), ("dv", dv, rv)):
        e = rel_fro(got.cpu().double().numpy(), ref)
        assert e <= TOL_GRAD_REL, f"{name} rel err {e}"


def test_config1_backward():
    cfg = wl.CONFIGS[1]
    tr = wl.config_tracks(1)
    q, k, v, do = wl.make_qkvdo(cfg.n, cfg.hq, cfg.hkv, cfg.d, device="cuda")
    pl = plan_for(cfg, tr)
    dq, dk, dv = run_backward(pl, q, k, v, do)
    _check_dense(tr, INF, q, k, v, do, dq, dk, dv)


@pytest.mark.parametrize("seed", range(8))
def test_random_packs_backward(seed):
    rng = np.random.default_rng(700 + seed)
    n = 128 * int(rng.choice([8, 16]))
    tr = wl.random_pack(rng, n, max_samples=int(rng.integers(1, 5)))
    d = int(rng.choice([64, 128]))
    hkv = int(rng.choice([1, 2]))
    hq = hkv * int(rng.choice([1, 2, 4]))
    P = int(rng.choice([1, 2, 4]))
    order = ["contiguous", "ptrr_block", "ptrr_chunk"][seed % 3]
    W = int(rng.choice([INF, 1, 60, 300]))
    q, k, v, do = wl.make_qkvdo(n, hq, hkv, d, device="cuda", seed=seed)
    pl = make_plan(tr, W, P, order, chunk_tokens=128)
    dq, dk, dv = run_backward(pl, q, k, v, do, needed=bool(seed % 2))
    _check_dense(tr, W, q, k, v, do, dq, dk, dv)


def test_fully_masked_rows_backward():
    samples = [[wl.Span("causal", 300), wl.Span("full", 200)], [wl.Span("causal", 12)]]
    tr = wl.tracks_from_samples(samples)
    q, k, v, do = wl.make_qkvdo(512, 2, 1, 128, device="cuda")
    pl = make_plan(tr, 0, 2)
    dq, dk, dv = run_backward(pl, q, k, v, do)
    for g in (dq, dk, dv):
        assert torch.isfinite(g).all()
    assert (dq[:300] == 0).all()
    _check_dense(tr, 0, q, k, v, do, dq, dk, dv)


@pytest.mark.parametrize("cid", [2, 3, 4, 5])
def test_mini_configs_backward(cid):
    cfg = wl.mini_config(cid, 4096, hq=4)
    tr = wl.config_tracks(cid, cfg.n)
    q, k, v, do = wl.make_qkvdo(cfg.n, cfg.hq, cfg.hkv, cfg.d, device="cuda")
    pl = plan_for(cfg, tr)
    dq, dk, dv = run_backward(pl, q, k, v, do, needed=cfg.needed)
    _check_dense(tr, cfg.window, q, k, v, do, dq, dk, dv)


def full_size_samples(cid, tr, shard, P, rng):
    """Rows for the dQ check and key columns for the dK/dV check at full size, with the kv
    heads to check: about 256 of each, spread over every shard of the plan and at block
    edges where the candidates allow.

    The fp64 oracle scores each sampled row against its legal keys and each sampled key
    against its visible queries, whose own rows it also needs; the candidates are
    restricted so that this stays within seconds:
      rows:    whole samples of at most 4096 tokens, the first 1024 tokens of every longer
               sample (a causal prefix, or the start of an image, sees at most its own span
               and the tokens before it) -- in the chunked 1M pack this takes rows inside
               the 512K causal generation;
      columns: whole samples of at most 1024 tokens and the last 128-token block of every
               longer sample (seen by the few queries after it) -- the last block of the
               512K causal generation in the 1M pack; in the grouped-image pack also 32 keys
               inside the first image of the shortest sample with a group (seen by the
               whole group), on kv head 0;
      window:  with the 4096-token window every token has at most 4096 partners, so any
               row qualifies, and the columns are two clusters of 128 keys around two shard
               boundaries (keys at the end of a shard are the remote blocks the next shard
               fetches), checked on every kv head."""
    st, en = mask.sample_runs(tr)
    n = len(st)
    idx = np.arange(n)
    L = en - st
    if cid == 3:
        rows = spread_tokens(idx, shard, P, 256, rng)
        bps = n // P
        cols = np.concatenate([np.arange(j * bps - 64, j * bps + 64) for j in (P // 4, 3 * P // 4)])
        return rows, cols, None
    rows = spread_tokens(idx[(L <= 4096) | (idx - st < 1024)], shard, P, 256, rng)
    cand = idx[(L <= 1024) | (en - idx <= 128)]
    cols = spread_tokens(cand, shard, P, 256, rng)
    if cid == 5:
        seg = np.asarray(tr["seg"])
        grouped = [a for a in np.unique(st) if
                   len(np.flatnonzero(np.diff(seg[a:en[a]]) != 0)) >= 3 and
                   np.bincount(seg[a:en[a]][seg[a:en[a]] >= 0]).max(initial=0) > 4096]
        a = min(grouped, key=lambda a_: en[a_] - a_)
        first_img = a + int(np.flatnonzero(seg[a:en[a]] >= 0)[0])
        e = (first_img // 128 + 2) * 128
        cols = np.union1d(cols, np.arange(e - 16, e + 16))
        return rows, cols, np.array([0])  # the group's keys are seen by ~15K queries each
    return rows, cols, np.array([0, -1])


@pytest.mark.parametrize("cid", [2, 3, 4, 5])
def test_full_configs_backward_sampled(cid):
    """dQ on ~256 rows (every q head) and dK/dV on ~256 key columns over every shard of the
    plan, against the fp64 oracle's exact gradients of those rows and columns."""
    cfg = wl.CONFIGS[cid]
    tr = wl.config_tracks(cid)
    q, k, v, do = wl.make_qkvdo(cfg.n, cfg.hq, cfg.hkv, cfg.d, device="cuda")
    pl = plan_for(cfg, tr)
    dq, dk, dv = run_backward(pl, q, k, v, do, needed=cfg.needed)
    for g in (dq, dk, dv):
        assert torch.isfinite(g).all()
    rng = np.random.default_rng(10 + cid)
    rows, cols, kvh = full_size_samples(cid, tr, token_shards(pl), cfg.shards, rng)
    kvh = np.arange(cfg.hkv) if kvh is None else np.unique(kvh % cfg.hkv)
    qc, kc, vc, dc = (t.cpu() for t in (q, k, v, do))
    ref = attention.rows_dq(qc, kc, vc, dc, tr, cfg.window, rows)
    got = dq[torch.as_tensor(rows).cuda()].cpu().double().numpy()
    assert rel_fro(got, ref) <= TOL_GRAD_REL
    rk, rv = attention.cols_backward(qc, kc, vc, dc, tr, cfg.window, cols, kv_heads=kvh)
    c_t, h_t = torch.as_tensor(cols).cuda(), torch.as_tensor(kvh).cuda()
    assert rel_fro(dk[c_t][:, h_t].cpu().double().numpy(), rk) <= TOL_GRAD_REL
    assert rel_fro(dv[c_t][:, h_t].cpu().double().numpy(), rv) <= TOL_GRAD_REL


def test_results_do_not_depend_on_stream_overlap():
    # the step-list calls spread launches over side streams; launches that add into the same
    # rows stay ordered, so every result is bit-identical with all launches on one stream
    import context_attention_metadata_gb300 as M
    from marble_testlib import run_forward
    cfg = wl.mini_config(2, 8192, hq=2)
    tr = wl.config_tracks(2, cfg.n)
    q, k, v, do = wl.make_qkvdo(cfg.n, cfg.hq, cfg.hkv, cfg.d, device="cuda", seed=4)
    pl = plan_for(cfg, tr)
    out = []
    try:
        for n_side in (4, 0):
            M.set_side_streams(n_side)
            O, L, _ = run_forward(pl, q, k, v)
            out.append((O, L) + tuple(run_backward(pl, q, k, v, do)))
    finally:
        M.set_side_streams(4)
    for a, b in zip(*out):
        assert torch.equal(a, b)
