"""Chunk-layout search (MARBLE post, section 03 "Chunked ring attention"): the library's
host search against the oracle's, bit-exact, on legal-pair matrices of random packs and on
arbitrary work matrices; and on the GPU, plans built with the searched layout against the
oracle planner, with attention parity on such a plan."""
import numpy as np
import pytest

import context_attention_metadata_gb300 as M
import workloads as wl
from oracle import attention, mask, plan as oplan

INF = wl.WINDOW_INF


def _same(o, c):
    C, k, rank, step = o
    assert (k, C, step) == c[:3]
    assert np.array_equal(rank, c[3])


@pytest.mark.parametrize("seed", range(4))
def test_search_matches_oracle_on_packs(seed):
    rng = np.random.default_rng(40 + seed)
    P = [2, 4, 8, 16][seed]
    nb = 64
    tr = wl.random_pack(rng, nb * 128, max_samples=int(rng.integers(1, 7)))
    W = int(rng.choice([INF, 300, 2000]))
    Wb = oplan.block_pair_counts(tr, W)
    for tau in (0, 1000, 50000, 10**10):
        _same(oplan.chunk_search(Wb, P, tau), M.chunk_layout_search(Wb, P, tau))


@pytest.mark.parametrize("seed", range(4))
def test_search_matches_oracle_on_arbitrary_work(seed):
    # ties (small integer work, many zeros) exercise the dealing order and the swap order
    rng = np.random.default_rng(60 + seed)
    P = [2, 3, 4, 6][seed]
    nb = P * [8, 16, 8, 4][seed]
    Wb = rng.integers(0, 4, (nb, nb)) * rng.integers(0, 2, (nb, nb))
    for tau in (0, 1, 7):
        _same(oplan.chunk_search(Wb, P, tau), M.chunk_layout_search(Wb, P, tau))


def test_search_argument_checks():
    w = np.ones((6, 6), np.int64)
    with pytest.raises(M.MarbleError):
        M.chunk_layout_search(w, 4)           # 6 blocks over 4 ranks
    with pytest.raises(M.MarbleError):
        M.chunk_layout_search(-w, 2)          # negative work
    with pytest.raises(M.MarbleError):
        M.chunk_layout_search(w, 2, range_cost=-1)


@pytest.mark.gpu
@pytest.mark.parametrize("seed", range(3))
def test_searched_plan_matches_oracle_plan(seed):
    from marble_testlib import make_plan
    from test_gpu_plan import _compare
    rng = np.random.default_rng(80 + seed)
    n = 128 * 64
    tr = wl.config_tracks(6, n) if seed == 0 else wl.random_pack(rng, n, max_samples=4)
    P = [4, 8, 2][seed]
    W = [INF, INF, 500][seed]
    tau = [0, 20000, 3 * 10**5][seed]
    pl = make_plan(tr, W, P, "chunk_search", range_cost=tau)
    opl = oplan.make_plan(tr, W, P, "chunk_search", range_cost=tau)
    _compare(pl, opl)
    C, k, _, step = oplan.chunk_search(oplan.block_pair_counts(tr, W), P, tau)
    st = pl.stats()
    assert (st["chunks_per_rank"], st["layout_cost"], st["layout_step_cost"]) == (k, C, step)
    assert st["step_cost_pairs"] == step


@pytest.mark.gpu
@pytest.mark.parametrize("order", ["contiguous", "ptrr_block", "ptrr_chunk"])
def test_step_cost_in_pairs_for_every_order(order):
    from marble_testlib import make_plan
    rng = np.random.default_rng(90)
    n, P = 128 * 64, 4
    tr = wl.random_pack(rng, n, max_samples=5)
    pl = make_plan(tr, INF, P, order, chunk_tokens=1024)
    opl = oplan.make_plan(tr, INF, P, order, chunk_tokens=1024)
    Wb = oplan.block_pair_counts(tr, INF)
    bps = opl.nb // P
    rank = np.repeat(np.arange(P), bps)  # new block -> its shard
    Wc = Wb[np.ix_(opl.block_perm, opl.block_perm)]
    assert pl.stats()["step_cost_pairs"] == oplan.layout_step_cost(Wc, rank, P)


@pytest.mark.gpu
def test_attention_on_searched_layout():
    import torch
    from marble_testlib import check_o_lse, plan_for, run_backward, run_forward
    from test_gpu_bwd import _check_dense
    # forward on an 8K pack of the long-video generation recipe, every row against the oracle
    cfg = wl.mini_config(6, 8192, hq=2)
    tr = wl.config_tracks(6, cfg.n)
    q, k, v, do = wl.make_qkvdo(cfg.n, cfg.hq, cfg.hkv, cfg.d, device="cuda", seed=6)
    pl = plan_for(cfg, tr)
    assert pl.stats()["chunks_per_rank"] >= 1
    O, L, _ = run_forward(pl, q, k, v)
    qc, kc, vc = (t.cpu() for t in (q, k, v))
    Oref, Lref = attention.rows_forward(qc, kc, vc, tr, cfg.window, np.arange(cfg.n))
    check_o_lse(O, L, Oref, Lref)
    # backward on a 4K pack, dense oracle
    cfg = wl.mini_config(6, 4096, hq=2)
    tr = wl.config_tracks(6, cfg.n)
    q, k, v, do = wl.make_qkvdo(cfg.n, cfg.hq, cfg.hkv, cfg.d, device="cuda", seed=7)
    pl = plan_for(cfg, tr)
    dq, dk, dv = run_backward(pl, q, k, v, do)
    _check_dense(tr, cfg.window, q, k, v, do, dq, dk, dv)


@pytest.mark.gpu
def test_full_video_generation_forward_sampled():
    # the 1M-token long-video generation pack on its searched layout (P = 16, fitted tau):
    # sampled rows of the output and LSE against the fp64 oracle
    import torch
    from marble_testlib import check_o_lse, plan_for, run_forward
    cfg = wl.EXTRA[6]
    tr = wl.config_tracks(6)
    q, k, v = wl.make_qkvdo(cfg.n, cfg.hq, cfg.hkv, cfg.d, device="cuda", seed=3)[:3]
    pl = plan_for(cfg, tr)
    st = pl.stats()
    assert st["chunks_per_rank"] >= 1 and st["layout_step_cost"] == st["step_cost_pairs"]
    O, L, _ = run_forward(pl, q, k, v)
    assert torch.isfinite(L).all()
    rng = np.random.default_rng(6)
    rows = np.sort(rng.choice(cfg.n, 24, replace=False))
    heads = np.array([0, cfg.hq - 1])
    qc, kc, vc = (t.cpu() for t in (q, k, v))
    Oref, Lref = attention.rows_forward(qc, kc, vc, tr, cfg.window, rows, heads=heads)
    rt, ht = torch.as_tensor(rows).cuda(), torch.as_tensor(heads).cuda()
    check_o_lse(O[rt][:, ht], L[ht][:, rt], Oref, Lref)
