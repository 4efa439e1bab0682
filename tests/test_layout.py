"""Vision-group layout (MARBLE post, section 04 "Layout transforms"): the library's transform
against the oracle's, and on the GPU, plans of the permuted pack (tokens carrying their
original positions) against the oracle planner, with attention on the permuted pack equal
to attention on the original one."""
import numpy as np
import pytest

import context_attention_metadata_gb300 as M
import workloads as wl
from oracle import attention, mask, plan as oplan

INF = wl.WINDOW_INF


@pytest.mark.parametrize("seed", range(6))
def test_layout_matches_oracle(seed):
    rng = np.random.default_rng(500 + seed)
    if seed < 4:
        tr = wl.random_pack(rng, 128 * int(rng.choice([8, 24, 64])), max_samples=5)
    else:
        tr = wl.config_tracks(7, 128 * 256) if seed == 4 else wl.config_tracks(5, 128 * 512)
    perm = M.layout_vision_groups(tr["sample"], tr["seg"])
    assert np.array_equal(perm, oplan.vision_group_layout(tr))
    assert np.array_equal(np.sort(perm), np.arange(len(perm)))


def test_layout_argument_checks():
    with pytest.raises(M.MarbleError):
        M.layout_vision_groups(np.array([1, 0], np.int32), np.array([-1, -1], np.int32))


def _layout_pack(cid, n):
    tr = wl.config_tracks(cid, n)
    perm = oplan.vision_group_layout(tr)
    return tr, perm, oplan.apply_layout(tr, perm)


@pytest.mark.gpu
@pytest.mark.parametrize("order", ["contiguous", "ptrr_block", "chunk_search"])
def test_plan_with_positions_matches_oracle(order):
    import torch
    from marble_testlib import device_tracks
    from test_gpu_plan import _compare
    tr, perm, trp = _layout_pack(7, 16384)
    s, g, z = device_tracks(trp)
    pos = torch.as_tensor(trp["pos"].astype(np.int32)).cuda()
    pl = M.Plan(s, g, z, INF, 4, order, 0, pos=pos, range_cost=20000)
    opl = oplan.make_plan(trp, INF, 4, order, range_cost=20000)
    _compare(pl, opl)
    st = pl.stats()
    assert pl.export("interval_blocks").any().item()   # exact intervals from the positions
    # fewer partial tiles than the same pack in its original order
    s0, g0, z0 = device_tracks(tr)
    st0 = M.Plan(s0, g0, z0, INF, 4, order, 0, range_cost=20000).stats()
    assert st["legal_pairs"] == st0["legal_pairs"]
    assert st["n_partial"] < 0.2 * st0["n_partial"]


@pytest.mark.gpu
def test_attention_on_layout_equals_original():
    import torch
    from marble_testlib import check_o_lse, device_tracks, rel_fro, TOL_GRAD_REL, run_backward, \
        run_forward
    cfg = wl.mini_config(7, 8192, hq=2)
    tr, perm, trp = _layout_pack(7, cfg.n)
    q, k, v, do = wl.make_qkvdo(cfg.n, cfg.hq, cfg.hkv, cfg.d, device="cuda", seed=7)
    pt = torch.as_tensor(perm).cuda()
    qn, kn, vn, don = (t[pt].contiguous() for t in (q, k, v, do))
    s, g, z = device_tracks(trp)
    pos = torch.as_tensor(trp["pos"].astype(np.int32)).cuda()
    pl = M.Plan(s, g, z, cfg.window, cfg.shards, cfg.order, cfg.chunk_tokens, pos=pos)
    O, L, _ = run_forward(pl, qn, kn, vn)
    qc, kc, vc = (t.cpu() for t in (q, k, v))
    Oref, Lref = attention.rows_forward(qc, kc, vc, tr, cfg.window, np.arange(cfg.n))
    check_o_lse(O, L, Oref[perm], Lref[:, perm])
    cfg = wl.mini_config(7, 4096, hq=2)
    tr, perm, trp = _layout_pack(7, cfg.n)
    q, k, v, do = wl.make_qkvdo(cfg.n, cfg.hq, cfg.hkv, cfg.d, device="cuda", seed=8)
    pt = torch.as_tensor(perm).cuda()
    s, g, z = device_tracks(trp)
    pos = torch.as_tensor(trp["pos"].astype(np.int32)).cuda()
    pl = M.Plan(s, g, z, cfg.window, cfg.shards, cfg.order, cfg.chunk_tokens, pos=pos)
    dq, dk, dv = run_backward(pl, *(t[pt].contiguous() for t in (q, k, v, do)))
    rq, rk, rv, _, _ = attention.backward(q, k, v, do, mask.dense_mask(tr, cfg.window))
    for got, ref in ((dq, rq), (dk, rk), (dv, rv)):
        assert rel_fro(got.cpu().double().numpy(), ref[perm]) <= TOL_GRAD_REL
