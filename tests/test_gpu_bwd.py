"""Backward parity: dQ, dK, dV from the CUDA backward ring steps (against the final LSE,
fp32 accumulation across steps) against the fp64 oracle's analytic gradients; relative
Frobenius error <= 1e-2.  Dense oracle on small packs, sampled rows/columns at full size."""
import numpy as np
import pytest
import torch

import workloads as wl
from marble_testlib import TOL_GRAD_REL, make_plan, plan_for, rel_fro, run_backward
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


@pytest.mark.parametrize("cid", [2, 3, 4, 5])
def test_full_configs_backward_sampled(cid):
    cfg = wl.CONFIGS[cid]
    tr = wl.config_tracks(cid)
    q, k, v, do = wl.make_qkvdo(cfg.n, cfg.hq, cfg.hkv, cfg.d, device="cuda")
    pl = plan_for(cfg, tr)
    dq, dk, dv = run_backward(pl, q, k, v, do, needed=cfg.needed)
    for g in (dq, dk, dv):
        assert torch.isfinite(g).all()
    qc, kc, vc, dc = (t.cpu() for t in (q, k, v, do))
    rng = np.random.default_rng(10 + cid)
    st = np.asarray(tr["sample"])
    lengths = np.bincount(st)
    # rows and key columns from samples small enough for the fp64 oracle to finish quickly
    small = np.flatnonzero(lengths[st] <= 8192)
    pool = small if len(small) >= 64 else np.arange(cfg.n)
    rows = np.sort(rng.choice(pool, 48, replace=False))
    heads = np.array([0, cfg.hq - 1])
    ref = attention.rows_dq(qc, kc, vc, dc, tr, cfg.window, rows, heads=heads)
    got = dq[torch.as_tensor(rows).cuda()][:, torch.as_tensor(heads).cuda()].cpu().double().numpy()
    assert rel_fro(got, ref) <= TOL_GRAD_REL
    # eight consecutive key columns (their visible-query sets overlap)
    c0 = int(rng.choice(pool))
    c0 = min(c0, cfg.n - 8)
    cols = np.arange(c0, c0 + 8)
    kvh = np.array([0])
    rk, rv = attention.cols_backward(qc, kc, vc, dc, tr, cfg.window, cols, kv_heads=kvh)
    c_t = torch.as_tensor(cols).cuda()
    assert rel_fro(dk[c_t][:, :1].cpu().double().numpy(), rk) <= TOL_GRAD_REL
    assert rel_fro(dv[c_t][:, :1].cpu().double().numpy(), rv) <= TOL_GRAD_REL


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
