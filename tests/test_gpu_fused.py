"""The fused ring (marble_attn_fwd_fused, marble_attn_bwd_fused) against the fp64 oracle
and against the per-step path.

MARBLE post, s03 "Exact ring attention accumulation": the carried fp32 state gives a
single GPU's result at every ring degree and in any step order.  The fused forward runs
every ring step of a row in one launch with the state on chip between steps, and the fused
backward keeps each kv shard's dK/dV on chip across its ring; the results must equal the
per-step path's up to fp32 summation order, and the oracle's within the stated tolerances."""
import os

import numpy as np
import pytest
import torch

import context_attention_metadata_gb300 as M
import workloads as wl
from marble_testlib import (TOL_GRAD_REL, check_o_lse, make_plan, plan_for, rel_fro,
                            run_backward, run_forward)
from oracle import attention, mask

pytestmark = pytest.mark.gpu
INF = wl.WINDOW_INF


def _canonical_orig(st, perm):
    l = st.l.cpu().double().numpy()
    m = st.m.cpu().double().numpy()
    o = st.o_acc.cpu().double().numpy()
    with np.errstate(divide="ignore", invalid="ignore"):
        on = np.where(l.T[:, :, None] > 0, o / l.T[:, :, None], 0)
        lse = np.where(l > 0, (m + np.log2(np.where(l > 0, l, 1))) * np.log(2), -np.inf)
    on_o, lse_o = np.empty_like(on), np.empty_like(lse)
    on_o[perm] = on
    lse_o[:, perm] = lse
    return on_o, lse_o


@pytest.mark.parametrize("cid,n,P", [(1, 2048, 4), (2, 8192, 8), (5, 16384, 16), (4, 8192, 8)])
def test_fused_forward_equals_oracle_and_steps(cid, n, P):
    cfg = wl.CONFIGS[1] if cid == 1 else wl.mini_config(cid, n, hq=2)
    tr = wl.config_tracks(cid) if cid == 1 else wl.config_tracks(cid, n)
    q, k, v = wl.make_qkvdo(n, cfg.hq, cfg.hkv, cfg.d, device="cuda", seed=60 + cid)[:3]
    pl = make_plan(tr, cfg.window, P, cfg.order, cfg.chunk_tokens)
    O, L, st_f = run_forward(pl, q, k, v, fused=True)
    Oref, Lref = attention.forward(q, k, v, mask.dense_mask(tr, cfg.window))
    check_o_lse(O, L, Oref, Lref)
    O2, L2, st_s = run_forward(pl, q, k, v)
    perm = pl.export("perm").long().cpu().numpy()
    a, la = _canonical_orig(st_f, perm)
    b, lb = _canonical_orig(st_s, perm)
    assert rel_fro(a, b) <= 1e-5
    fin = np.isfinite(lb)
    assert (np.isfinite(la) == fin).all()
    assert (np.abs(la[fin] - lb[fin]) / np.maximum(1, np.abs(lb[fin]))).max() <= 1e-5


def test_fused_forward_rows_without_tiles():
    # W = 0: causal rows see nothing and have no tile at all; they must come out as
    # (O = 0, LSE = -inf), written by the fused launch like the FIRST step writes them
    samples = [[wl.Span("causal", 300), wl.Span("full", 200)], [wl.Span("causal", 12)]]
    tr = wl.tracks_from_samples(samples)
    q, k, v = wl.make_qkvdo(512, 2, 2, 128, device="cuda")[:3]
    pl = make_plan(tr, 0, 2)
    O, L, _ = run_forward(pl, q, k, v, fused=True)
    Oref, Lref = attention.forward(q, k, v, mask.dense_mask(tr, 0))
    check_o_lse(O, L, Oref, Lref)
    assert (O[:300] == 0).all() and torch.isinf(L[:, :300]).all()


def _backward_from(pl, qp, kp, vp, dop, o, lse, delta, kind, sched=None):
    """One backward of `kind` ("steps" or "fused") from given forward outputs (plan order);
    gradients in original order."""
    n, hq, d = qp.shape
    hkv = kp.shape[1]
    g = [torch.zeros((n, hq, d), device="cuda"), torch.zeros((n, hkv, d), device="cuda"),
         torch.zeros((n, hkv, d), device="cuda")]
    if kind == "fused":
        M.attn_bwd_fused(pl, qp, kp, vp, dop, lse, delta, *g)
    else:
        M.attn_bwd_steps(pl, qp, kp, vp, dop, lse, delta,
                         sched if sched is not None else M.ring_schedule(pl.num_shards), *g)
    pl.check()
    return [pl.permute(x, inverse=True) for x in g]


def _both_backwards(pl, q, k, v, do, calibrate=None):
    """One per-step forward, then the per-step and the fused backward from the same O, LSE
    and delta: gradients in original order, [per-step, fused].  With calibrate = (tracks,
    window) two more: the per-step backward with every (q shard, kv shard) step in a random
    order, and the per-step backward of a one-shard plan of the same pack from the same
    forward outputs (every unit then accumulates its whole column in TMEM, as the fused
    backward does)."""
    n, hq, d = q.shape
    qp, kp, vp, dop = (pl.permute(t) for t in (q, k, v, do))
    st = M.State(n, hq, d)
    o = torch.empty((n, hq, d), dtype=torch.bfloat16, device="cuda")
    lse = torch.empty((hq, n), dtype=torch.float32, device="cuda")
    M.forward(pl, qp, kp, vp, st, o, lse)
    delta = torch.empty_like(lse)
    M.attn_bwd_prep(pl, o, dop, delta)
    out = [_backward_from(pl, qp, kp, vp, dop, o, lse, delta, "steps"),
           _backward_from(pl, qp, kp, vp, dop, o, lse, delta, "fused")]
    if calibrate is None:
        return out
    P = pl.num_shards
    rng = np.random.default_rng(5)
    pairs = [(r, j) for r in range(P) for j in range(P)]
    shuf = [(pairs[i][0], pairs[i][1], False) for i in rng.permutation(len(pairs))]
    out.append(_backward_from(pl, qp, kp, vp, dop, o, lse, delta, "steps", shuf))
    # the same forward outputs in the order of a one-shard plan
    tr, window = calibrate
    perm = pl.export("perm").long()
    o0 = pl.permute(o, inverse=True)
    lse0, delta0 = torch.empty_like(lse), torch.empty_like(delta)
    lse0[:, perm] = lse
    delta0[:, perm] = delta
    pl1 = make_plan(tr, window, 1, "contiguous")
    perm1 = pl1.export("perm").long()
    out.append(_backward_from(pl1, *(pl1.permute(t) for t in (q, k, v, do)), pl1.permute(o0),
                              lse0[:, perm1].contiguous(), delta0[:, perm1].contiguous(),
                              "steps"))
    return out


def _close_to_steps(fused, steps, shuffled, one_shard, names=("dq", "dk", "dv")):
    """The fused and the per-step backward add the same products in another grouping.  Two
    scales are measured rather than assumed: a shuffled step order (the order of the fp32
    additions in memory) and a one-shard plan (TMEM accumulation over whole columns, which
    the tensor core does not round like a chain of IEEE fp32 additions).  The fused result
    must lie within 4x the larger of them of the per-step one (and within 1e-5 where both
    cost less)."""
    for name, a, b, c, e1 in zip(names, fused, steps, shuffled, one_shard):
        a, b, c, e1 = (x.cpu().double().numpy() for x in (a, b, c, e1))
        scale = max(rel_fro(c, b), rel_fro(e1, b))
        e = rel_fro(a, b)
        print(f"{name}: fused vs per-step {e:.3e}; reorder {rel_fro(c, b):.3e}, "
              f"one-shard plan {rel_fro(e1, b):.3e}")
        assert e <= max(1e-5, 4 * scale), f"{name}: fused vs per-step {e}, scales {scale}"


@pytest.mark.parametrize("cid,n,P", [(2, 4096, 8), (4, 4096, 8), (5, 16384, 16)])
def test_fused_backward_equals_oracle_and_steps(cid, n, P):
    cfg = wl.mini_config(cid, n, hq=2)
    tr = wl.config_tracks(cid, n)
    q, k, v, do = wl.make_qkvdo(n, cfg.hq, cfg.hkv, cfg.d, device="cuda", seed=70 + cid)
    pl = make_plan(tr, cfg.window, P, cfg.order, cfg.chunk_tokens)
    got = run_backward(pl, q, k, v, do, fused=True)
    rq, rk, rv, _, _ = attention.backward(q, k, v, do, mask.dense_mask(tr, cfg.window))
    for name, g, ref in zip(("dq", "dk", "dv"), got, (rq, rk, rv)):
        e = rel_fro(g.cpu().double().numpy(), ref)
        assert e <= TOL_GRAD_REL, f"{name} rel err {e}"
    # from the same forward outputs the two backwards differ only in how the fp32 sums group
    steps, fused, shuf, one = _both_backwards(pl, q, k, v, do, calibrate=(tr, cfg.window))
    _close_to_steps(fused, steps, shuf, one)


def _with_env(env, fn):
    os.environ.update(env)
    try:
        return fn()
    finally:
        for k in env:
            del os.environ[k]


def _with_cap(mb, fn):
    return _with_env({"MARBLE_DS_SCRATCH_CAP_MB": str(mb)}, fn)


# whole-row dQ GEMMs regardless of row balance (on a small pack one long row would otherwise
# send the backward to the per-step GEMMs)
WHOLE = {"MARBLE_WHOLE_ROWS": "always"}


@pytest.mark.parametrize("hq,hkv,d", [(2, 2, 128), (4, 2, 64)])
def test_backward_scratch_modes(hq, hkv, d):
    """The backward's three ways of holding the dS^T tiles, reached through the scratch cap
    (and, on this small pack, MARBLE_WHOLE_ROWS=always): every tile of the pack at once (one
    whole-row dQ GEMM after every dK/dV launch); a few q shards' tiles at a time (whole-row
    dQ per q shard, buffers taken over in turn); and a few steps' tiles at a time (a dQ GEMM
    after each step; the fused backward splits each kv shard's ring into ranges).  All agree
    up to fp32 summation order and each matches the oracle; with and without grouped kv
    heads, at both head dims."""
    cfg = wl.mini_config(2, 8192, hq=hq, hkv=hkv)
    tr = wl.config_tracks(2, 8192)
    q, k, v, do = wl.make_qkvdo(8192, hq, hkv, d, device="cuda", seed=81)
    pl = make_plan(tr, cfg.window, 8, "ptrr_block")
    st = pl.stats()
    assert st["shard_cost_max"] * cfg.hq * 32768 * 3 < st["nnz"] * cfg.hq * 32768
    assert st["shard_cost_max"] * cfg.hq * 32768 * 2 > 4 << 20  # 4 MB: two q shards do not fit
    steps_whole, fused_whole = _with_env(WHOLE, lambda: _both_backwards(pl, q, k, v, do))
    # three q shards' tiles fit, the whole pack does not
    mb = -(-st["shard_cost_max"] * cfg.hq * 32768 * 3 // (1 << 20))
    steps_shards = _with_env({**WHOLE, "MARBLE_DS_SCRATCH_CAP_MB": str(mb)},
                             lambda: _both_backwards(pl, q, k, v, do))[0]
    steps, split, shuf, one = _with_cap(4, lambda: _both_backwards(pl, q, k, v, do,
                                                                   calibrate=(tr, cfg.window)))
    _close_to_steps(split, steps, shuf, one)
    _close_to_steps(fused_whole, steps, shuf, one)
    _close_to_steps(steps_whole, steps, shuf, one)
    _close_to_steps(steps_shards, steps, shuf, one)
    rq, rk, rv, _, _ = attention.backward(q, k, v, do, mask.dense_mask(tr, cfg.window))
    for got in (split, steps, steps_whole, steps_shards, fused_whole):
        for g, ref in zip(got, (rq, rk, rv)):
            assert rel_fro(g.cpu().double().numpy(), ref) <= TOL_GRAD_REL


def test_fused_full_size_packed_64k_equals_steps():
    """The 64K packed pack at full size (16 heads, d = 128, P = 8, PTRR): fused forward and
    backward against the per-step path, every element."""
    cfg = wl.CONFIGS[2]
    tr = wl.config_tracks(2)
    q, k, v, do = wl.make_qkvdo(cfg.n, cfg.hq, cfg.hkv, cfg.d, device="cuda")
    pl = plan_for(cfg, tr)
    O1, L1, _ = run_forward(pl, q, k, v, fused=True)
    O2, L2, _ = run_forward(pl, q, k, v)
    assert (O1.float() - O2.float()).abs().max() <= 2 ** -7
    assert (L1 - L2).abs().max() <= 1e-4
    g2, g1, g3, g4 = _both_backwards(pl, q, k, v, do, calibrate=(tr, cfg.window))
    for a in g1:
        assert torch.isfinite(a).all()
    _close_to_steps(g1, g2, g3, g4)
