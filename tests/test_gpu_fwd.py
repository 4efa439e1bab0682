"""Forward parity: the CUDA ring steps + finalize against the fp64 oracle (dense on small
packs, sampled rows at full size), P- and step-order invariance of the carried fp32 state,
needed-block mode, fully masked rows and GQA / d = 64 variants."""
import numpy as np
import pytest
import torch

import context_attention_metadata_gb300 as M
import workloads as wl
from marble_testlib import check_o_lse, make_plan, plan_for, rel_fro, run_forward
from oracle import attention, mask, ring

pytestmark = pytest.mark.gpu
INF = wl.WINDOW_INF


def _qkv(n, hq, hkv, d, seed=0):
    return wl.make_qkvdo(n, hq, hkv, d, device="cuda", seed=seed)[:3]


def _dense_ref(tr, W, q, k, v):
    return attention.forward(q, k, v, mask.dense_mask(tr, W))


def test_config1_forward():
    cfg = wl.CONFIGS[1]
    tr = wl.config_tracks(1)
    q, k, v = _qkv(cfg.n, cfg.hq, cfg.hkv, cfg.d)
    pl = plan_for(cfg, tr)
    O, L, _ = run_forward(pl, q, k, v)
    Oref, Lref = _dense_ref(tr, INF, q, k, v)
    check_o_lse(O, L, Oref, Lref)


@pytest.mark.parametrize("seed", range(8))
def test_random_packs_forward(seed):
    rng = np.random.default_rng(500 + seed)
    n = 128 * int(rng.choice([8, 16, 24]))
    tr = wl.random_pack(rng, n, max_samples=int(rng.integers(1, 6)))
    d = int(rng.choice([64, 128]))
    hkv = int(rng.choice([1, 2]))
    hq = hkv * int(rng.choice([1, 2, 3]))
    P = int(rng.choice([1, 2, 4]))
    order = ["contiguous", "ptrr_block", "ptrr_chunk"][seed % 3]
    W = int(rng.choice([INF, 1, 50, 200]))
    q, k, v = _qkv(n, hq, hkv, d, seed=seed)
    pl = make_plan(tr, W, P, order, chunk_tokens=128)
    O, L, _ = run_forward(pl, q, k, v, needed=bool(seed % 2))
    Oref, Lref = _dense_ref(tr, W, q, k, v)
    check_o_lse(O, L, Oref, Lref)


def test_fully_masked_rows():
    # W = 0: causal tokens see nothing (O = 0, LSE = -inf); bidirectional spans see
    # themselves; whole tiles of masked rows must not produce NaN
    samples = [[wl.Span("causal", 300), wl.Span("full", 200)], [wl.Span("causal", 12)]]
    tr = wl.tracks_from_samples(samples)
    n = 512
    q, k, v = _qkv(n, 2, 2, 128)
    pl = make_plan(tr, 0, 2)
    O, L, _ = run_forward(pl, q, k, v)
    Oref, Lref = _dense_ref(tr, 0, q, k, v)
    assert torch.isfinite(O.float()).all()
    check_o_lse(O, L, Oref, Lref)
    assert (O[:300] == 0).all() and torch.isinf(L[:, :300]).all()


def _canonical(st, n):
    l = st.l.cpu().double().numpy()
    m = st.m.cpu().double().numpy()
    o = st.o_acc.cpu().double().numpy()
    with np.errstate(divide="ignore", invalid="ignore"):
        on = np.where(l.T[:, :, None] > 0, o / l.T[:, :, None], 0)
        lse = np.where(l > 0, (m + np.log2(np.where(l > 0, l, 1))) * np.log(2), -np.inf)
    return on, lse


@pytest.mark.parametrize("merge", ["carried", "fp32"])
def test_state_is_invariant_to_P_and_step_order(merge):
    """MARBLE s03: the online kernel's results equal a single GPU's at every ring degree.
    The carried fp32 state (canonicalised as O_acc / l and m + log l) agrees across
    P in {1, 2, 4, 8, 16} and under a shuffled step order to 1e-5 relative; so does the
    state of the merge of fp32 partials (O_acc normalised, l = 1, m the base-2 LSE)."""
    cfg = wl.CONFIGS[1]
    tr = wl.config_tracks(1)
    q, k, v = _qkv(cfg.n, cfg.hq, cfg.hkv, cfg.d)
    ref = None
    rng = np.random.default_rng(0)
    for P in (1, 2, 4, 8, 16):
        for shuffled in (False, True):
            pl = make_plan(tr, INF, P)
            sched = M.ring_schedule(P)
            if shuffled:
                sched = []
                for r in range(P):
                    js = list(rng.permutation(P))
                    sched += [(r, int(j), s == 0) for s, j in enumerate(js)]
            _, _, st = run_forward(pl, q, k, v, schedule=sched, merge=merge)
            on, lse = _canonical(st, cfg.n)  # contiguous order: plan order = original
            if ref is None:
                ref = (on, lse)
                continue
            assert rel_fro(on, ref[0]) <= 1e-5
            fin = np.isfinite(ref[1])
            d = np.abs(lse[fin] - ref[1][fin]) / np.maximum(1, np.abs(ref[1][fin]))
            assert d.max() <= 1e-5


@pytest.mark.parametrize("cid,n", [(2, 8192), (5, 16384)])
def test_production_state_is_invariant_to_P_and_step_order(cid, n):
    """MARBLE s03 ("Exact ring attention accumulation"): results equal a single GPU's at
    every ring degree.  The production path -- d = 128, PTRR block order (the token order
    itself changes with P), key intervals on, image groups in the grouped-image recipe --
    gives the same carried fp32 state, canonicalised as (O_acc / l, m + log l) in original
    token order, for P in {1, 2, 4, 8, 16} and under a shuffled step order, to 1e-5
    relative (Frobenius) and 1e-5 max(1, |LSE|) absolute.  The grouped pack is 16K tokens,
    the smallest of its recipe that holds an image group of two images."""
    cfg = wl.mini_config(cid, n, hq=2)
    tr = wl.config_tracks(cid, n)
    q, k, v = _qkv(n, cfg.hq, cfg.hkv, cfg.d, seed=40 + cid)
    assert cfg.d == 128 and cfg.order == "ptrr_block"
    ref = None
    rng = np.random.default_rng(cid)
    for P in (1, 2, 4, 8, 16):
        pl = make_plan(tr, cfg.window, P, "ptrr_block")
        perm = pl.export("perm").long().cpu().numpy()
        for shuffled in (False, True):
            sched = M.ring_schedule(P)
            if shuffled:
                sched = []
                for r in range(P):
                    js = list(rng.permutation(P))
                    sched += [(r, int(j), s == 0) for s, j in enumerate(js)]
            _, _, st = run_forward(pl, q, k, v, schedule=sched)
            on_p, lse_p = _canonical(st, n)
            on = np.empty_like(on_p)
            lse = np.empty_like(lse_p)
            on[perm] = on_p             # plan order -> original order
            lse[:, perm] = lse_p
            if ref is None:
                ref = (on, lse)
                continue
            assert rel_fro(on, ref[0]) <= 1e-5, (P, shuffled)
            fin = np.isfinite(ref[1])
            assert (np.isfinite(lse) == fin).all()
            d = np.abs(lse[fin] - ref[1][fin]) / np.maximum(1, np.abs(ref[1][fin]))
            assert d.max() <= 1e-5, (P, shuffled)
        if P == 8:
            assert pl.export("interval_blocks").any()  # the interval test is in use


def test_needed_mode_equals_ring_steps():
    cfg = wl.mini_config(3, 8192)
    tr = wl.config_tracks(3, cfg.n)
    q, k, v = _qkv(cfg.n, cfg.hq, cfg.hkv, cfg.d)
    pl = plan_for(cfg, tr)
    O1, L1, _ = run_forward(pl, q, k, v, needed=True)
    O2, L2, _ = run_forward(pl, q, k, v, needed=False)
    assert (O1.float() - O2.float()).abs().max() <= 1e-2
    Oref, Lref = _dense_ref(tr, cfg.window, q, k, v)
    check_o_lse(O1, L1, Oref, Lref)
    check_o_lse(O2, L2, Oref, Lref)


@pytest.mark.parametrize("cid", [2, 3, 4, 5])
def test_mini_configs_forward(cid):
    cfg = wl.mini_config(cid, 8192)
    tr = wl.config_tracks(cid, cfg.n)
    q, k, v = _qkv(cfg.n, cfg.hq, cfg.hkv, cfg.d)
    pl = plan_for(cfg, tr)
    O, L, _ = run_forward(pl, q, k, v, needed=cfg.needed)
    qc, kc, vc = (t.cpu() for t in (q, k, v))
    Oref, Lref = attention.rows_forward(qc, kc, vc, tr, cfg.window, np.arange(cfg.n))
    check_o_lse(O, L, Oref, Lref)


def _sample_rows(cfg, rng, count):
    n = cfg.n
    bps = n // 128 // cfg.shards
    rows = set(rng.choice(n, count, replace=False).tolist())
    for r in (0, cfg.shards - 1):  # first and last block of two shards (contiguous view)
        a = r * bps * 128
        rows.update(range(a, a + 128))
        rows.update(range(a + (bps - 1) * 128, a + bps * 128))
    return np.array(sorted(rows))


@pytest.mark.parametrize("cid", [2, 3, 4, 5])
def test_full_configs_forward_sampled(cid):
    cfg = wl.CONFIGS[cid]
    tr = wl.config_tracks(cid)
    q, k, v = _qkv(cfg.n, cfg.hq, cfg.hkv, cfg.d)
    pl = plan_for(cfg, tr)
    O, L, _ = run_forward(pl, q, k, v, needed=cfg.needed)
    assert torch.isfinite(L).all()
    rng = np.random.default_rng(cid)
    rows = _sample_rows(cfg, rng, 128 if cid >= 4 else 256)
    heads = np.arange(cfg.hq) if cid in (2, 3) else np.array([0, cfg.hq - 1])
    rows_t = torch.as_tensor(rows).cuda()
    qc, kc, vc = (t.cpu() for t in (q, k, v))
    Oref, Lref = attention.rows_forward(qc, kc, vc, tr, cfg.window, rows, heads=heads)
    hs = torch.as_tensor(heads).cuda()
    check_o_lse(O[rows_t][:, hs], L[hs][:, rows_t], Oref, Lref)


def _bf16_merge_case(n=8192, hq=2, d=128, seed=21):
    cfg = wl.mini_config(2, n, hq=hq)
    tr = wl.config_tracks(2, n)
    q, k, v = _qkv(n, cfg.hq, cfg.hkv, d, seed=seed)
    return cfg, tr, q, k, v


def test_bf16_merge_matches_its_oracle():
    # the standard ring merge (bf16 partial per step, bf16 running output, log-sum-exp
    # weights) in the same ring order and on the same plan-ordered shards as the oracle
    cfg, tr, q, k, v = _bf16_merge_case()
    pl = plan_for(cfg, tr)
    O, L, st = run_forward(pl, q, k, v, merge="bf16")
    perm = pl.export("perm").long().cpu().numpy()
    Mp = mask.dense_mask(tr, cfg.window, rows=perm, cols=perm)  # plan order, original positions
    Ob, Lb = ring.ring_forward_bf16_merge(q.cpu()[perm], k.cpu()[perm], v.cpu()[perm], Mp,
                                          P=cfg.shards)
    inv = np.empty_like(perm)
    inv[perm] = np.arange(len(perm))
    check_o_lse(O, L, Ob[inv], Lb[:, inv])
    # the stored running output is bf16-valued and l is 1 on live rows, 0 on dead ones
    acc = st.o_acc.cpu()
    assert torch.equal(acc, acc.to(torch.bfloat16).float())
    lv = st.l.cpu().numpy()
    assert set(np.unique(lv)) <= {0.0, 1.0}


def test_bf16_merge_single_pass_is_rounded_exact():
    # needed-block mode runs one call per q shard: one rounded partial, nothing to merge
    cfg, tr, q, k, v = _bf16_merge_case(n=4096, seed=22)
    pl = plan_for(cfg, tr)
    O, L, _ = run_forward(pl, q, k, v, needed=True, merge="bf16")
    Oref, Lref = _dense_ref(tr, cfg.window, q, k, v)
    check_o_lse(O, L, ring.round_bf16(Oref), Lref)


def test_bf16_merge_error_exceeds_carried_fp32():
    # the accuracy gap the carried fp32 state removes: same inputs, same plan, P = 8
    cfg, tr, q, k, v = _bf16_merge_case(seed=23)
    pl = plan_for(cfg, tr)
    Oref, _ = _dense_ref(tr, cfg.window, q, k, v)
    O32, _, _ = run_forward(pl, q, k, v)
    O16, _, _ = run_forward(pl, q, k, v, merge="bf16")
    e32 = np.abs(O32.float().cpu().numpy() - Oref).mean()
    e16 = np.abs(O16.float().cpu().numpy() - Oref).mean()
    print(f"mean |O - O_exact|: carried fp32 {e32:.3e}, bf16 merge {e16:.3e}, "
          f"ratio {e16 / e32:.3f}")
    assert e16 > 1.05 * e32


def test_bf16_merge_flag_is_uniform_per_call():
    cfg, tr, q, k, v = _bf16_merge_case(n=2048, seed=24)
    pl = plan_for(cfg, tr)
    st = M.State(cfg.n, cfg.hq, cfg.d)
    qp, kp, vp = pl.permute(q), pl.permute(k), pl.permute(v)
    import ctypes
    c = M._qkv(pl, qp, kp, vp, 0.0)
    s = st._c()
    qs = (ctypes.c_int32 * 2)(0, 0)
    ks = (ctypes.c_int32 * 2)(0, 1)
    fl = (ctypes.c_uint32 * 2)(M.STEP_FIRST | M.STEP_BF16_MERGE, 0)
    rc = M.lib().marble_attn_steps(pl.handle, ctypes.byref(c), 2, qs, ks, fl,
                                   ctypes.byref(s), None)
    assert rc == 1  # MARBLE_ERR_INVALID_ARG, nothing launched


@pytest.mark.parametrize("cid", [2, 3, 5])
def test_fp32_merge_matches_exact(cid):
    # the merge of fp32 partials is exact to fp32: same bar as the carried state against the
    # fp64 oracle, and within one bf16 step of the carried state's output
    cfg = wl.mini_config(cid, 8192, hq=2)
    tr = wl.config_tracks(cid, cfg.n)
    q, k, v = _qkv(cfg.n, cfg.hq, cfg.hkv, cfg.d, seed=30 + cid)
    pl = plan_for(cfg, tr)
    O, L, _ = run_forward(pl, q, k, v, merge="fp32", needed=cfg.needed)
    Oref, Lref = _dense_ref(tr, cfg.window, q, k, v)
    check_o_lse(O, L, Oref, Lref)
    Oc, Lc, _ = run_forward(pl, q, k, v, needed=cfg.needed)
    assert ((O.float() - Oc.float()).abs() <= 2.0**-7 * Oc.float().abs().clamp(min=1)).all()
    fin = torch.isfinite(Lc)
    assert torch.equal(torch.isfinite(L), fin)
    assert (L[fin] - Lc[fin]).abs().max() <= 1e-4


def test_fp32_merge_error_matches_carried_and_beats_bf16():
    cfg, tr, q, k, v = _bf16_merge_case(seed=25)
    pl = plan_for(cfg, tr)
    Oref, _ = _dense_ref(tr, cfg.window, q, k, v)
    err = {}
    for merge in ("carried", "fp32", "bf16"):
        O, _, _ = run_forward(pl, q, k, v, merge=merge)
        err[merge] = np.abs(O.float().cpu().numpy() - Oref).mean()
    print("mean |O - O_exact|:", {k_: f"{v_:.3e}" for k_, v_ in err.items()})
    assert abs(err["fp32"] / err["carried"] - 1) < 0.05
    assert err["bf16"] > 1.05 * err["fp32"]


def test_merge_flags_are_checked():
    import ctypes
    cfg, tr, q, k, v = _bf16_merge_case(n=2048, seed=26)
    pl = plan_for(cfg, tr)
    st = M.State(cfg.n, cfg.hq, cfg.d)
    qp, kp, vp = pl.permute(q), pl.permute(k), pl.permute(v)
    c = M._qkv(pl, qp, kp, vp, 0.0)
    s_ = st._c()
    both = M.STEP_FIRST | M.STEP_BF16_MERGE | M.STEP_FP32_MERGE
    assert M.lib().marble_attn_step(pl.handle, ctypes.byref(c), 0, 0, ctypes.byref(s_),
                                    both, None) == 1
    qs = (ctypes.c_int32 * 2)(0, 0)
    ks = (ctypes.c_int32 * 2)(0, 1)
    fl = (ctypes.c_uint32 * 2)(M.STEP_FIRST | M.STEP_FP32_MERGE, M.STEP_BF16_MERGE)
    assert M.lib().marble_attn_steps(pl.handle, ctypes.byref(c), 2, qs, ks, fl,
                                     ctypes.byref(s_), None) == 1
    with pytest.raises(ValueError):
        M.attn_step(pl, qp, kp, vp, 0, 0, st, first=True, merge="fp16")
