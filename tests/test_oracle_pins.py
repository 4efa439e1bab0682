"""Pins for the CPU oracle: values the pages print, closed forms, invariants, brute force.

None of these tests needs a GPU.  Each one is chosen so that a plausible mistake in the
oracle (a dropped term, a wrong sign or index, a transposed operand) fails it.
"""
import math
import os

import numpy as np
import pytest

import workloads as wl
from oracle import attention, counts, mask, plan, ring

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")
INF = wl.WINDOW_INF


def _golden_kv(name):
    out = {}
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            k, v = line.split(None, 1)
            out[k] = v
    return out


def _golden_rows(name):
    rows = []
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.strip()
            if line and not line.startswith("#"):
                rows.append([int(x) for x in line.split()])
    return rows


def _rand_qkv(rng, n, hq, hkv, d):
    return (rng.standard_normal((n, hq, d)), rng.standard_normal((n, hkv, d)),
            rng.standard_normal((n, hkv, d)))


# --------------------------------------------------------------------------------------
# ring / online recurrence
# --------------------------------------------------------------------------------------
def _worked_example_inputs():
    """Inputs of the worked example on the ring-attention simulation page (section "The
    whole algorithm, simulated"): 16 tokens, head dim 8, numpy default_rng(0), with Q, K
    and V drawn in that order as standard normals and stored as float32."""
    rng = np.random.default_rng(0)
    return tuple(rng.normal(size=(16, 8)).astype(np.float32) for _ in range(3))


def test_worked_example_ring_equals_full_attention_f32():
    g = _golden_kv("ring_worked_example.txt")
    Q, K, V = _worked_example_inputs()
    assert Q.shape == (int(g["tokens"]), int(g["head_dim"]))
    P = int(g["devices"])
    O, _ = ring.ring_forward(Q[:, None, :], K[:, None, :], V[:, None, :], None, P=P,
                             dtype=np.float32)
    # the oracle's own dense softmax attention, evaluated in float32 like the page's reference
    ref = attention.forward(Q[:, None, :], K[:, None, :], V[:, None, :],
                            np.ones((16, 16), bool), dtype=np.float32)[0][:, 0, :]
    diff = float(np.abs(O[:, 0, :] - ref).max())
    page = float(g["max_difference"])
    # same arithmetic in float32: the page's figure is one or two ulp-scale roundings
    assert diff <= 1e-6
    assert abs(diff - page) <= 1e-6
    assert np.allclose(O[:, 0, :], ref, atol=float(g["allclose_atol"])) == (g["allclose"] == "True")
    # the fp64 ring agrees with fp64 dense to rounding
    O64, _ = ring.ring_forward(Q[:, None, :], K[:, None, :], V[:, None, :], None, P=P)
    ref64, _ = attention.forward(Q[:, None, :], K[:, None, :], V[:, None, :],
                                 np.ones((16, 16), bool))
    assert np.abs(O64 - ref64).max() < 1e-13


@pytest.mark.parametrize("P", [1, 2, 4, 8, 16])
def test_ring_fp64_equals_dense_any_P_and_step_order(P):
    rng = np.random.default_rng(7)
    n = 256
    tr = wl.random_pack(rng, n)
    M = mask.dense_mask(tr, INF)
    q, k, v = _rand_qkv(rng, n, 4, 2, 16)
    O, L = attention.forward(q, k, v, M)
    Or, Lr = ring.ring_forward(q, k, v, M, P=P)
    assert np.abs(Or - O).max() < 1e-12
    fin = np.isfinite(L)
    assert (np.isfinite(Lr) == fin).all()
    assert np.abs(Lr[fin] - L[fin]).max() < 1e-12
    order = [list(rng.permutation(P)) for _ in range(P)]
    Or2, Lr2 = ring.ring_forward(q, k, v, M, P=P, step_order=order)
    assert np.abs(Or2 - O).max() < 1e-12
    assert np.abs(Lr2[fin] - L[fin]).max() < 1e-12


def test_ring_with_window_mask_and_plan_order():
    rng = np.random.default_rng(3)
    n = 1024
    tr = wl.random_pack(rng, n)
    W = 200
    pl = plan.make_plan(tr, W, 4, "ptrr_block")
    trp = pl.tracks_perm
    Mp = mask.dense_mask(trp, W)
    q, k, v = _rand_qkv(rng, n, 2, 2, 8)
    Or, Lr = ring.ring_forward(q[pl.perm], k[pl.perm], v[pl.perm], Mp, P=4)
    O, L = attention.forward(q, k, v, mask.dense_mask(tr, W))
    assert np.abs(Or - O[pl.perm]).max() < 1e-12
    fin = np.isfinite(L[:, pl.perm])
    assert np.abs(Lr[fin] - L[:, pl.perm][fin]).max() < 1e-12


def test_fully_masked_rows_give_zero_output_and_neg_inf_lse():
    # W = 0 and causal tokens: the causal test 0 <= dp < 0 never holds, so a causal
    # token sees nothing; a bidirectional span still sees its own span.
    samples = [[wl.Span("causal", 5), wl.Span("full", 4)], [wl.Span("causal", 3)]]
    tr = wl.tracks_from_samples(samples)
    n = 12
    M = mask.dense_mask(tr, 0)
    assert not M[:5].any() and not M[9:].any() and M[5:9, 5:9].all()
    rng = np.random.default_rng(0)
    q, k, v = _rand_qkv(rng, n, 2, 1, 4)
    O, L = attention.forward(q, k, v, M)
    assert (O[:5] == 0).all() and (O[9:] == 0).all()
    assert np.isneginf(L[:, :5]).all() and np.isneginf(L[:, 9:]).all()
    Or, Lr = ring.ring_forward(q[:12], k[:12], v[:12], M, P=4)
    assert (Or[:5] == 0).all() and np.isneginf(Lr[:, 9:]).all()
    # the live rows equal attention restricted to the bidirectional span
    O2, _ = attention.forward(q[5:9], k[5:9], v[5:9], np.ones((4, 4), bool))
    assert np.abs(O[5:9] - O2).max() < 1e-13
    # and their gradients vanish where no key is legal
    do = rng.standard_normal(q.shape)
    dq, dk, dv, _, _ = attention.backward(q, k, v, do, M)
    assert (dq[:5] == 0).all() and (dk[:5] == 0).all() and (dv[9:] == 0).all()


def test_uniform_scores_closed_form():
    # K = 0 makes every legal score 0: softmax is uniform over the legal keys, so
    # O_q = mean of V over them and LSE_q = ln(number of legal keys).
    rng = np.random.default_rng(1)
    n = 300
    tr = wl.random_pack(rng, n)
    M = mask.dense_mask(tr, 37)
    q, _, v = _rand_qkv(rng, n, 2, 2, 8)
    k = np.zeros_like(v)
    O, L = attention.forward(q, k, v, M)
    cnt = M.sum(1)
    for h in range(2):
        want = (M.astype(float) @ v[:, h, :]) / np.maximum(cnt, 1)[:, None]
        assert np.abs(O[:, h, :] - want).max() < 1e-12
        assert np.abs(L[h][cnt > 0] - np.log(cnt[cnt > 0])).max() < 1e-12


def test_single_legal_key_closed_form():
    # W = 1 on causal tokens: each query sees only itself -> O_q = V_q, LSE = q.k_q/sqrt(d)
    n, d = 64, 8
    tr = wl.tracks_from_samples([[wl.Span("causal", n)]])
    M = mask.dense_mask(tr, 1)
    assert (M == np.eye(n, dtype=bool)).all()
    rng = np.random.default_rng(2)
    q, k, v = _rand_qkv(rng, n, 4, 2, d)
    O, L = attention.forward(q, k, v, M)
    for h in range(4):
        kh = h // 2
        assert np.abs(O[:, h, :] - v[:, kh, :]).max() < 1e-13
        s = (q[:, h, :] * k[:, kh, :]).sum(1) / math.sqrt(d)
        assert np.abs(L[h] - s).max() < 1e-13


def test_gqa_head_grouping():
    # q heads 2 and 3 must read kv head 1; zero its keys -> those heads become uniform.
    rng = np.random.default_rng(5)
    n = 40
    M = np.tril(np.ones((n, n), bool))
    q, k, v = _rand_qkv(rng, n, 4, 2, 8)
    k[:, 1, :] = 0
    O, L = attention.forward(q, k, v, M)
    cnt = np.arange(1, n + 1)
    for h in (2, 3):
        assert np.abs(L[h] - np.log(cnt)).max() < 1e-12
        assert np.abs(O[:, h, :] - np.cumsum(v[:, 1, :], 0) / cnt[:, None]).max() < 1e-12
    for h in (0, 1):
        assert np.abs(L[h] - np.log(cnt)).max() > 1e-3


def test_backward_matches_finite_differences():
    rng = np.random.default_rng(11)
    samples = [[wl.Span("causal", 6), wl.Span("full", 5), wl.Span("noise", 3),
                wl.Span("causal", 4)], [wl.Span("group", 3, 0), wl.Span("causal", 2),
                                        wl.Span("group", 3, 0)]]
    tr = wl.tracks_from_samples(samples)
    n = 26
    M = mask.dense_mask(tr, 5)
    q, k, v = _rand_qkv(rng, n, 2, 1, 4)
    do = rng.standard_normal(q.shape)

    def loss(q_, k_, v_):
        O, _ = attention.forward(q_, k_, v_, M)
        return float((O * do).sum())

    dq, dk, dv, _, _ = attention.backward(q, k, v, do, M)
    eps = 1e-6
    for X, G in ((q, dq), (k, dk), (v, dv)):
        for idx in [tuple(rng.integers(0, s) for s in X.shape) for _ in range(25)]:
            Xp = X.copy()
            Xm = X.copy()
            Xp[idx] += eps
            Xm[idx] -= eps
            args_p = [Xp if Y is X else Y for Y in (q, k, v)]
            args_m = [Xm if Y is X else Y for Y in (q, k, v)]
            num = (loss(*args_p) - loss(*args_m)) / (2 * eps)
            assert abs(num - G[idx]) < 1e-7 * max(1.0, abs(num)), (idx, num, G[idx])


def test_permuting_tokens_with_their_tracks_permutes_the_output():
    rng = np.random.default_rng(4)
    n = 200
    tr = wl.random_pack(rng, n)
    perm = rng.permutation(n)
    trp = {k: np.asarray(v)[perm] for k, v in tr.items()}
    trp["pos"] = perm
    q, k, v = _rand_qkv(rng, n, 2, 1, 8)
    O, L = attention.forward(q, k, v, mask.dense_mask(tr, 50))
    Op, Lp = attention.forward(q[perm], k[perm], v[perm], mask.dense_mask(trp, 50))
    assert np.abs(Op - O[perm]).max() < 1e-12


# --------------------------------------------------------------------------------------
# mask semantics
# --------------------------------------------------------------------------------------
def _span_semantics(samples, W):
    """Legality from the mode table of the MARBLE post (section 01) and its prose, per
    pair, written without the four-track predicate: within a span by its mode; a later
    span reads an earlier one unless the earlier one is a noise span; spans of one group
    read each other in both directions; the window limits causal distance only; no
    pair crosses samples."""
    spans = []  # (sample, index in sample, start, end, mode, group)
    t = 0
    for si, s in enumerate(samples):
        for ji, sp in enumerate(s):
            spans.append((si, ji, t, t + sp.length, sp.mode, sp.group))
            t += sp.length
    n = t
    owner = np.empty(n, np.int64)
    for i, (_, _, a, b, _, _) in enumerate(spans):
        owner[a:b] = i
    out = np.zeros((n, n), bool)
    for qi in range(n):
        A = spans[owner[qi]]
        for ki in range(n):
            B = spans[owner[ki]]
            if A[0] != B[0]:
                continue
            dp = qi - ki
            if owner[qi] == owner[ki]:
                ok = (0 <= dp < W) if A[4] == "causal" else True
            elif A[4] == "group" and B[4] == "group" and A[5] == B[5]:
                ok = True
            elif B[3] <= A[2]:  # key span lies before the query span
                ok = B[4] != "noise" and dp < W
            else:
                ok = False
            out[qi, ki] = ok
    return out


@pytest.mark.parametrize("seed", range(6))
def test_mask_equals_span_semantics_brute_force(seed):
    rng = np.random.default_rng(100 + seed)
    samples = wl.random_samples(rng, 160)
    tr = wl.tracks_from_samples(samples)
    for W in (INF, 1, 7, 40):
        assert (mask.dense_mask(tr, W) == _span_semantics(samples, W)).all()


def test_mask_hand_derived_cases():
    S = wl.Span
    samples = [[S("causal", 4), S("noise", 3), S("causal", 2)],            # 0..8
               [S("group", 2, 0), S("causal", 2), S("group", 2, 0)],       # 9..14
               [S("full", 3), S("causal", 2)]]                             # 15..19
    tr = wl.tracks_from_samples(samples)
    M = mask.dense_mask(tr, INF)
    assert M[5, 0] and M[5, 6] and M[4, 6]          # noise span: sees prompt and itself
    assert not M[7, 4] and not M[8, 6]               # later text cannot see the noise span
    assert M[7, 3] and not M[3, 7]                   # causal text
    assert M[9, 13] and M[13, 9]                     # group: earlier frame sees later frame
    assert not M[9, 11] and M[13, 11]                # ... but not the text between them
    assert M[15, 17] and M[17, 15] and M[18, 17] and not M[17, 18]
    assert not M[9, 8] and not M[15, 14] and not M[0, 19]   # never across samples
    Mw = mask.dense_mask(tr, 2)
    assert Mw[3, 2] and Mw[3, 3] and not Mw[3, 1]    # last W tokens, the query included
    assert Mw[15, 17] and Mw[9, 13]                  # spans are not cut by the window


# --------------------------------------------------------------------------------------
# legal-pair counts (Libra Eq. 2, Eq. 6)
# --------------------------------------------------------------------------------------
def test_legal_pairs_closed_forms():
    lens = [300, 17, 1024, 5, 256]
    causal = wl.tracks_from_samples([[wl.Span("causal", L)] for L in lens])
    bidi = wl.tracks_from_samples([[wl.Span("full", L)] for L in lens])
    want_c = sum(L * (L + 1) // 2 for L in lens)
    want_b = sum(L * L for L in lens)
    assert counts.by_brute_force(causal, INF) == want_c
    assert counts.by_key_classes(causal, INF) == want_c
    assert counts.by_brute_force(bidi, INF) == want_b
    assert counts.by_key_classes(bidi, INF) == want_b
    # Libra Eq. 6 per block of query rows
    rows = mask.dense_mask(causal, INF).sum(1)
    n = len(rows)
    per_block = rows[: n // 128 * 128].reshape(-1, 128).sum(1)
    assert (counts.causal_block_rows(lens)[: n // 128] == per_block).all()


def test_legal_pairs_config1_and_config3():
    tr1 = wl.config_tracks(1)
    want1 = 768 * 769 // 2 + 1024 ** 2 + 256 * 257 // 2
    assert want1 == 1376768
    assert counts.by_brute_force(tr1, INF) == want1
    assert counts.by_key_classes(tr1, INF) == want1
    tr3 = wl.config_tracks(3)
    N, W = 262144, 4096
    want3 = W * (W + 1) // 2 + (N - W) * W
    assert want3 == 1065355264
    assert counts.by_key_classes(tr3, W) == want3


@pytest.mark.parametrize("seed", range(5))
def test_legal_pair_counters_agree(seed):
    rng = np.random.default_rng(seed)
    tr = wl.random_pack(rng, 700)
    for W in (INF, 1, 33):
        assert counts.by_key_classes(tr, W) == counts.by_brute_force(tr, W)
        assert (counts.per_row_by_key_classes(tr, W) == mask.dense_mask(tr, W).sum(1)).all()


# --------------------------------------------------------------------------------------
# tile map
# --------------------------------------------------------------------------------------
def test_tile_map_config1_exact():
    tr = wl.config_tracks(1)
    T = plan.classify(plan.block_summaries(tr), INF)
    assert (T == plan.FULL).sum() == 80
    assert (T == plan.PARTIAL).sum() == 8
    assert (T == plan.EMPTY).sum() == 168
    # sample A = blocks 0..5 (causal): partial diagonal, full below
    for a in range(6):
        assert T[a, a] == plan.PARTIAL
        assert all(T[a, b] == plan.FULL for b in range(a))
        assert all(T[a, b] == plan.EMPTY for b in range(a + 1, 16))
    assert (T[6:14, 6:14] == plan.FULL).all()
    assert T[14, 14] == T[15, 15] == plan.PARTIAL and T[15, 14] == plan.FULL


def test_tile_map_config3_structure():
    tr = wl.config_tracks(3)
    summ = plan.block_summaries(tr)
    rows = np.array([0, 1, 31, 32, 33, 500, 2047])
    T = plan.classify(summ, 4096, rows)
    for i, b in enumerate(rows):
        full = set(np.flatnonzero(T[i] == plan.FULL))
        part = set(np.flatnonzero(T[i] == plan.PARTIAL))
        assert full == set(range(max(0, b - 31), b))
        assert part == ({b, b - 32} if b >= 32 else {b})


@pytest.mark.parametrize("seed", range(4))
def test_tile_map_is_sound_by_brute_force(seed):
    rng = np.random.default_rng(50 + seed)
    n = 128 * 12
    tr = wl.random_pack(rng, n, max_samples=3)
    for W in (INF, 100, 300):
        T = plan.classify(plan.block_summaries(tr), W)
        M = mask.dense_mask(tr, W)
        for a in range(12):
            for b in range(12):
                blk = M[a * 128:(a + 1) * 128, b * 128:(b + 1) * 128]
                if T[a, b] == plan.FULL:
                    assert blk.all()
                elif T[a, b] == plan.EMPTY:
                    assert not blk.any()


# --------------------------------------------------------------------------------------
# order, step lists, needed index
# --------------------------------------------------------------------------------------
def test_ptrr_reproduces_zigzag():
    tr = wl.tracks_from_samples([[wl.Span("causal", 8 * 128)]])
    pl = plan.make_plan(tr, INF, 4, "ptrr_block")
    gold = _golden_rows("zigzag_p4.txt")
    for dev, a, b, work in gold:
        blocks = sorted(pl.block_perm[dev * 2:(dev + 1) * 2].tolist())
        assert blocks == sorted([a, b])
        assert int(pl.cost[blocks].sum()) == work


def test_contiguous_causal_imbalance():
    tr = wl.tracks_from_samples([[wl.Span("causal", 4 * 128)]])
    pl = plan.make_plan(tr, INF, 4, "contiguous")
    Wm = plan.shard_work(pl)
    for dev, blocks in _golden_rows("causal_contiguous_p4.txt"):
        assert Wm[dev].sum() == blocks
        assert (Wm[dev, : dev + 1] == 1).all() and (Wm[dev, dev + 1:] == 0).all()


def test_ptrr_chunk_units_and_tie_break():
    # equal costs: ties are broken by ascending unit index
    assert plan.ptrr_assign([5, 5, 5, 5], 2) == [[0, 3], [1, 2]]
    assert plan.ptrr_assign([1, 2, 3, 4, 5, 6], 3) == [[0, 5], [1, 4], [2, 3]]
    tr = wl.tracks_from_samples([[wl.Span("causal", 16 * 128)]])
    pl = plan.make_plan(tr, INF, 2, "ptrr_chunk", chunk_tokens=512)
    # 4 chunks of 4 blocks, causal costs grow with the chunk index: ranks {3,0}, {2,1}
    assert pl.block_perm.tolist() == [0, 1, 2, 3, 12, 13, 14, 15, 4, 5, 6, 7, 8, 9, 10, 11]


def test_needed_index_config3():
    tr = wl.config_tracks(3)
    pl = plan.make_plan(tr, 4096, 16, "contiguous")
    sizes = np.diff(pl.needed_ptr)
    assert sizes[0] == 128 and (sizes[1:] == 160).all()
    r = 5
    assert pl.needed[pl.needed_ptr[r]:pl.needed_ptr[r + 1]].tolist() == list(
        range(128 * r - 32, 128 * r + 128))


@pytest.mark.parametrize("order", ["contiguous", "ptrr_block", "ptrr_chunk"])
def test_step_lists_partition_the_tile_map(order):
    rng = np.random.default_rng(9)
    n = 128 * 32
    tr = wl.random_pack(rng, n, max_samples=4)
    P = 4
    pl = plan.make_plan(tr, 700, P, order, chunk_tokens=512)
    nb = pl.nb
    T = plan.classify(plan.block_summaries(tr), 700)
    bps = nb // P
    seen = np.zeros((nb, nb), np.int8)
    for nq in range(nb):
        for j in range(P):
            a, b = pl.step_ptr[nq * P + j], pl.step_ptr[nq * P + j + 1]
            cols = pl.step_col[a:b]
            assert (np.diff(cols) > 0).all() and ((cols // bps) == j).all()
            seen[nq, cols] = pl.step_tag[a:b]
    assert (seen == T[np.ix_(pl.block_perm, pl.block_perm)]).all()
    seenT = np.zeros((nb, nb), np.int8)
    for nk in range(nb):
        for r in range(P):
            a, b = pl.colT_ptr[nk * P + r], pl.colT_ptr[nk * P + r + 1]
            rows = pl.colT_row[a:b]
            assert (np.diff(rows) > 0).all() and ((rows // bps) == r).all()
            seenT[rows, nk] = pl.colT_tag[a:b]
    assert (seenT == seen).all()
    for r in range(P):
        want = np.flatnonzero(seen[r * bps:(r + 1) * bps].any(0))
        assert pl.needed[pl.needed_ptr[r]:pl.needed_ptr[r + 1]].tolist() == want.tolist()
    # permuted tracks carry the original positions
    assert (pl.tracks_perm["pos"] == pl.perm).all()
    assert (pl.tracks_perm["sample"] == tr["sample"][pl.perm]).all()


# --------------------------------------------------------------------------------------
# sampled-row / sampled-column oracle paths agree with the dense oracle
# --------------------------------------------------------------------------------------
@pytest.mark.parametrize("seed,W,pos", [(21, 120, False), (22, INF, False), (23, 0, False),
                                        (24, 1, False), (25, 300, True), (26, INF, True)])
def test_sampled_rows_and_columns_equal_dense(seed, W, pos):
    # the sampled paths score each token against a superset of its legal partners (window
    # and span members, or the whole sample with a position track): they must agree with
    # the dense oracle for every window, including none, W = 0 and W = 1
    rng = np.random.default_rng(seed)
    n = 900
    tr = wl.random_pack(rng, n, max_samples=4)
    if pos:
        tr = dict(tr, pos=np.arange(n, dtype=np.int32))
    M = mask.dense_mask(tr, W)
    q, k, v = _rand_qkv(rng, n, 4, 2, 8)
    do = rng.standard_normal(q.shape)
    dq, dk, dv, O, L = attention.backward(q, k, v, do, M)
    rows = np.sort(rng.choice(n, 200, replace=False))
    O2, L2 = attention.rows_forward(q, k, v, tr, W, rows)
    assert np.abs(O2 - O[rows]).max() < 1e-12
    fin = np.isfinite(L[:, rows])
    assert (np.isfinite(L2) == fin).all() and np.abs(L2[fin] - L[:, rows][fin]).max() < 1e-12
    dq2 = attention.rows_dq(q, k, v, do, tr, W, rows)
    assert np.abs(dq2 - dq[rows]).max() < 1e-10
    cols = np.sort(rng.choice(n, 60, replace=False))
    dk2, dv2 = attention.cols_backward(q, k, v, do, tr, W, cols)
    assert np.abs(dk2 - dk[cols]).max() < 1e-10
    assert np.abs(dv2 - dv[cols]).max() < 1e-10
    dk3, dv3 = attention.cols_backward(q, k, v, do, tr, W, cols, kv_heads=[1])
    assert np.abs(dk3[:, 0] - dk[cols, 1]).max() < 1e-10


def test_round_bf16_ties_and_library_conversion():
    # bfloat16 keeps 7 stored mantissa bits: at 1 the spacing is 2^-7, so 1 + 2^-8 is a tie
    # that goes to the even neighbour 1, and 1 + 3 * 2^-8 ties up to 1 + 2^-6
    x = np.array([1 + 2.0**-8, 1 + 3 * 2.0**-8, -(1 + 2.0**-8), 1 + 2.0**-8 + 2.0**-20,
                  0.0, -0.0, np.inf, -np.inf, 3.40e38])
    r = ring.round_bf16(x)
    assert r[0] == 1.0 and r[1] == 1 + 2.0**-6 and r[2] == -1.0 and r[3] == 1 + 2.0**-7
    assert r[4] == 0.0 and np.signbit(r[5]) and r[6] == np.inf and r[7] == -np.inf
    assert r[8] == np.inf  # past the midpoint between the largest finite bfloat16 (about 3.3895e38) and 2^128
    torch = pytest.importorskip("torch")
    rng = np.random.default_rng(5)
    y = rng.standard_normal(20000) * 10.0 ** rng.integers(-30, 30, 20000)
    lib = torch.from_numpy(y.astype(np.float32)).to(torch.bfloat16).to(torch.float64).numpy()
    assert np.array_equal(ring.round_bf16(y), lib)


def test_bf16_merge_without_rounding_is_exact_attention():
    # with the identity in place of both roundings, the log-sum-exp merge of normalised
    # partials is an exact identity: the result equals dense attention for any P and order
    rng = np.random.default_rng(11)
    n = 256
    tr = wl.random_pack(rng, n)
    M = mask.dense_mask(tr, 96)
    q, k, v = _rand_qkv(rng, n, 4, 2, 16)
    O, L = attention.forward(q, k, v, M)
    fin = np.isfinite(L)
    for P in (1, 2, 8):
        order = [list(rng.permutation(P)) for _ in range(P)]
        Ob, Lb = ring.ring_forward_bf16_merge(q, k, v, M, P=P, step_order=order,
                                              rounding=lambda x: x)
        assert np.abs(Ob - O).max() < 1e-12
        assert (np.isfinite(Lb) == fin).all()
        assert np.abs(Lb[fin] - L[fin]).max() < 1e-12


def test_bf16_merge_single_step_is_rounded_exact_output():
    # P = 1: one partial (rounded once) merged into the empty state (weight 1, rounded again,
    # which leaves a bf16 value unchanged)
    rng = np.random.default_rng(12)
    n = 128
    tr = wl.random_pack(rng, n)
    M = mask.dense_mask(tr, INF)
    q, k, v = _rand_qkv(rng, n, 2, 2, 16)
    O, L = attention.forward(q, k, v, M)
    Ob, Lb = ring.ring_forward_bf16_merge(q, k, v, M, P=1)
    assert np.array_equal(Ob, ring.round_bf16(O))
    fin = np.isfinite(L)
    assert np.abs(Lb[fin] - L[fin]).max() < 1e-12


def test_bf16_merge_two_steps_by_hand():
    # one row, one head, two keys in two shards of one token each: the merge written out
    q = np.array([[[0.3, -1.2]], [[0.0, 0.0]]])
    k = np.array([[[1.1, 0.4]], [[-0.7, 2.0]]])
    v = np.array([[[0.123456, -2.5]], [[1.75, 0.333333]]])
    Ob, Lb = ring.ring_forward_bf16_merge(q, k, v, None, P=2, step_order=[[0, 1], [1, 0]],
                                          scale=1.0)
    s0 = 0.3 * 1.1 - 1.2 * 0.4
    s1 = 0.3 * -0.7 - 1.2 * 2.0
    lse = math.log(math.exp(s0) + math.exp(s1))
    o0 = ring.round_bf16(v[0, 0])          # step 1: the partial is V of key 0, lse_1 = s0
    o1 = ring.round_bf16(v[1, 0])          # step 2: V of key 1, lse_2 = s1
    want = ring.round_bf16(o0 * math.exp(s0 - lse) + o1 * math.exp(s1 - lse))
    assert np.array_equal(Ob[0, 0], want)
    assert abs(Lb[0, 0] - lse) < 1e-14


def test_bf16_merge_masked_rows_and_error_gap():
    rng = np.random.default_rng(13)
    n = 512
    tr = wl.random_pack(rng, n)
    M = mask.dense_mask(tr, INF)
    M[:3] = False  # rows with no legal key at all
    q, k, v = _rand_qkv(rng, n, 2, 2, 32)
    O, L = attention.forward(q, k, v, M)
    Ob, Lb = ring.ring_forward_bf16_merge(q, k, v, M, P=8)
    assert (Ob[:3] == 0).all() and np.isneginf(Lb[:, :3]).all()
    # bf16 rounding after every step costs more than one rounding of the exact result
    e_once = np.abs(ring.round_bf16(O) - O).mean()
    e_merge = np.abs(Ob - O).mean()
    assert e_merge > 1.2 * e_once


def test_fp32_merge_is_exact_to_fp32_rounding():
    # fp32 partials merged in fp32: the error against fp64 attention is a few fp32 ulps of
    # the output, far below one bf16 rounding, for any P and step order
    rng = np.random.default_rng(14)
    n = 512
    tr = wl.random_pack(rng, n)
    M = mask.dense_mask(tr, INF)
    q, k, v = _rand_qkv(rng, n, 2, 2, 32)
    O, L = attention.forward(q, k, v, M)
    fin = np.isfinite(L)
    for P in (1, 4, 16):
        order = [list(rng.permutation(P)) for _ in range(P)]
        Of, Lf = ring.ring_forward_fp32_merge(q, k, v, M, P=P, step_order=order)
        assert np.abs(Of - O).max() < 8 * 2.0**-24 * max(1.0, np.abs(O).max())
        assert np.abs(Lf[fin] - L[fin]).max() < 1e-12
    assert ring.round_f32(1 + 2.0**-24) == 1.0 and ring.round_f32(1 + 3 * 2.0**-24) == 1 + 2.0**-22


def test_layout_step_cost_by_hand_and_brute_force():
    # P = 2, one chunk per rank: W = Wc, steps s = 0 (diagonal) and s = 1 (off-diagonal)
    Wc = np.array([[5, 7], [2, 9]])
    assert plan.layout_step_cost(Wc, [0, 1], 2) == max(5, 9) + max(7, 2)
    assert plan.layout_step_cost(Wc, [1, 0], 2) == max(9, 5) + max(2, 7)
    rng = np.random.default_rng(20)
    for P in (2, 3, 4):
        K = 3 * P
        Wc = rng.integers(0, 1000, (K, K))
        rank = rng.permutation(np.repeat(np.arange(P), 3))
        Wr = [[sum(int(Wc[a, b]) for a in range(K) for b in range(K)
                   if rank[a] == r and rank[b] == j) for j in range(P)] for r in range(P)]
        want = sum(max(Wr[r][(r - s) % P] for r in range(P)) for s in range(P))
        assert plan.layout_step_cost(Wc, rank, P) == want


def _search_case(seed, nblocks=64, P=4):
    rng = np.random.default_rng(seed)
    tr = wl.random_pack(rng, nblocks * 128, max_samples=5)
    return tr, plan.block_pair_counts(tr, INF), P


@pytest.mark.parametrize("seed", [0, 1, 2])
def test_chunk_search_is_a_local_optimum_below_both_starts(seed):
    tr, Wb, P = _search_case(seed)
    assert Wb.sum() == counts.by_brute_force(tr, INF)
    C, k, rank, cost = plan.chunk_search(Wb, P, tau=1000)
    K = k * P
    assert C == cost + 1000 * P * k
    assert sorted(np.bincount(rank, minlength=P)) == [k] * P
    cs = Wb.shape[0] // K
    Wc = Wb.reshape(K, cs, K, cs).sum(axis=(1, 3))
    assert plan.layout_step_cost(Wc, rank, P) == cost
    # no single swap between ranks lowers the step cost
    for a in range(K):
        for b in range(a + 1, K):
            if rank[a] != rank[b]:
                r2 = rank.copy()
                r2[a], r2[b] = r2[b], r2[a]
                assert plan.layout_step_cost(Wc, r2, P) >= cost
    # and it is no worse than either PTRR start
    for costs in (Wc.sum(axis=1), np.zeros(K)):
        r0 = np.empty(K, np.int64)
        for r, units in enumerate(plan.ptrr_assign(costs, P)):
            r0[units] = r
        assert cost <= plan.layout_step_cost(Wc, r0, P)


def test_chunk_search_range_cost_trades_chunks():
    tr, Wb, P = _search_case(3)
    # no per-range cost: the best step cost over all chunk counts; a huge one: one chunk
    C0, k0, _, cost0 = plan.chunk_search(Wb, P, tau=0)
    assert C0 == cost0
    C1, k1, _, _ = plan.chunk_search(Wb, P, tau=10**12)
    assert k1 == 1
    # uniform work (one bidirectional sample): every layout costs P * (nb / P)^2 * 128^2
    samples = [[wl.Span("full", 64 * 128)]]
    tru = wl.tracks_from_samples(samples)
    Wu = plan.block_pair_counts(tru, INF)
    assert (Wu == 128 * 128).all()
    Cu, ku, _, costu = plan.chunk_search(Wu, 4, tau=0)
    assert costu == 4 * 16 * 16 * 128 * 128 and ku == 1


def test_chunk_search_plan_realises_the_searched_cost():
    # the plan built from the search's layout has exactly the searched step cost when its
    # shard work is summed in legal pairs from its own step lists
    tr, Wb, P = _search_case(4)
    tau = 5000
    C, k, rank, cost = plan.chunk_search(Wb, P, tau)
    pl = plan.make_plan(tr, INF, P, "chunk_search", range_cost=tau)
    nb, bps = pl.nb, pl.nb // P
    Wr = np.zeros((P, P), np.int64)
    for nq in range(nb):
        for j in range(P):
            for e in range(pl.step_ptr[nq * P + j], pl.step_ptr[nq * P + j + 1]):
                Wr[nq // bps, j] += Wb[pl.block_perm[nq], pl.block_perm[pl.step_col[e]]]
    assert sum(max(Wr[r, (r - s) % P] for r in range(P)) for s in range(P)) == cost
    # each rank holds k contiguous chunks, ascending
    cs = nb // (k * P)
    chunks = pl.block_perm.reshape(-1, cs)
    assert (np.diff(chunks, axis=1) == 1).all() and (chunks[:, 0] % cs == 0).all()
    for r in range(P):
        mine = chunks[r * k:(r + 1) * k, 0] // cs
        assert (np.diff(mine) > 0).all() and (rank[mine] == r).all()


def test_key_intervals_closed_forms():
    # one sample: causal text of 300, a bidirectional span of 200, a noise span of 100, then
    # causal text of 424; positions are indices
    samples = [[wl.Span("causal", 300), wl.Span("full", 200), wl.Span("noise", 100),
                wl.Span("causal", 424)]]
    tr = wl.tracks_from_samples(samples)
    n = 1024
    W = INF
    lo, hi, ex = plan.key_intervals(tr, W)
    assert ex.all()
    k = np.arange(n)
    # causal keys: themselves up to the end of the sample, except that the noise span [500, 600)
    # sees clean keys too, so the range stays [k, n)
    for kk in (0, 17, 299, 600, 1023):
        assert (lo[kk], hi[kk]) == (kk, n)
    # bidirectional span keys: from the span start to the end of the sample
    for kk in (300, 399, 499):
        assert (lo[kk], hi[kk]) == (300, n)
    # noise keys: only the noise span itself
    for kk in (500, 550, 599):
        assert (lo[kk], hi[kk]) == (500, 600)
    # a window of 50: causal keys see [k, k + 50), span keys at least their span
    lo, hi, ex = plan.key_intervals(tr, 50)
    assert ex.all() and (lo[10], hi[10]) == (10, 60) and (lo[310], hi[310]) == (300, 500)
    assert (lo[480], hi[480]) == (300, 530)


def test_key_intervals_group_is_not_contiguous():
    # image group of two spans with text between: a key of the second image is seen by the
    # first image (same group) but not by the text between them
    samples = [[wl.Span("causal", 128), wl.Span("group", 128, 0), wl.Span("causal", 128),
                wl.Span("group", 128, 0), wl.Span("causal", 128)]]
    tr = wl.tracks_from_samples(samples)
    lo, hi, ex = plan.key_intervals(tr, INF)
    assert not ex[384:512].any() and (lo[400], hi[400]) == (128, 640)
    assert ex[:384].all() and ex[512:].all()
    assert list(plan.interval_blocks(ex)) == [True, True, True, False, True]
    # W = 0: a causal key is seen by nobody
    lo, hi, ex = plan.key_intervals(tr, 0)
    assert (lo[5], hi[5]) == (0, 0) and ex[5]


@pytest.mark.parametrize("seed", range(3))
def test_key_intervals_reproduce_the_mask(seed):
    # where exact, the interval test equals the mask on every pair
    rng = np.random.default_rng(70 + seed)
    n = 512
    tr = wl.random_pack(rng, n, max_samples=4)
    W = [INF, 64, 300][seed]
    lo, hi, ex = plan.key_intervals(tr, W)
    M = mask.dense_mask(tr, W)
    q = np.arange(n)[:, None]
    test = (q >= lo[None, :]) & (q < hi[None, :])
    assert (test[:, ex] == M[:, ex]).all()
    assert (M[:, ~ex] & ~test[:, ~ex]).sum() == 0  # the interval always covers the visible set


def test_vision_group_layout_by_hand_and_contiguity():
    # T0 G1a T1 G1b T2 G2a T3 G2b: text first, then the group spans last first
    L = 40
    samples = [[wl.Span("causal", L), wl.Span("group", L, 1), wl.Span("causal", L),
                wl.Span("group", L, 1), wl.Span("causal", L), wl.Span("group", L, 2),
                wl.Span("causal", L), wl.Span("group", L, 2)],
               [wl.Span("causal", 16), wl.Span("full", 24)]]
    tr = wl.tracks_from_samples(samples)
    perm = plan.vision_group_layout(tr)
    T = [np.arange(i * L, (i + 1) * L) for i in range(8)]
    want = np.concatenate([T[0], T[2], T[4], T[6], T[7], T[5], T[3], T[1],
                           np.arange(8 * L, 8 * L + 40)])
    assert np.array_equal(perm, want)
    trp = plan.apply_layout(tr, perm)
    n = len(perm)
    # the mask is the same mask, read in the new order
    assert np.array_equal(mask.dense_mask(trp, INF), mask.dense_mask(tr, INF)[np.ix_(perm, perm)])
    # before: keys of later group spans see a broken range; after: every key's is one range
    _, _, ex0 = plan.key_intervals(tr, INF)
    _, _, ex1 = plan.key_intervals(trp, INF)
    assert not ex0.all() and ex1.all()


def test_vision_group_layout_is_identity_without_groups():
    rng = np.random.default_rng(31)
    tr = wl.tracks_from_samples(wl.packed_mix_samples(rng, 4096))
    assert np.array_equal(plan.vision_group_layout(tr), np.arange(4096))
