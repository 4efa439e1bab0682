"""fp64 masked attention and its gradients, written from the plain definition.

Libra paper, section 2.2, Eq. 1: CoreAttn(Q, K, V; M) = softmax(QK^T / sqrt(d_h) + M) V,
with M = 0 on legal pairs and -inf elsewhere (the mask is the MARBLE packed mask).
LSE is the natural log of the softmax denominator of each row.  A row with no legal key
has output 0 and LSE = -inf.

Backward (standard softmax calculus; MARBLE post section 03 "Exact ring attention
accumulation" runs it against the final LSE):
    P = exp(S - LSE),  dV = P^T dO,  dP = dO V^T,  D = rowsum(dO * O),
    dS = P * (dP - D),  dQ = dS K / sqrt(d),  dK = dS^T Q / sqrt(d).

Grouped-query attention: q head h reads kv head h // (Hq / Hkv); gradients of a kv head
are summed over its q heads.
"""
from __future__ import annotations

import math

import numpy as np

from .mask import allowed, sample_runs


def _f64(x):
    try:
        import torch
        if isinstance(x, torch.Tensor):
            return x.detach().to("cpu", torch.float64).numpy()
    except ImportError:  # pragma: no cover
        pass
    return np.asarray(x, np.float64)


def _group(hq, hkv):
    if hq % hkv:
        raise ValueError("Hq must be a multiple of Hkv")
    return hq // hkv


def forward(q, k, v, mask, scale=None, dtype=np.float64):
    """q [Nq, Hq, d], k/v [Nk, Hkv, d], mask [Nq, Nk] bool -> O [Nq, Hq, d], LSE [Hq, Nq]."""
    q, k, v = (_f64(x).astype(dtype) for x in (q, k, v))
    nq, hq, d = q.shape
    g = _group(hq, k.shape[1])
    scale = dtype(1.0 / math.sqrt(d)) if scale is None else dtype(scale)
    O = np.zeros((nq, hq, d), dtype)
    LSE = np.full((hq, nq), -np.inf, dtype)
    for h in range(hq):
        kh = h // g
        S = (q[:, h, :] @ k[:, kh, :].T) * scale
        S = np.where(mask, S, -np.inf)
        m = S.max(axis=1)
        has = np.isfinite(m)
        E = np.exp(S - np.where(has, m, 0)[:, None])
        l = E.sum(axis=1)
        O[:, h, :] = np.where(has[:, None], (E @ v[:, kh, :]) / np.where(has, l, 1)[:, None], 0)
        LSE[h] = np.where(has, m + np.log(np.where(has, l, 1)), -np.inf)
    return O, LSE


def backward(q, k, v, do, mask, scale=None):
    """Gradients (dQ, dK, dV) plus (O, LSE) of the masked attention above, in fp64."""
    q, k, v, do = (_f64(x) for x in (q, k, v, do))
    nq, hq, d = q.shape
    g = _group(hq, k.shape[1])
    scale = 1.0 / math.sqrt(d) if scale is None else scale
    O, LSE = forward(q, k, v, mask, scale)
    dq = np.zeros_like(q)
    dk = np.zeros_like(k)
    dv = np.zeros_like(v)
    for h in range(hq):
        kh = h // g
        S = (q[:, h, :] @ k[:, kh, :].T) * scale
        fin = np.isfinite(LSE[h])
        P = np.where(mask & fin[:, None], np.exp(S - np.where(fin, LSE[h], 0)[:, None]), 0.0)
        dv[:, kh, :] += P.T @ do[:, h, :]
        dP = do[:, h, :] @ v[:, kh, :].T
        D = (do[:, h, :] * O[:, h, :]).sum(axis=1)
        dS = P * (dP - D[:, None])
        dq[:, h, :] = (dS @ k[:, kh, :]) * scale
        dk[:, kh, :] += (dS.T @ q[:, h, :]) * scale
    return dq, dk, dv, O, LSE


# --------------------------------------------------------------------------------------
# sampled rows / columns for packs too large for the dense oracle
# --------------------------------------------------------------------------------------
def _partners(tr, W, idx, a, b, keys_of_queries):
    """Tokens of the sample run [a, b) that may be legal partners of any token of idx
    (inside the run): keys of those queries (keys_of_queries) or queries of those keys.

    The result is a superset of the legal partners, which the predicate then decides.  A
    pair is legal only if it is causal (0 <= pos_q - pos_k < W) or in one span (seg_q ==
    seg_k >= 0), the MARBLE post's section 01 predicate.  With positions equal to indices
    (no position track), a partner outside the causal window of every token of idx and
    outside their spans fails both terms and is illegal whatever the other terms say, so it
    can be left out.  With a position track the whole run is returned."""
    if "pos" in tr:
        return np.arange(a, b)
    run = b - a
    w = int(min(W, run))
    cover = np.zeros(run + 1, np.int64)
    if w > 0:
        i = np.asarray(idx, np.int64) - a
        if keys_of_queries:  # the keys of query t: (t - w, t]
            lo, hi = np.maximum(i - w + 1, 0), i + 1
        else:                # the queries of key t: [t, t + w)
            lo, hi = i, np.minimum(i + w, run)
        np.add.at(cover, lo, 1)
        np.add.at(cover, hi, -1)
    inside = np.cumsum(cover[:-1]) > 0
    seg = np.asarray(tr["seg"])
    spans = np.unique(seg[np.asarray(idx, np.int64)])
    spans = spans[spans >= 0]
    if len(spans):
        inside |= np.isin(seg[a:b], spans)
    return a + np.flatnonzero(inside)


def _by_run(tr, idx, chunk=512, reach=8192):
    """Positions into idx grouped by sample run, in chunks of at most `chunk` tokens that
    lie within `reach` of the chunk's first one (so that a chunk's partners stay few):
    yields (run start, run end, positions)."""
    idx = np.asarray(idx, np.int64)
    st, en = sample_runs(tr)
    starts = st[idx]
    for a in np.unique(starts):
        sel_all = np.flatnonzero(starts == a)
        sel_all = sel_all[np.argsort(idx[sel_all], kind="stable")]
        b = int(en[idx[sel_all[0]]])
        c0 = 0
        while c0 < len(sel_all):
            c1 = c0 + 1
            while (c1 < len(sel_all) and c1 - c0 < chunk and
                   idx[sel_all[c1]] - idx[sel_all[c0]] < reach):
                c1 += 1
            yield int(a), b, sel_all[c0:c1]
            c0 = c1


def rows_forward(q, k, v, tr, W, rows, heads=None, scale=None):
    """Exact O and LSE for selected query tokens (original order).

    Keys outside a query's sample run fail same_sample, so only that run is scored, and
    within it only the partners _partners cannot rule out.  q/k/v may be torch tensors or
    arrays in original token order.
    Returns O [len(rows), len(heads), d], LSE [len(heads), len(rows)]."""
    rows = np.asarray(rows, np.int64)
    hq = q.shape[1]
    g = _group(hq, k.shape[1])
    heads = np.arange(hq) if heads is None else np.asarray(heads)
    d = q.shape[2]
    scale = 1.0 / math.sqrt(d) if scale is None else scale
    O = np.zeros((len(rows), len(heads), d))
    LSE = np.full((len(heads), len(rows)), -np.inf)
    for a, b, sel in _by_run(tr, rows):
        kk = _partners(tr, W, rows[sel], a, b, keys_of_queries=True)
        if len(kk) == 0:
            continue  # no key can be legal: O = 0, LSE = -inf as initialised
        ks = _f64(k[kk])
        vs = _f64(v[kk])
        m = allowed(tr, W, rows[sel][:, None], kk[None, :])
        qs = _f64(q[rows[sel]])
        for hi, h in enumerate(heads):
            kh = h // g
            S = (qs[:, h, :] @ ks[:, kh, :].T) * scale
            S = np.where(m, S, -np.inf)
            mx = S.max(axis=1)
            has = np.isfinite(mx)
            E = np.exp(S - np.where(has, mx, 0)[:, None])
            l = E.sum(axis=1)
            O[sel, hi, :] = np.where(has[:, None],
                                     (E @ vs[:, kh, :]) / np.where(has, l, 1)[:, None], 0)
            LSE[hi, sel] = np.where(has, mx + np.log(np.where(has, l, 1)), -np.inf)
    return O, LSE


def _grad_block(qs, ks, vs, dos, O, lse, m, scale):
    """The backward of one head on a block of query rows x key columns, exactly as in
    backward() above: P = exp(S - LSE) on legal pairs of rows with a finite LSE,
    dS = P * (dP - D).  Returns (dS, P)."""
    fin = np.isfinite(lse)
    S = (qs @ ks.T) * scale
    P = np.where(m & fin[:, None], np.exp(S - np.where(fin, lse, 0)[:, None]), 0.0)
    dP = dos @ vs.T
    D = (dos * O).sum(axis=1)
    return P * (dP - D[:, None]), P


def cols_backward(q, k, v, do, tr, W, cols, kv_heads=None, scale=None):
    """Exact dK and dV for selected key tokens (original order) and kv heads.

    For each key, every query of its sample run that may attend it contributes; those
    queries' LSE and D = rowsum(dO * O) come from full rows (rows_forward).
    Returns dK, dV [len(cols), len(kv_heads), d]."""
    cols = np.asarray(cols, np.int64)
    hq, hkv, d = q.shape[1], k.shape[1], q.shape[2]
    g = _group(hq, hkv)
    kv_heads = np.arange(hkv) if kv_heads is None else np.asarray(kv_heads)
    scale = 1.0 / math.sqrt(d) if scale is None else scale
    heads = np.array([h for kh in kv_heads for h in range(kh * g, (kh + 1) * g)])
    dK = np.zeros((len(cols), len(kv_heads), d))
    dV = np.zeros((len(cols), len(kv_heads), d))
    for a, b, sel in _by_run(tr, cols):
        qq = _partners(tr, W, cols[sel], a, b, keys_of_queries=False)
        m = allowed(tr, W, qq[:, None], cols[sel][None, :])
        live = m.any(axis=1)
        qq, m = qq[live], m[live]
        if len(qq) == 0:
            continue
        O, LSE = rows_forward(q, k, v, tr, W, qq, heads=heads, scale=scale)
        qs, dos = _f64(q[qq]), _f64(do[qq])
        kc, vc = _f64(k[cols[sel]]), _f64(v[cols[sel]])
        for ki, kh in enumerate(kv_heads):
            for j in range(g):
                h = kh * g + j
                hi = ki * g + j
                dS, P = _grad_block(qs[:, h, :], kc[:, kh, :], vc[:, kh, :], dos[:, h, :],
                                    O[:, hi, :], LSE[hi], m, scale)
                dV[sel, ki] += P.T @ dos[:, h, :]
                dK[sel, ki] += (dS.T @ qs[:, h, :]) * scale
    return dK, dV


def rows_dq(q, k, v, do, tr, W, rows, heads=None, scale=None):
    """Exact dQ for selected query tokens: dQ_t = scale * sum_k P[t,k](dP[t,k] - D_t) K_k."""
    rows = np.asarray(rows, np.int64)
    hq = q.shape[1]
    g = _group(hq, k.shape[1])
    heads = np.arange(hq) if heads is None else np.asarray(heads)
    d = q.shape[2]
    scale = 1.0 / math.sqrt(d) if scale is None else scale
    O, LSE = rows_forward(q, k, v, tr, W, rows, heads=heads, scale=scale)
    dQ = np.zeros((len(rows), len(heads), d))
    for a, b, sel in _by_run(tr, rows):
        kk = _partners(tr, W, rows[sel], a, b, keys_of_queries=True)
        if len(kk) == 0:
            continue
        m = allowed(tr, W, rows[sel][:, None], kk[None, :])
        ks, vs = _f64(k[kk]), _f64(v[kk])
        qs, dos = _f64(q[rows[sel]]), _f64(do[rows[sel]])
        for hi, h in enumerate(heads):
            kh = h // g
            dS, _ = _grad_block(qs[:, h, :], ks[:, kh, :], vs[:, kh, :], dos[:, h, :],
                                O[sel, hi, :], LSE[hi, sel], m, scale)
            dQ[sel, hi] = (dS @ ks[:, kh, :]) * scale
    return dQ
