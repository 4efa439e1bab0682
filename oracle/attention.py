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
def rows_forward(q, k, v, tr, W, rows, heads=None, scale=None):
    """Exact O and LSE for selected query tokens (original order).

    Keys outside a query's sample run fail same_sample, so only that run is scored.
    q/k/v may be torch tensors or arrays in original token order.
    Returns O [len(rows), len(heads), d], LSE [len(heads), len(rows)]."""
    rows = np.asarray(rows, np.int64)
    hq = q.shape[1]
    g = _group(hq, k.shape[1])
    heads = np.arange(hq) if heads is None else np.asarray(heads)
    d = q.shape[2]
    scale = 1.0 / math.sqrt(d) if scale is None else scale
    st, en = sample_runs(tr)
    O = np.zeros((len(rows), len(heads), d))
    LSE = np.full((len(heads), len(rows)), -np.inf)
    # group rows by sample run
    keys = st[rows]
    for a in np.unique(keys):
        sel_all = np.flatnonzero(keys == a)
        b = int(en[rows[sel_all[0]]])
        kk = np.arange(int(a), b)
        ks = _f64(k[int(a):b])
        vs = _f64(v[int(a):b])
        for c0 in range(0, len(sel_all), 512):
            sel = sel_all[c0:c0 + 512]
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
    st, en = sample_runs(tr)
    # all queries that can see any selected key
    need = []
    vis = []
    for c in cols:
        qq = np.arange(int(st[c]), int(en[c]))
        ok = allowed(tr, W, qq, int(c))
        vis.append(qq[ok])
        need.append(qq[ok])
    allq = np.unique(np.concatenate(need)) if need else np.zeros(0, np.int64)
    heads = np.array([h for kh in kv_heads for h in range(kh * g, (kh + 1) * g)])
    O, LSE = rows_forward(q, k, v, tr, W, allq, heads=heads, scale=scale)
    idx = {int(t): i for i, t in enumerate(allq)}
    qa = _f64(q[allq]) if len(allq) else np.zeros((0, hq, d))
    da = _f64(do[allq]) if len(allq) else np.zeros((0, hq, d))
    dK = np.zeros((len(cols), len(kv_heads), d))
    dV = np.zeros((len(cols), len(kv_heads), d))
    for ci, c in enumerate(cols):
        rows_i = np.array([idx[int(t)] for t in vis[ci]], np.int64)
        if len(rows_i) == 0:
            continue
        kc = _f64(k[int(c)])
        vc = _f64(v[int(c)])
        for ki, kh in enumerate(kv_heads):
            for j in range(g):
                h = kh * g + j
                hi = ki * g + j
                qs = qa[rows_i, h, :]
                s = (qs @ kc[kh]) * scale
                p = np.exp(s - LSE[hi, rows_i])
                dos = da[rows_i, h, :]
                dV[ci, ki] += p @ dos
                dp = dos @ vc[kh]
                D = (dos * O[rows_i, hi, :]).sum(axis=1)
                ds = p * (dp - D)
                dK[ci, ki] += (ds @ qs) * scale
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
    st, en = sample_runs(tr)
    dQ = np.zeros((len(rows), len(heads), d))
    for ri, t in enumerate(rows):
        a, b = int(st[t]), int(en[t])
        kk = np.arange(a, b)
        m = allowed(tr, W, int(t), kk)
        ks = _f64(k[a:b])[m]
        vs = _f64(v[a:b])[m]
        qt = _f64(q[int(t)])
        dot = _f64(do[int(t)])
        for hi, h in enumerate(heads):
            kh = h // g
            if not np.isfinite(LSE[hi, ri]):
                continue
            s = (ks[:, kh, :] @ qt[h]) * scale
            p = np.exp(s - LSE[hi, ri])
            dp = vs[:, kh, :] @ dot[h]
            D = float(dot[h] @ O[ri, hi])
            dQ[ri, hi] = ((p * (dp - D)) @ ks[:, kh, :]) * scale
    return dQ
