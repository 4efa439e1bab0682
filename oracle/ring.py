"""Ring simulation: queries of shard r meet the KV shards one step at a time while the
unnormalised state (O, m, l) is carried between steps.

RingAttention tutorial page, "The Online Softmax Formulation": for a new block j with
scores S_j, the running maximum becomes m_new = max(m, rowmax S_j); the old state is
rescaled by exp(m - m_new); the new block adds exp(S_j - m_new) to l and exp(S_j - m_new) V_j
to O.  Only the end divides O by l.  "Execution Algorithm" (same page) and the MARBLE
post (section 03): at step s, shard r meets KV shard (r - s) mod P.

A row that has met no legal key yet keeps m = -inf; its rescale factor is taken as 1
(O and l are still 0), never exp(-inf - (-inf)).
"""
from __future__ import annotations

import math

import numpy as np

from .attention import _f64, _group


def ring_forward(q, k, v, mask=None, P=4, step_order=None, scale=None, dtype=np.float64,
                 return_state=False):
    """Simulated ring over P contiguous shards of the given token order.

    q [N, Hq, d], k/v [N, Hkv, d]; mask [N, N] bool or None (all legal).
    step_order[r] is the sequence of kv shards that q shard r visits (default (r - s) mod P).
    Returns (O, LSE) or, with return_state, the raw (O_acc, m, l) per token/head."""
    q, k, v = (_f64(x).astype(dtype) for x in (q, k, v))
    n, hq, d = q.shape
    if n % P:
        raise ValueError("N must be divisible by P")
    g = _group(hq, k.shape[1])
    S_ = n // P
    scale = dtype(1.0 / math.sqrt(d)) if scale is None else dtype(scale)
    if step_order is None:
        step_order = [[(r - s) % P for s in range(P)] for r in range(P)]
    Oacc = np.zeros((n, hq, d), dtype)
    m = np.full((hq, n), -np.inf, dtype)
    l = np.zeros((hq, n), dtype)
    for r in range(P):
        qs = slice(r * S_, (r + 1) * S_)
        for j in step_order[r]:
            ks = slice(j * S_, (j + 1) * S_)
            blk = None if mask is None else mask[qs, ks]
            for h in range(hq):
                kh = h // g
                s = (q[qs, h, :] @ k[ks, kh, :].T) * scale
                if blk is not None:
                    s = np.where(blk, s, -np.inf)
                m_old = m[h, qs]
                m_new = np.maximum(m_old, s.max(axis=1))
                live = np.isfinite(m_new)
                base = np.where(live, m_new, 0).astype(dtype)
                alpha = np.where(live, np.exp(m_old - base), 1).astype(dtype)
                p = np.exp(s - base[:, None])
                l[h, qs] = alpha * l[h, qs] + p.sum(axis=1)
                Oacc[qs, h, :] = alpha[:, None] * Oacc[qs, h, :] + p @ v[ks, kh, :]
                m[h, qs] = m_new
    if return_state:
        return Oacc, m, l
    has = l > 0
    O = np.where(has.T[:, :, None], Oacc / np.where(has, l, 1).T[:, :, None], 0)
    LSE = np.where(has, m + np.log(np.where(has, l, 1)), -np.inf)
    return O.astype(dtype), LSE.astype(dtype)


def dense_unmasked_f32(q, k, v):
    """Single-device float32 softmax attention without a mask (one head), for the
    worked example of the ring simulation page: subtract the row max, exponentiate,
    normalise, multiply by V."""
    q, k, v = (np.asarray(x, np.float32) for x in (q, k, v))
    s = (q @ k.T) * np.float32(1.0 / np.sqrt(q.shape[1]))
    s = s - s.max(axis=1, keepdims=True)
    e = np.exp(s)
    return (e / e.sum(axis=1, keepdims=True)) @ v


def worked_example_inputs():
    """Inputs of the ring simulation page's worked example: 16 tokens, head dim 8,
    numpy default_rng(0), Q, K, V drawn in that order as standard normals -> float32."""
    rng = np.random.default_rng(0)
    Q, K, V = (rng.normal(size=(16, 8)).astype(np.float32) for _ in range(3))
    return Q, K, V
