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


def round_bf16(x):
    """Round to the nearest bfloat16 (ties to even), returned as float64: the value goes to
    float32 first (a CUDA kernel holds it in fp32), then keeps the top 16 bits of its
    encoding after round-to-nearest-even on the lower 16 (the bfloat16 format: 8 exponent
    bits, 7 stored mantissa bits)."""
    f = np.asarray(x, np.float64).astype(np.float32)
    u = f.view(np.uint32).astype(np.uint64)
    finite = np.isfinite(f)
    r = ((u + 0x7FFF + ((u >> 16) & 1)) & 0xFFFF0000).astype(np.uint32)
    out = np.where(finite, r.view(np.float32), f)
    return out.astype(np.float64)


def ring_forward_bf16_merge(q, k, v, mask=None, P=4, step_order=None, scale=None,
                            rounding=round_bf16):
    """Standard ring attention, the baseline MARBLE post section 03 ("Exact ring attention
    accumulation") measures against: every step runs one attention over the step's keys and
    emits a normalised partial output rounded to bf16 plus its log-sum-exp; the running
    output is merged with it by a log-sum-exp rescale and rounded to bf16 again.

    Per row and head, with running (O, lse) starting at (0, -inf) and a step's legal scores s:
      lse_s = max s + ln sum exp(s - max s),  O_s = round(sum softmax(s) V)
      lse'  = ln(exp(lse) + exp(lse_s)),      O'  = round(O exp(lse - lse') + O_s exp(lse_s - lse'))
    A step with no legal key for the row leaves it unchanged.  fp64 between roundings;
    `rounding` is the rounding applied at both points (bf16 by default).  Returns (O, LSE)."""
    q, k, v = (_f64(x) for x in (q, k, v))
    n, hq, d = q.shape
    if n % P:
        raise ValueError("N must be divisible by P")
    g = _group(hq, k.shape[1])
    S_ = n // P
    scale = 1.0 / math.sqrt(d) if scale is None else float(scale)
    if step_order is None:
        step_order = [[(r - s) % P for s in range(P)] for r in range(P)]
    O = np.zeros((n, hq, d))
    lse = np.full((hq, n), -np.inf)
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
                mx = s.max(axis=1)
                live = np.isfinite(mx)
                base = np.where(live, mx, 0.0)
                e = np.exp(s - base[:, None])
                l_s = e.sum(axis=1)
                O_s = rounding((e @ v[ks, kh, :]) / np.where(live, l_s, 1.0)[:, None])
                lse_s = np.where(live, base + np.log(np.where(live, l_s, 1.0)), -np.inf)
                lse_old = lse[h, qs]
                lse_new = np.logaddexp(lse_old, lse_s)
                w_old = np.where(np.isfinite(lse_old), np.exp(lse_old - np.where(live | np.isfinite(lse_old), lse_new, 0.0)), 0.0)
                w_new = np.where(live, np.exp(lse_s - np.where(live, lse_new, 0.0)), 0.0)
                merged = rounding(O[qs, h, :] * w_old[:, None] + O_s * w_new[:, None])
                O[qs, h, :] = np.where(live[:, None], merged, O[qs, h, :])
                lse[h, qs] = np.where(live, lse_new, lse_old)
    return O, lse


def round_f32(x):
    """Round to the nearest float32 (ties to even), returned as float64."""
    return np.asarray(x, np.float64).astype(np.float32).astype(np.float64)


def ring_forward_fp32_merge(q, k, v, mask=None, P=4, step_order=None, scale=None):
    """The same per-step merge with fp32 in place of bf16 at both rounding points: every
    call's output is an fp32 partial with its LSE and the partials are merged in fp32, the
    route to exactness the MARBLE post gives for Blackwell's split-KV partials (section 03,
    "Exact ring attention accumulation"; section 06).  Returns (O, LSE)."""
    return ring_forward_bf16_merge(q, k, v, mask, P=P, step_order=step_order, scale=scale,
                                   rounding=round_f32)
