"""The packed-mask predicate, written out from its definition.

MARBLE post, section 01 "Packed multimodal masks": a query q may attend a key k iff

    (causal(q, k) or same_span(q, k)) and keep_noise(q, k) and same_sample(q, k)

with causal = 0 <= pos[q] - pos[k] < W (W infinite on globally causal layers),
same_span = seg[q] == seg[k] >= 0, keep_noise = noise[k] < 0 or noise[q] == noise[k],
same_sample = sample[q] == sample[k].  ``pos`` is the original position (the token's index
in the pack before any reordering).
"""
from __future__ import annotations

import numpy as np


def tracks_with_pos(tr):
    """Return (sample, seg, noise, pos) as int64 arrays; pos defaults to the index."""
    n = len(tr["sample"])
    pos = tr.get("pos")
    if pos is None:
        pos = np.arange(n, dtype=np.int64)
    return (np.asarray(tr["sample"], np.int64), np.asarray(tr["seg"], np.int64),
            np.asarray(tr["noise"], np.int64), np.asarray(pos, np.int64))


def allowed(tr, W, q, k):
    """Boolean mask for index arrays q, k (broadcast against each other)."""
    sample, seg, noise, pos = tracks_with_pos(tr)
    dp = pos[q] - pos[k]
    causal = (dp >= 0) & (dp < W)
    same_span = (seg[q] == seg[k]) & (seg[q] >= 0)
    keep_noise = (noise[k] < 0) | (noise[q] == noise[k])
    same_sample = sample[q] == sample[k]
    return (causal | same_span) & keep_noise & same_sample


def dense_mask(tr, W, rows=None, cols=None):
    """Explicit [len(rows), len(cols)] boolean mask (all tokens by default)."""
    n = len(tr["sample"])
    rows = np.arange(n) if rows is None else np.asarray(rows)
    cols = np.arange(n) if cols is None else np.asarray(cols)
    return allowed(tr, W, rows[:, None], cols[None, :])


def sample_runs(tr):
    """Per token, [start, end) of the maximal run of equal sample ids containing it.

    Used to restrict per-row evaluation to one sample: when each sample occupies one run
    (true of every pack here), every key outside the run fails same_sample and is illegal
    by the definition above."""
    s = np.asarray(tr["sample"])
    n = len(s)
    change = np.flatnonzero(s[1:] != s[:-1]) + 1
    starts = np.concatenate([[0], change])
    ends = np.concatenate([change, [n]])
    run = np.zeros(n, np.int64)
    run[change] = 1
    run = np.cumsum(run)
    return starts[run], ends[run]
