"""Legal-pair counters.

The effective-FLOP numerator counts legal (unmasked) query/key pairs.  Libra paper,
section 2.3, Eq. 2: the attention workload of a pack is proportional to sum_j l_j^2
(causal factor absorbed); Eq. 6 counts the causal pairs of the query rows of one block as
sum over intersected samples of sum_{q=a}^{e-1} (q + 1) with sample-local positions.

Two independent counters of the MARBLE packed mask:
  * ``by_brute_force`` evaluates the mask on every pair of every sample (small packs);
  * ``by_key_classes`` counts, for each query, the legal keys of each class of keys
    sharing (seg, noise) inside its sample with a sorted-position search, using the
    mask's structure (same span -> whole class, otherwise the causal window).
"""
from __future__ import annotations

import numpy as np

from .mask import allowed, sample_runs, tracks_with_pos


def by_brute_force(tr, W) -> int:
    st, en = sample_runs(tr)
    total = 0
    for a in np.unique(st):
        b = int(en[a])
        idx = np.arange(int(a), b)
        for c0 in range(0, len(idx), 2048):
            rows = idx[c0:c0 + 2048]
            total += int(allowed(tr, W, rows[:, None], idx[None, :]).sum())
    return total


def per_row_by_key_classes(tr, W) -> np.ndarray:
    """Legal keys of every query token (int64 [N])."""
    sample, seg, noise, pos = tracks_with_pos(tr)
    st, en = sample_runs(tr)
    W = np.int64(W)
    cnt = np.zeros(len(sample), np.int64)
    for a in np.unique(st):
        b = int(en[a])
        sl = slice(int(a), b)
        g_q, n_q, p_q = seg[sl], noise[sl], pos[sl]
        classes = np.unique(np.stack([seg[sl], noise[sl]], 1), axis=0)
        for gk, nk in classes:
            members = np.flatnonzero((seg[sl] == gk) & (noise[sl] == nk))
            pk = np.sort(pos[sl][members])
            keep = (nk < 0) | (n_q == nk)
            same = (g_q == gk) & (gk >= 0)
            in_win = (np.searchsorted(pk, p_q, side="right")
                      - np.searchsorted(pk, p_q - W, side="right"))
            cnt[sl] += np.where(keep, np.where(same, len(pk), in_win), 0)
    return cnt


def by_key_classes(tr, W) -> int:
    return int(per_row_by_key_classes(tr, W).sum())


def causal_block_rows(lengths, block=128) -> np.ndarray:
    """Libra Eq. 6 for a pack of purely causal samples: per block of query rows, the sum
    over the samples it intersects of (sample-local position + 1) over its rows."""
    lengths = list(lengths)
    n = sum(lengths)
    local = np.concatenate([np.arange(L) for L in lengths])
    nb = (n + block - 1) // block
    out = np.zeros(nb, np.int64)
    for b in range(nb):
        out[b] = int((local[b * block:(b + 1) * block] + 1).sum())
    return out
