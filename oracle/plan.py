"""Oracle planner: block summaries, tile classes, PTRR order, per-step lists, needed index.

Sources (MARBLE post):
  * section 03 "Block classification": per 128-token block, the min and max of every
    metadata track plus a small bitmap of the segments the block holds; a block pair is
    *full* if every pair is provably legal, *empty* if every pair is provably illegal,
    *partial* otherwise.  One test per block pair.
  * section 03 "PTRR": sort query blocks by cost, deal them to ranks in rounds of R with
    every other round reversed, keep each rank's blocks in sequence order.
  * section 03 "Chunked ring attention": PTRR's rule applied to contiguous chunks, and the
    layout search over the number of chunks per rank that minimises the layout cost
    C = sum_s max_r W[r, (r - s) mod R] + tau * R * k (W in legal pairs).
  * section 03 "Block classification" (ring steps): at step s, rank r pairs its queries
    with the key/value shard of rank (r - s) mod R.
  * section 04 "Sparse all-to-all": each rank needs exactly the key/value blocks its
    queries can see (local blocks included; one pass over local + fetched keys).
  * section 04 "Layout transforms": tokens are permuted once, carrying their metadata
    and original position.

The exact summary test is not printed on the page; the reading used here (and by the
CUDA planner, written separately) is:

  per block X: Slo/Shi (sample), Plo/Phi (pos), Nlo/Nhi (noise), over tokens with seg >= 0
  Glo/Ghi, hasseg (any seg >= 0), allseg (all seg >= 0), Gbits = OR of 1 << (seg mod 64).

  For q block A and k block B:
    samp_all   = Slo_A == Shi_A == Slo_B == Shi_B
    samp_none  = Shi_A < Slo_B  or  Shi_B < Slo_A
    caus_all   = Plo_A - Phi_B >= 0  and  Phi_A - Plo_B < W
    caus_none  = Phi_A - Plo_B < 0   or   Plo_A - Phi_B >= W
    span_all   = allseg_A and allseg_B and Glo_A == Ghi_A == Glo_B == Ghi_B
    span_none  = not hasseg_A or not hasseg_B or (Gbits_A & Gbits_B) == 0
                 or Ghi_A < Glo_B or Ghi_B < Glo_A
    noise_all  = Nhi_B < 0  or  Nlo_A == Nhi_A == Nlo_B == Nhi_B >= 0
    noise_none = Nlo_B >= 0 and (Nhi_A < Nlo_B or Nhi_B < Nlo_A)

    empty = samp_none or noise_none or (caus_none and span_none)
    full  = samp_all and noise_all and (caus_all or span_all)      (when not empty)
    partial otherwise.

The oracle evaluates the rule on all nb x nb block pairs (no candidate band).
"""
from __future__ import annotations

import dataclasses
from typing import Dict, List

import numpy as np

from .mask import dense_mask, tracks_with_pos

BLOCK = 128
EMPTY, FULL, PARTIAL = 0, 1, 2
NO_SEG_LO = 2**31 - 1
NO_SEG_HI = -1


def block_summaries(tr) -> Dict[str, np.ndarray]:
    sample, seg, noise, pos = tracks_with_pos(tr)
    n = len(sample)
    if n % BLOCK:
        raise ValueError("n must be a multiple of 128")
    nb = n // BLOCK
    S = sample.reshape(nb, BLOCK)
    P = pos.reshape(nb, BLOCK)
    N = noise.reshape(nb, BLOCK)
    G = seg.reshape(nb, BLOCK)
    has = G >= 0
    glo = np.where(has, G, NO_SEG_LO).min(1)
    ghi = np.where(has, G, NO_SEG_HI).max(1)
    bits = np.zeros(nb, np.uint64)
    for b in range(nb):
        for g in np.unique(G[b][has[b]]):
            bits[b] |= np.uint64(1) << np.uint64(int(g) & 63)
    return {
        "slo": S.min(1), "shi": S.max(1),
        "plo": P.min(1), "phi": P.max(1),
        "nlo": N.min(1), "nhi": N.max(1),
        "glo": glo, "ghi": ghi,
        "hasseg": has.any(1), "allseg": has.all(1),
        "gbits": bits,
    }


def classify(summ, W, rows=None) -> np.ndarray:
    """Tile class matrix [len(rows), nb] (0 empty, 1 full, 2 partial) by the rule above."""
    nb = len(summ["slo"])
    rows = np.arange(nb) if rows is None else np.asarray(rows)
    A = {k: v[rows][:, None] for k, v in summ.items()}
    B = {k: v[None, :] for k, v in summ.items()}
    W = np.int64(W)

    samp_all = (A["slo"] == A["shi"]) & (A["shi"] == B["slo"]) & (B["slo"] == B["shi"])
    samp_none = (A["shi"] < B["slo"]) | (B["shi"] < A["slo"])
    caus_all = (A["plo"] - B["phi"] >= 0) & (A["phi"] - B["plo"] < W)
    caus_none = (A["phi"] - B["plo"] < 0) | (A["plo"] - B["phi"] >= W)
    span_all = (A["allseg"] & B["allseg"] & (A["glo"] == A["ghi"]) & (A["ghi"] == B["glo"])
                & (B["glo"] == B["ghi"]))
    span_none = ((~A["hasseg"]) | (~B["hasseg"]) | ((A["gbits"] & B["gbits"]) == 0)
                 | (A["ghi"] < B["glo"]) | (B["ghi"] < A["glo"]))
    noise_all = (B["nhi"] < 0) | ((A["nlo"] == A["nhi"]) & (A["nhi"] == B["nlo"])
                                  & (B["nlo"] == B["nhi"]) & (B["nhi"] >= 0))
    noise_none = (B["nlo"] >= 0) & ((A["nhi"] < B["nlo"]) | (B["nhi"] < A["nlo"]))

    empty = samp_none | noise_none | (caus_none & span_none)
    full = samp_all & noise_all & (caus_all | span_all) & ~empty
    out = np.full(empty.shape, PARTIAL, np.int8)
    out[empty] = EMPTY
    out[full] = FULL
    return out


def tile_csr(summ, W, row_chunk: int = 512):
    """Global tile map in original block coordinates as CSR (row_ptr int64, col int32,
    tag uint8 with 1 = full, 2 = partial; empty tiles are not stored)."""
    nb = len(summ["slo"])
    ptr = np.zeros(nb + 1, np.int64)
    cols: List[np.ndarray] = []
    tags: List[np.ndarray] = []
    for a in range(0, nb, row_chunk):
        rows = np.arange(a, min(nb, a + row_chunk))
        c = classify(summ, W, rows)
        for i, r in enumerate(rows):
            nz = np.flatnonzero(c[i])
            cols.append(nz.astype(np.int32))
            tags.append(c[i][nz].astype(np.uint8))
            ptr[r + 1] = len(nz)
    ptr = np.cumsum(ptr)
    col = np.concatenate(cols) if cols else np.zeros(0, np.int32)
    tag = np.concatenate(tags) if tags else np.zeros(0, np.uint8)
    return ptr, col, tag


# --------------------------------------------------------------------------------------
# token order
# --------------------------------------------------------------------------------------
def ptrr_assign(cost, P):
    """PTRR over units with the given costs.

    Sort by (cost descending, unit index ascending); the t-th round of P units goes to
    ranks 0..P-1 when t is even and P-1..0 when t is odd; each rank then keeps its units
    in ascending index order.  Returns the list of units of each rank."""
    cost = np.asarray(cost)
    U = len(cost)
    if U % P:
        raise ValueError("number of units must be divisible by P")
    order = sorted(range(U), key=lambda u: (-int(cost[u]), u))
    rank = np.empty(U, np.int64)
    for p, u in enumerate(order):
        t, i = divmod(p, P)
        rank[u] = i if t % 2 == 0 else P - 1 - i
    return [[u for u in range(U) if rank[u] == r] for r in range(P)]


@dataclasses.dataclass
class Plan:
    nb: int
    P: int
    W: int
    row_ptr: np.ndarray      # global tile CSR, original block coordinates
    col: np.ndarray
    tag: np.ndarray
    cost: np.ndarray         # per original q block: number of non-empty tiles
    block_perm: np.ndarray   # new block -> original block
    inv_block_perm: np.ndarray
    perm: np.ndarray         # new token -> original token
    tracks_perm: Dict[str, np.ndarray]  # sample, seg, noise, pos in new order
    step_ptr: np.ndarray     # [nb*P + 1]; entries of (new q block nq, kv shard j) at nq*P + j
    step_col: np.ndarray     # new kv block
    step_tag: np.ndarray
    colT_ptr: np.ndarray     # [nb*P + 1]; entries of (new kv block nk, q shard r) at nk*P + r
    colT_row: np.ndarray     # new q block
    colT_tag: np.ndarray
    needed_ptr: np.ndarray   # [P + 1]
    needed: np.ndarray       # sorted unique new kv blocks per q shard


def make_plan(tr, W, P, order="contiguous", chunk_tokens=0, range_cost=0) -> Plan:
    summ = block_summaries(tr)
    nb = len(summ["slo"])
    if nb % P:
        raise ValueError("number of blocks must be divisible by P")
    row_ptr, col, tag = tile_csr(summ, W)
    cost = np.diff(row_ptr)

    if order == "contiguous":
        per = nb // P
        units_of_rank = [list(range(r * per, (r + 1) * per)) for r in range(P)]
        unit_blocks = 1
    elif order == "ptrr_block":
        units_of_rank = ptrr_assign(cost, P)
        unit_blocks = 1
    elif order == "ptrr_chunk":
        if chunk_tokens <= 0 or chunk_tokens % BLOCK or (nb * BLOCK) % chunk_tokens:
            raise ValueError("bad chunk size")
        unit_blocks = chunk_tokens // BLOCK
        ccost = cost.reshape(-1, unit_blocks).sum(1)
        units_of_rank = ptrr_assign(ccost, P)
    elif order == "chunk_search":
        _, k, rank, _ = chunk_search(block_pair_counts(tr, W), P, range_cost)
        unit_blocks = nb // (k * P)
        units_of_rank = [[u for u in range(k * P) if rank[u] == r] for r in range(P)]
    else:
        raise ValueError(order)

    block_perm = np.array([u * unit_blocks + i for r in range(P) for u in units_of_rank[r]
                           for i in range(unit_blocks)], np.int64)
    inv = np.empty(nb, np.int64)
    inv[block_perm] = np.arange(nb)
    tok = np.arange(nb * BLOCK)
    perm = block_perm[tok // BLOCK] * BLOCK + tok % BLOCK
    sample, seg, noise, pos = tracks_with_pos(tr)
    tracks_perm = {"sample": sample[perm], "seg": seg[perm], "noise": noise[perm],
                   "pos": pos[perm]}

    bps = nb // P
    # every non-empty tile as (new q block nq, new kv block nk, tag)
    qb_of = np.repeat(np.arange(nb), np.diff(row_ptr))
    nq = inv[qb_of]
    nk = inv[col.astype(np.int64)]

    def grouped(major, minor, shard_of_minor):
        """Lists keyed by (major, shard of minor), each ascending in minor, as CSR over
        major * P + shard."""
        key = major * P + shard_of_minor
        o = np.lexsort((minor, key))
        ptr = np.zeros(nb * P + 1, np.int64)
        ptr[1:] = np.cumsum(np.bincount(key, minlength=nb * P))
        return ptr, minor[o].astype(np.int32), tag[o].astype(np.uint8)

    # forward / dQ: per (q block, kv shard j) the kv blocks of step j
    step_ptr, step_col, step_tag = grouped(nq, nk, nk // bps)
    # dK / dV: per (kv block, q shard r) the q blocks
    colT_ptr, colT_row, colT_tag = grouped(nk, nq, nq // bps)

    # needed kv blocks of each q shard: sorted unique over all its rows' tiles
    pairs = np.unique((nq // bps) * nb + nk)
    needed = (pairs % nb).astype(np.int32)
    needed_ptr = np.zeros(P + 1, np.int64)
    needed_ptr[1:] = np.cumsum(np.bincount(pairs // nb, minlength=P))

    return Plan(nb, P, W, row_ptr, col, tag, cost, block_perm, inv, perm, tracks_perm,
                step_ptr, step_col, step_tag, colT_ptr, colT_row, colT_tag,
                needed_ptr, needed)


def shard_work(plan: Plan) -> np.ndarray:
    """W[r, j] = non-empty tiles between q shard r and kv shard j (tile units)."""
    P, nb = plan.P, plan.nb
    Wm = np.zeros((P, P), np.int64)
    bps = nb // P
    for nq in range(nb):
        for j in range(P):
            Wm[nq // bps, j] += plan.step_ptr[nq * P + j + 1] - plan.step_ptr[nq * P + j]
    return Wm


def step_cost(plan: Plan) -> int:
    """sum over steps s of max over ranks r of W[r, (r - s) mod P] (chunk-layout cost C
    of the chunked-ring section without the per-range overhead term), in tiles."""
    Wm = shard_work(plan)
    P = plan.P
    return int(sum(max(Wm[r, (r - s) % P] for r in range(P)) for s in range(P)))


# --------------------------------------------------------------------------------------
# chunk-layout search (chunked ring attention)
# --------------------------------------------------------------------------------------
CHUNKS_PER_RANK = (1, 2, 4, 8, 16, 32, 64)
MAX_CHUNKS = 1024        # the search skips chunk counts above this many chunks in all
MAX_SWAP_PASSES = 64     # greedy-swap passes per chunk count at most


def block_pair_counts(tr, W) -> np.ndarray:
    """[nb, nb] legal (q, k) pairs between every q block and kv block (original order):
    128 * 128 on full tiles, counted from the explicit mask on partial ones."""
    summ = block_summaries(tr)
    nb = len(summ["slo"])
    row_ptr, col, tag = tile_csr(summ, W)
    out = np.zeros((nb, nb), np.int64)
    for a in range(nb):
        for e in range(row_ptr[a], row_ptr[a + 1]):
            b = int(col[e])
            if tag[e] == 1:
                out[a, b] = BLOCK * BLOCK
            else:
                rows = np.arange(a * BLOCK, (a + 1) * BLOCK)
                cols = np.arange(b * BLOCK, (b + 1) * BLOCK)
                out[a, b] = int(dense_mask(tr, W, rows, cols).sum())
    return out


def layout_step_cost(Wc, rank, P) -> int:
    """sum over steps s of max over ranks r of W[r, (r - s) mod P], where W[r, j] sums the
    chunk-pair work Wc[a, b] over chunks a of rank r and b of rank j (MARBLE post,
    section 03 "Chunked ring attention": the first term of the layout cost C)."""
    rank = np.asarray(rank)
    Wr = np.zeros((P, P), np.int64)
    np.add.at(Wr, (rank[:, None], rank[None, :]), Wc)
    return int(sum(max(Wr[r, (r - s) % P] for r in range(P)) for s in range(P)))


def chunk_search(Wb, P, tau):
    """The chunked ring's layout search (MARBLE post, section 03 "Chunked ring attention"):
    for 1, 2, 4, ..., 64 chunks per rank (chunk counts that divide the blocks evenly and
    stay within MAX_CHUNKS), deal the contiguous chunks to ranks with PTRR's rule once in
    the order of their work (legal pairs of their queries) and once in sequence order,
    start from the layout with the lower step cost (the work order on a tie), then swap
    chunks between ranks whenever that strictly lowers the step cost: passes over the chunk
    pairs (a, b), a < b, in ascending order, first improvement taken, until a pass makes no
    swap (MAX_SWAP_PASSES at most).  The layout costs C = step cost + tau * P * k with k
    chunks per rank; the lowest C wins (the fewer chunks on a tie).

    Wb: [nb, nb] legal pairs between blocks.  Returns (C, k, rank of every chunk,
    step cost)."""
    nb = Wb.shape[0]
    best = None
    for k in CHUNKS_PER_RANK:
        K = k * P
        if K > nb or nb % K or K > MAX_CHUNKS:
            continue
        cs = nb // K
        Wc = Wb.reshape(K, cs, K, cs).sum(axis=(1, 3))
        starts = []
        for costs in (Wc.sum(axis=1), np.zeros(K, np.int64)):
            rank = np.empty(K, np.int64)
            for r, units in enumerate(ptrr_assign(costs, P)):
                rank[units] = r
            starts.append((layout_step_cost(Wc, rank, P), rank))
        cur, rank = starts[0] if starts[0][0] <= starts[1][0] else starts[1]
        rank = rank.copy()
        for _ in range(MAX_SWAP_PASSES):
            swapped = False
            for a in range(K):
                for b in range(a + 1, K):
                    if rank[a] == rank[b]:
                        continue
                    rank[a], rank[b] = rank[b], rank[a]
                    c = layout_step_cost(Wc, rank, P)
                    if c < cur:
                        cur, swapped = c, True
                    else:
                        rank[a], rank[b] = rank[b], rank[a]
            if not swapped:
                break
        C = cur + tau * P * k
        if best is None or C < best[0]:
            best = (C, k, rank.copy(), cur)
    if best is None:
        raise ValueError("no chunk count divides the blocks evenly")
    return best


# --------------------------------------------------------------------------------------
# key intervals
# --------------------------------------------------------------------------------------
def key_intervals(tr, W):
    """Per key k (original order): the smallest interval [lo_k, hi_k) of query indices that
    holds every query allowed to see k, and whether the interval is exact, i.e. every query
    inside it sees k (MARBLE post, section 03: each key's visible queries form one range,
    so a partial tile can test lo_k <= pos_q < hi_k).  A key no query sees gets (0, 0),
    exact.  Queries of other samples never see a key, so each sample is treated alone.
    Returns lo, hi (int64) and exact (bool)."""
    sample = np.asarray(tr["sample"])
    n = len(sample)
    lo = np.zeros(n, np.int64)
    hi = np.zeros(n, np.int64)
    exact = np.ones(n, bool)
    starts = np.flatnonzero(np.r_[True, sample[1:] != sample[:-1]])
    ends = np.r_[starts[1:], n]
    for a, b in zip(starts, ends):
        idx = np.arange(a, b)
        Mk = dense_mask(tr, W, idx, idx)          # [query, key] within the sample
        for j in range(b - a):
            vis = np.flatnonzero(Mk[:, j])
            if len(vis) == 0:
                continue
            lo[a + j] = a + vis[0]
            hi[a + j] = a + vis[-1] + 1
            exact[a + j] = len(vis) == vis[-1] - vis[0] + 1
    return lo, hi, exact


def interval_blocks(exact) -> np.ndarray:
    """Per 128-token block: True if every key of the block has an exact interval."""
    return np.asarray(exact).reshape(-1, BLOCK).all(axis=1)


# --------------------------------------------------------------------------------------
# vision-group layout
# --------------------------------------------------------------------------------------
def vision_group_layout(tr) -> np.ndarray:
    """The vision-group layout transform (MARBLE post, section 04 "Layout transforms"): in
    every sample, first every token outside an image group, in order ("all the text first"),
    then the group's spans, the last span first ("its group spans after in reverse").  An
    image group is a segment id that forms more than one run of consecutive tokens in the
    sample; a span is one such run.  Tokens keep their original positions, so the mask is
    unchanged.  Returns perm: new index -> original index."""
    sample = np.asarray(tr["sample"])
    seg = np.asarray(tr["seg"])
    n = len(sample)
    out = []
    starts = np.flatnonzero(np.r_[True, sample[1:] != sample[:-1]])
    ends = np.r_[starts[1:], n]
    for a, b in zip(starts, ends):
        runs = []                      # (start, end, seg) of every run in the sample
        i = a
        while i < b:
            j = i + 1
            while j < b and seg[j] == seg[i]:
                j += 1
            runs.append((i, j, int(seg[i])))
            i = j
        nruns = {}
        for _, _, g in runs:
            if g >= 0:
                nruns[g] = nruns.get(g, 0) + 1
        grouped = [r for r in runs if r[2] >= 0 and nruns[r[2]] > 1]
        for r in runs:
            if not (r[2] >= 0 and nruns[r[2]] > 1):
                out.extend(range(r[0], r[1]))
        for r in reversed(grouped):
            out.extend(range(r[0], r[1]))
    return np.asarray(out, np.int64)


def apply_layout(tr, perm):
    """Tracks of the permuted pack, each token carrying its original position."""
    sample, seg, noise, pos = tracks_with_pos(tr)
    return {"sample": sample[perm], "seg": seg[perm], "noise": noise[perm], "pos": pos[perm]}
