"""Helpers shared by the GPU tests: run the CUDA path through the Python binding of the
C ABI and bring results back to original token order for comparison with the oracle."""
import numpy as np
import torch

import context_attention_metadata_gb300 as M
import workloads as wl

TOL_O_MAX = 2e-2
TOL_O_MEAN = 2e-3
TOL_LSE = 1e-3
TOL_GRAD_REL = 1e-2


def device_tracks(tr):
    return [torch.as_tensor(np.asarray(tr[k], np.int32)).cuda() for k in ("sample", "seg", "noise")]


def make_plan(tr, W, P, order="contiguous", chunk_tokens=0, range_cost=0):
    s, g, z = device_tracks(tr)
    return M.Plan(s, g, z, W, P, order, chunk_tokens, range_cost=range_cost)


def plan_for(cfg, tr):
    return make_plan(tr, cfg.window, cfg.shards, cfg.order, cfg.chunk_tokens, cfg.range_cost)


def run_forward(pl, q, k, v, needed=False, schedule=None, merge="carried", fused=False):
    """q/k/v in ORIGINAL order on the GPU.  Returns (O, LSE, state) with O [N, hq, d]
    and LSE [hq, N] in original order and the raw state in plan order."""
    n, hq, d = q.shape
    qp, kp, vp = pl.permute(q), pl.permute(k), pl.permute(v)
    st = M.State(n, hq, d)
    o = torch.empty((n, hq, d), dtype=torch.bfloat16, device="cuda")
    lse = torch.empty((hq, n), dtype=torch.float32, device="cuda")
    if schedule is None:
        M.forward(pl, qp, kp, vp, st, o, lse, needed=needed, merge=merge, fused=fused)
    else:
        for r, j, first in schedule:
            M.attn_step(pl, qp, kp, vp, r, j, st, first=first, merge=merge)
        M.attn_finalize(pl, st, o, lse)
    pl.check()
    perm = pl.export("perm").long()
    O = pl.permute(o, inverse=True)
    LSE = torch.empty_like(lse)
    LSE[:, perm] = lse
    return O, LSE, st


def run_backward(pl, q, k, v, do, needed=False, fused=False):
    """Full forward + backward through the C ABI; gradients in original order (fp32)."""
    n, hq, d = q.shape
    hkv = k.shape[1]
    qp, kp, vp, dop = pl.permute(q), pl.permute(k), pl.permute(v), pl.permute(do)
    st = M.State(n, hq, d)
    o = torch.empty((n, hq, d), dtype=torch.bfloat16, device="cuda")
    lse = torch.empty((hq, n), dtype=torch.float32, device="cuda")
    M.forward(pl, qp, kp, vp, st, o, lse, needed=needed, fused=fused)
    delta = torch.empty((hq, n), dtype=torch.float32, device="cuda")
    dq = torch.zeros((n, hq, d), dtype=torch.float32, device="cuda")
    dk = torch.zeros((n, hkv, d), dtype=torch.float32, device="cuda")
    dv = torch.zeros((n, hkv, d), dtype=torch.float32, device="cuda")
    M.backward(pl, qp, kp, vp, o, dop, lse, delta, dq, dk, dv, needed=needed, fused=fused)
    pl.check()
    return (pl.permute(dq, inverse=True), pl.permute(dk, inverse=True),
            pl.permute(dv, inverse=True))


def check_o_lse(O, LSE, O_ref, LSE_ref):
    O = O.float().cpu().numpy()
    LSE = LSE.cpu().numpy()
    err = np.abs(O - O_ref)
    assert err.max() <= TOL_O_MAX, f"O max abs err {err.max()}"
    assert err.mean() <= TOL_O_MEAN, f"O mean abs err {err.mean()}"
    fin = np.isfinite(LSE_ref)
    assert (np.isfinite(LSE) == fin).all(), "LSE -inf pattern differs"
    if fin.any():
        e = np.abs(LSE[fin] - LSE_ref[fin]).max()
        assert e <= TOL_LSE, f"LSE abs err {e}"
    return float(err.max()), float(err.mean())


def rel_fro(a, b):
    a = np.asarray(a, np.float64)
    b = np.asarray(b, np.float64)
    return float(np.linalg.norm(a - b) / max(np.linalg.norm(b), 1e-30))


def token_shards(pl):
    """Shard of the plan that every original token lands in (plan order is shard-major)."""
    perm = pl.export("perm").cpu().numpy().astype(np.int64)
    inv = np.empty_like(perm)
    inv[perm] = np.arange(len(perm))
    return (inv // wl.BLOCK) // pl.blocks_per_shard


def spread_tokens(cands, shard, P, count, rng):
    """About `count` tokens of `cands`, spread as evenly as the candidates allow over the
    plan's P shards, half of each shard's share at block edges (first or last token of a
    128-token block) where it has any."""
    cands = np.unique(np.asarray(cands, np.int64))
    per = -(-count // P)
    out = []
    for r in range(P):
        c = cands[shard[cands] == r]
        if len(c) == 0:
            continue
        at_edge = (c % wl.BLOCK == 0) | (c % wl.BLOCK == wl.BLOCK - 1)
        edge = rng.permutation(c[at_edge])[:(per + 1) // 2]
        rest = rng.permutation(c[~at_edge])[:per - len(edge)]
        out += list(edge) + list(rest)
    return np.sort(np.array(out, np.int64))
