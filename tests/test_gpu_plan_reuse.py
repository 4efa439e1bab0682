"""One plan per batch, each destroyed as soon as its backward is queued, as a training loop
runs them.  marble_plan_destroy keeps a plan's bf16 dS^T scratch for the next plan's
backward, which takes it in stream order: the gradients must equal those of the first plan
(same inputs, same mask, the same deterministic launches), and a loop of such plans must not
grow the device memory in use after its first steps."""
import pytest
import torch

import context_attention_metadata_gb300 as M
import workloads as wl
from marble_testlib import plan_for

pytestmark = pytest.mark.gpu


def _step(cfg, tr, q, k, v, do, close=True):
    pl = plan_for(cfg, tr)
    n, hq, d = q.shape
    hkv = k.shape[1]
    qp, kp, vp, dop = pl.permute(q), pl.permute(k), pl.permute(v), pl.permute(do)
    st = M.State(n, hq, d)
    o = torch.empty((n, hq, d), dtype=torch.bfloat16, device="cuda")
    lse = torch.empty((hq, n), dtype=torch.float32, device="cuda")
    delta = torch.empty_like(lse)
    M.forward(pl, qp, kp, vp, st, o, lse)
    dq = torch.zeros((n, hq, d), dtype=torch.float32, device="cuda")
    dk = torch.zeros((n, hkv, d), dtype=torch.float32, device="cuda")
    dv = torch.zeros((n, hkv, d), dtype=torch.float32, device="cuda")
    M.backward(pl, qp, kp, vp, o, dop, lse, delta, dq, dk, dv)
    out = [pl.permute(g, inverse=True) for g in (dq, dk, dv)]
    if close:
        pl.close()  # stream-ordered: nothing waits here
        return out, None
    return out, pl


def test_back_to_back_plans_reuse_the_scratch_in_stream_order():
    cfg = wl.mini_config(2, n=8192, hq=8)
    tr = wl.config_tracks(2, cfg.n)
    q, k, v, do = wl.make_qkvdo(cfg.n, cfg.hq, cfg.hkv, cfg.d, device="cuda", seed=5)
    ref, pl0 = _step(cfg, tr, q, k, v, do, close=False)
    pl0.check()  # synchronises and reports any in-kernel timeout of the first plan
    pl0.close()
    bufs = [[torch.empty_like(g) for g in ref] for _ in range(6)]
    free = []
    for i in range(6):
        out = _step(cfg, tr, q, k, v, do)[0]
        for b, g in zip(bufs[i], out):
            b.copy_(g)
        del out
        if i in (1, 5):
            torch.cuda.synchronize()
            free.append(torch.cuda.mem_get_info()[0])
    torch.cuda.synchronize()
    for got in bufs:
        for g, g0 in zip(got, ref):
            torch.testing.assert_close(g, g0, rtol=1e-6, atol=1e-6)
    assert free[1] >= free[0], (free, "device memory grew over back-to-back plans")


def test_release_memory_gives_back_the_kept_scratch():
    """marble_release_memory returns the scratch a destroyed plan left for later plans, and
    the pool's unused blocks, to the device."""
    cfg = wl.mini_config(2, n=8192, hq=8)
    tr = wl.config_tracks(2, cfg.n)
    q, k, v, do = wl.make_qkvdo(cfg.n, cfg.hq, cfg.hkv, cfg.d, device="cuda", seed=6)
    _step(cfg, tr, q, k, v, do)  # warms torch's own allocator for the same tensors
    torch.cuda.synchronize()
    M.release_memory()
    free0 = torch.cuda.mem_get_info()[0]
    _step(cfg, tr, q, k, v, do)  # the plan and its scratch come from the pool again
    torch.cuda.synchronize()
    free1 = torch.cuda.mem_get_info()[0]
    assert free1 < free0, (free0, free1)
    M.release_memory()
    free2 = torch.cuda.mem_get_info()[0]
    assert free2 > free1, (free1, free2)
    assert free2 >= free0 - (64 << 20), (free0, free2)
