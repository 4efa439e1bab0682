"""Benchmark: attention fwd+bwd effective TFLOP/s on legal-pair (unmasked) FLOPs.

Workload (default): the packed multimodal 64K pack -- N = 65536 tokens, 16 q / 16 kv heads,
d = 128, bf16 Q/K/V/dO ~ N(0, 1) (seed 0), lognormal 60/30/10 text/image/generated sample
mix, P = 8 virtual shards in PTRR order.  One step = every forward ring step (P^2 calls,
r-major), the finalize, the backward preprocessing and every backward ring step (P^2
calls), all through the C ABI on one GPU.  The plan is built once per pack (it is reused by
every layer, forward and backward) and is timed separately.

Effective FLOPs per step = 14 * d * legal_pairs * Hq (forward 4 d, backward 10 d per legal
pair); legal_pairs comes from the library's own counter (marble_plan_stats).

Usage: python bench.py [--gpus N] [--steps K] [--warmup W] [--impl marble|reference]
For N > 1 (torchrun) every rank runs an independent replica (the path has no exchange
step on one GPU); rank 0 prints the line with the max-over-ranks time.
"""
from __future__ import annotations

import os

# More hardware work queues than CUDA's default 8: the library's side streams and teardown
# stream, torch's stream and the end-to-end loop's copy streams then do not share queues, so
# a copy never waits behind kernels of an unrelated stream.  Read when the CUDA context is
# created, so set before anything touches the GPU (a value the caller set is kept).
os.environ.setdefault("CUDA_DEVICE_MAX_CONNECTIONS", "32")

import argparse
import json
import statistics
import subprocess
import sys
import threading
import time

# DRAM bytes (dram__bytes_read.sum + dram__bytes_write.sum) of one launch of each kernel on
# the 64K packed workload, from one ncu capture (its command and summary are in profiles/),
# with the digest of the kernel's source files at the time of the capture: a figure is
# reported only while the source is unchanged, null otherwise.
KERNEL_DRAM_BYTES_PER_LAUNCH = {
    "k_bwd_dkdv": (468.4e6, "profiles/k_bwd_dkdv_packed_multimodal.md", "d72216ed9c132231"),
    "k_bwd_dq": (12848.1e6, "profiles/k_bwd_dq_packed_multimodal.md", "d72216ed9c132231"),
    "k_attn_fwd": (151.3e6, "profiles/k_attn_fwd_packed_multimodal.md", "5ac2f710191f7577"),
}
KERNEL_SOURCES = {"k_bwd_dkdv": ("attn_bwd.cu", "common.cuh"),
                  "k_bwd_dq": ("attn_bwd.cu", "common.cuh"),
                  "k_attn_fwd": ("attn_fwd.cu", "common.cuh")}


def kernel_source_digest(kernel: str) -> str:
    import hashlib
    h = hashlib.sha256()
    for f in KERNEL_SOURCES[kernel]:
        with open(os.path.join(ROOT, "context_attention_metadata_gb300", "csrc", f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def kernel_traffic(kernel: str):
    """(DRAM bytes per launch, source of the figure) if the capture matches the kernel's
    current source, else (None, why)."""
    if kernel not in KERNEL_DRAM_BYTES_PER_LAUNCH:
        return None, "no capture"
    b, where, digest = KERNEL_DRAM_BYTES_PER_LAUNCH[kernel]
    if kernel_source_digest(kernel) != digest:
        return None, f"kernel source changed since the capture in {where}"
    return b, f"ncu capture in {where} (dram__bytes_read.sum + dram__bytes_write.sum per launch)"

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "attn fwd+bwd effective TFLOP/s (unmasked FLOPs) and % of GB300 bf16 peak"
UNIT = "TFLOP/s"


def _peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            p = json.load(f)
        return float(p["bf16_tflops"]), float(p.get("bf16_tflops_sustained", 0)) or None, \
            float(p["hbm_gbs"]), "measured"
    except Exception:
        return 1900.0, 1700.0, 6800.0, "fallback"


def _dist():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    if ws <= 1:
        return 0, 1, 0, None
    import torch.distributed as dist
    backend = os.environ.get("MARBLE_BENCH_BACKEND", "nccl")
    dist.init_process_group(backend=backend)
    return dist.get_rank(), dist.get_world_size(), int(os.environ.get("LOCAL_RANK", "0")), dist


def max_over_ranks(x: float, dist) -> float:
    """Max of a per-rank scalar over all ranks (identity without a process group)."""
    if dist is None:
        return x
    import torch
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([x], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


class ClockSampler:
    """nvidia-smi clock / throttle-reason samples during the timed region."""

    def __init__(self, index: int):
        self.index = index
        self.rows = []
        self.proc = None

    def __enter__(self):
        q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.index}", f"--query-gpu={q}",
                 "--format=csv,noheader,nounits", "-lms", "50"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
            # the timed region starts once the sampler is producing rows
            t0 = time.perf_counter()
            while not self.rows and time.perf_counter() - t0 < 5.0:
                time.sleep(0.01)
            self.rows.clear()
        except Exception:
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.rows.append([x.strip() for x in line.split(",")])

    def __exit__(self, *a):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()

    def summary(self):
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for r in self.rows:
            try:
                sm.append(float(r[1]))
                mx = float(r[2])
                for nm, val in zip(names, r[5:9]):
                    if val.strip().lower() == "active":
                        reasons.add(nm)
            except (ValueError, IndexError):
                continue
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": mx,
                "reasons": sorted(reasons), "samples": len(sm)}


# --------------------------------------------------------------------------------------
# CPU oracle baseline (bounded sample of the same workload)
# --------------------------------------------------------------------------------------
def oracle_sample_rate(cfg, tr, budget_s: float, seed: int = 0):
    """Time the fp64 oracle's dense forward+backward on whole samples of the pack (all q
    heads) until ``budget_s`` seconds are spent; return effective TFLOP/s on legal pairs."""
    import numpy as np
    import torch

    from oracle import attention, counts, mask

    st = np.asarray(tr["sample"])
    ids = np.unique(st)
    rng = np.random.default_rng(seed)
    order = rng.permutation(ids)
    g = torch.Generator().manual_seed(seed)
    pairs = 0
    tokens = 0
    nsamp = 0
    elapsed = 0.0
    small = [sid for sid in order if np.count_nonzero(st == sid) <= 4096]
    for sid in (small or order[:1]):
        # whole samples of at most 4096 tokens; a pack without any: the first 4096 tokens of
        # one sample (its mask restricted to them is the same predicate on those tokens)
        idx = np.flatnonzero(st == sid)[:4096]
        L = len(idx)
        sub = {k: np.asarray(v)[idx] for k, v in tr.items()}
        if "pos" not in tr:
            sub["pos"] = idx
        q = torch.randn((L, cfg.hq, cfg.d), generator=g).to(torch.bfloat16)
        k = torch.randn((L, cfg.hkv, cfg.d), generator=g).to(torch.bfloat16)
        v = torch.randn((L, cfg.hkv, cfg.d), generator=g).to(torch.bfloat16)
        do = torch.randn((L, cfg.hq, cfg.d), generator=g).to(torch.bfloat16)
        t0 = time.perf_counter()
        if cfg.bwd:
            attention.backward(q, k, v, do, mask.dense_mask(sub, cfg.window))
        else:
            attention.forward(q, k, v, mask.dense_mask(sub, cfg.window))
        elapsed += time.perf_counter() - t0
        pairs += counts.by_key_classes(sub, cfg.window)
        tokens += L
        nsamp += 1
        if elapsed >= budget_s:
            break
    flops = (14.0 if cfg.bwd else 4.0) * cfg.d * pairs * cfg.hq
    return flops / elapsed / 1e12, elapsed, nsamp, tokens


def workload(args):
    """The configuration and tracks the command line asks for: one of the numbered
    workloads, optionally a smaller pack of its recipe (--tokens) and another token order
    (--order, --chunk-tokens, --range-cost)."""
    import dataclasses
    import workloads as wl
    cid = args.config
    base = wl.CONFIGS[cid] if cid in wl.CONFIGS else wl.EXTRA[cid]
    cfg = base if args.tokens <= 0 else wl.mini_config(cid, args.tokens, hq=base.hq)
    if args.order:
        cfg = dataclasses.replace(cfg, order=args.order, chunk_tokens=args.chunk_tokens,
                                  range_cost=args.range_cost,
                                  name=f"{cfg.name}_{args.order}")
    elif args.range_cost:
        cfg = dataclasses.replace(cfg, range_cost=args.range_cost)
    tr = wl.config_tracks(cid) if args.tokens <= 0 else wl.config_tracks(cid, cfg.n)
    if args.layout == "vision_groups":
        # the tokens in the vision-group order, each carrying its original position
        import numpy as np
        import context_attention_metadata_gb300 as M
        perm = M.layout_vision_groups(tr["sample"], tr["seg"]).astype(np.int64)
        tr = {"sample": tr["sample"][perm], "seg": tr["seg"][perm], "noise": tr["noise"][perm],
              "pos": perm.astype(np.int32)}
        cfg = dataclasses.replace(cfg, name=f"{cfg.name}_vision_groups")
    return cfg, tr


def run_reference(args, rank, world, dist):
    """The oracle as it stands, timed on the host cores (rank 0 only)."""
    cfg, tr = workload(args)
    if rank != 0:
        return
    for _ in range(args.warmup):
        oracle_sample_rate(cfg, tr, args.ref_budget)
    rates, times = [], []
    desc = None
    for i in range(args.steps):
        r, el, ns, tok = oracle_sample_rate(cfg, tr, args.ref_budget, seed=i)
        rates.append(r)
        times.append(el)
        desc = (f"{ns} whole samples ({tok} tokens) of the {cfg.name} pack, all {cfg.hq} q "
                f"heads, fp64 dense {'forward+backward' if cfg.bwd else 'forward'}, "
                f"~{args.ref_budget:.0f} s per step")
    value = statistics.mean(rates)
    cores = os.cpu_count()
    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": 1e3 * statistics.mean(times),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic", "impl": "reference",
        "config": {"workload": cfg.name, "n_tokens": cfg.n, "heads": f"{cfg.hq}/{cfg.hkv}",
                   "d": cfg.d, "shards": cfg.shards, "order": cfg.order},
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": cores, "kind": "oracle",
                         "sample": desc},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


# --------------------------------------------------------------------------------------
# the CUDA path
# --------------------------------------------------------------------------------------
def run_marble(args, rank, world, local, dist):
    import numpy as np
    import torch

    import context_attention_metadata_gb300 as M
    import workloads as wl
    from context_attention_metadata_gb300 import _build

    torch.cuda.set_device(local)
    _build.build()
    cfg, tr = workload(args)
    n, hq, hkv, d, P = cfg.n, cfg.hq, cfg.hkv, cfg.d, cfg.shards
    needed = cfg.needed
    trk = [torch.as_tensor(np.asarray(tr[x], np.int32)).cuda() for x in ("sample", "seg", "noise")]
    pos_t = torch.as_tensor(np.asarray(tr["pos"], np.int32)).cuda() if "pos" in tr else None
    stream = torch.cuda.current_stream()

    # plan: built once per pack, timed on its own (best of 3)
    plan_ms = []
    pl = None
    for _ in range(3):
        if pl is not None:
            pl.close()
        torch.cuda.synchronize()
        t0 = time.perf_counter()
        pl = M.Plan(trk[0], trk[1], trk[2], cfg.window, P, cfg.order, cfg.chunk_tokens,
                    range_cost=cfg.range_cost, key_intervals=not args.no_key_intervals,
                    pos=pos_t)
        torch.cuda.synchronize()
        plan_ms.append(1e3 * (time.perf_counter() - t0))
    stats = pl.stats()
    pairs = stats["legal_pairs"]
    with_bwd = cfg.bwd
    flops_fwd = 4.0 * d * pairs * hq
    flops_bwd = 10.0 * d * pairs * hq if with_bwd else 0.0
    flops = flops_fwd + flops_bwd

    q, k, v, do = wl.make_qkvdo(n, hq, hkv, d, device="cuda", seed=0)
    qp, kp, vp, dop = (pl.permute(t) for t in (q, k, v, do))
    st = M.State(n, hq, d)
    o = torch.empty((n, hq, d), dtype=torch.bfloat16, device="cuda")
    lse = torch.empty((hq, n), dtype=torch.float32, device="cuda")
    delta = torch.empty_like(lse)
    dq = torch.empty((n, hq, d), dtype=torch.float32, device="cuda")
    dk = torch.empty((n, hkv, d), dtype=torch.float32, device="cuda")
    dv = torch.empty((n, hkv, d), dtype=torch.float32, device="cuda")
    sched = M.ring_schedule(P, needed)
    ev = lambda: torch.cuda.Event(enable_timing=True)

    def step(marks=None):
        if marks:
            marks[0].record(stream)
        M.attn_steps(pl, qp, kp, vp, sched, st)
        if marks:
            marks[1].record(stream)
        M.attn_finalize(pl, st, o, lse)
        if with_bwd:
            M.attn_bwd_prep(pl, o, dop, delta)
            dq.zero_()
            dk.zero_()
            dv.zero_()
        if marks:
            marks[2].record(stream)
        if with_bwd:
            M.attn_bwd_steps(pl, qp, kp, vp, dop, lse, delta, sched, dq, dk, dv)
        if marks:
            marks[3].record(stream)

    for _ in range(max(3, args.warmup)):
        step()
    pl.check()
    torch.cuda.synchronize()
    if dist is not None:
        dist.barrier()
    marks = [[ev() for _ in range(4)] for _ in range(args.steps)]
    M.timing_read()  # drop anything recorded before the timed region
    M.timing_enable(True)
    with ClockSampler(torch.cuda.current_device()) as clk:
        torch.cuda.synchronize()
        t_wall = time.perf_counter()
        for i in range(args.steps):
            step(marks[i])
        torch.cuda.synchronize()
        t_wall = time.perf_counter() - t_wall
    M.timing_enable(False)
    ktime = M.timing_read()  # per-kernel device time, CUDA events on each kernel's stream
    if dist is not None:
        dist.barrier()
    pl.check()
    step_ms = [m[0].elapsed_time(m[3]) for m in marks]
    fwd_ms = [m[0].elapsed_time(m[1]) for m in marks]
    bwd_ms = [m[2].elapsed_time(m[3]) for m in marks]
    mid_ms = [m[1].elapsed_time(m[2]) for m in marks]
    dev_s = max_over_ranks(sum(step_ms) / 1e3, dist)
    value = world * flops * args.steps / dev_s / 1e12
    ms_per_step = 1e3 * dev_s / args.steps

    peak, peak_sus, hbm, peak_kind = _peaks()
    mf, mb = statistics.mean(fwd_ms), statistics.mean(bwd_ms)

    def roofline_of(kt, n_steps, note):
        """Roofline of the dominant kernel from per-kernel device times: its algorithmic
        FLOPs (forward: S and PV, 4 d per legal pair and q head; dK/dV kernel: S, dP, dV and
        dK, 8 d; dQ kernel: dQ, 2 d) over its own summed duration, per launch."""
        kern = {"k_attn_fwd": (flops_fwd, kt["fwd_ms"], kt["fwd_launches"])}
        if with_bwd:
            kern["k_bwd_dkdv"] = (0.8 * flops_bwd, kt["dkdv_ms"], kt["dkdv_launches"])
            kern["k_bwd_dq"] = (0.2 * flops_bwd, kt["dq_ms"], kt["dq_launches"])
        dom = max(kern, key=lambda k_: kern[k_][1])
        f_step, k_ms, k_launches = kern[dom]
        mpl = k_ms / max(k_launches, 1)
        fpl = f_step * n_steps / max(k_launches, 1)
        ach = fpl / (mpl / 1e3) / 1e12
        tot = sum(v_[1] for v_ in kern.values())
        traffic, traffic_src = kernel_traffic(dom)
        return {"bound": "tensor", "achieved": ach, "peak": peak, "unit": "TFLOP/s",
                "frac": ach / peak, "traffic": traffic, "traffic_source": traffic_src,
                "kernel": dom, "launches": k_launches, "ms_per_launch": mpl,
                "flops_per_launch": fpl,
                "peak_source": f"{peak_kind} bf16 dense burst (MEASURED_PEAKS.json)",
                "kernel_ms": {k_: round(v_[1] / n_steps, 3) for k_, v_ in kern.items()},
                "kernel_share": {k_: round(v_[1] / tot, 3) for k_, v_ in kern.items()},
                "kernel_tflops": {k_: (v_[0] * n_steps / (v_[1] / 1e3) / 1e12 if v_[1] else None)
                                  for k_, v_ in kern.items()},
                "note": note}

    roof_situ = roofline_of(
        ktime, args.steps,
        "per-launch spans inside the timed step, whose launches overlap on several streams: a "
        "span includes time spent waiting for SMs held by other launches")

    # The dominant kernel's own duration: the same step with every launch in list order on
    # one stream (no overlap), warm; each kernel's span is then its duration.
    iso_steps = 2
    M.set_side_streams(0)
    step()
    torch.cuda.synchronize()
    M.timing_read()
    M.timing_enable(True)
    for _ in range(iso_steps):
        step()
    torch.cuda.synchronize()
    M.timing_enable(False)
    kt_iso = M.timing_read()
    M.set_side_streams(4)
    pl.check()
    roof = roofline_of(kt_iso, iso_steps,
                       "each launch alone on one stream, warm, after the timed steps: the "
                       "kernel's own duration (CUDA events on its stream)")

    # HBM-bound helpers, each timed alone (CUDA events, warm, mean of 5), against the measured
    # copy bandwidth; bytes per call from the algorithmic formulas (reads + writes)
    def time_call(fn, reps=5):
        fn()
        evs = [(ev(), ev()) for _ in range(reps)]
        for e0, e1 in evs:
            e0.record(stream)
            fn()
            e1.record(stream)
        torch.cuda.synchronize()
        return statistics.mean(e0.elapsed_time(e1) for e0, e1 in evs)

    helpers = {}
    th = time_call(lambda: M.attn_finalize(pl, st, o, lse))
    by = n * hq * (6 * d + 12)
    helpers["finalize"] = {"ms": th, "bytes": by, "gbs": by / th / 1e6}
    if with_bwd:
        th = time_call(lambda: M.attn_bwd_prep(pl, o, dop, delta))
        by = n * hq * (4 * d + 4)
        helpers["bwd_prep"] = {"ms": th, "bytes": by, "gbs": by / th / 1e6}
    th = time_call(lambda: pl.permute(q, out=qp))
    by = 2 * n * hq * d * 2
    helpers["permute_q"] = {"ms": th, "bytes": by, "gbs": by / th / 1e6}
    if with_bwd:
        dq_bf = torch.empty((n, hq, d), dtype=torch.bfloat16, device="cuda")
        th = time_call(lambda: pl.permute_cast_bf16(dq, inverse=True, out=dq_bf))
        by = n * hq * d * (4 + 2)
        helpers["permute_cast_dq"] = {"ms": th, "bytes": by, "gbs": by / th / 1e6}
        del dq_bf
    plan_bytes = n * (12 + 4 + 16) + 3 * 5 * stats["nnz"]
    helpers["plan"] = {"ms": min(plan_ms), "bytes": plan_bytes,
                       "gbs": plan_bytes / min(plan_ms) / 1e6,
                       "note": "marble_plan end to end (host wall clock, it synchronises its "
                               "stream to size its arrays): 12 B of tracks in, perm and "
                               "permuted tracks out per token, 5 B per non-empty tile in each "
                               "of three tile lists"}
    for v_ in helpers.values():
        v_["frac_of_hbm"] = v_["gbs"] / hbm
    helpers["hbm_peak_gbs"] = hbm

    # end to end through the public API: H2D of the step's inputs from pinned memory,
    # plan, permutation, forward, backward, inverse permutation (with the bf16 cast of the
    # gradients), D2H results.  Steps are pipelined the way a training loop runs them: the
    # next step's inputs are copied in on one copy stream and its tracks copied and its plan
    # built on another while this step computes, and this step's results are copied out on a
    # third while the next step computes (double-buffered inputs and outputs; O leaves as
    # soon as the forward has made it).  Each plan is destroyed as soon as its step is
    # queued: the library frees it in stream order, without synchronising.
    e2e = None
    if args.e2e_steps > 0:
        hq_pin = [t.cpu().pin_memory() for t in ((q, k, v, do) if with_bwd else (q, k, v))]
        htr = [t.cpu().pin_memory() for t in trk + ([pos_t] if pos_t is not None else [])]
        shapes = ((n, hq, d), (n, hq, d), (n, hkv, d), (n, hkv, d)) if with_bwd else ((n, hq, d),)
        out_pin = [[torch.empty(s_, dtype=torch.bfloat16).pin_memory() for s_ in shapes]
                   for _ in range(2)]
        outs = [[torch.empty(s_, dtype=torch.bfloat16, device="cuda") for s_ in shapes]
                for _ in range(2)]
        dev_in = [[torch.empty_like(t, device="cuda") for t in hq_pin] for _ in range(2)]
        dev_tr = [[torch.empty_like(t, device="cuda") for t in htr] for _ in range(2)]
        cs = torch.cuda.Stream()       # host -> device: tracks, then the plan
        cs_in = torch.cuda.Stream()    # host -> device: Q, K, V, dO
        cs_out = torch.cuda.Stream()   # device -> host (the two directions overlap)
        comp = torch.cuda.current_stream()

        def e2e_run(K):
            plans = [None] * K
            ev_qkv, ev_do, ev_used, ev_o, ev_out, ev_d2h, ev_plan = (
                [torch.cuda.Event() for _ in range(2)] for _ in range(7))

            def h2d_and_plan(i):
                # the step's tracks, then its plan, on one copy stream; its Q/K/V (then dO) on
                # another.  The tracks go first, so that the planner's own synchronisation
                # waits for their small copy only, not for the inputs' copy nor for the
                # previous step's compute.  marble_plan has read its tracks when it returns,
                # so their buffer is free again at once.
                b = i % 2
                with torch.cuda.stream(cs):
                    for dst, src in zip(dev_tr[b], htr):
                        dst.copy_(src, non_blocking=True)
                with torch.cuda.stream(cs_in):
                    if i >= 2:
                        cs_in.wait_event(ev_used[b])   # step i - 2 is done with buffer b
                    for j, (dst, src) in enumerate(zip(dev_in[b], hq_pin)):
                        dst.copy_(src, non_blocking=True)
                        if j == 2:
                            ev_qkv[b].record(cs_in)  # the forward needs Q, K and V only
                    ev_do[b].record(cs_in)
                plans[i] = M.Plan(dev_tr[b][0], dev_tr[b][1], dev_tr[b][2], cfg.window, P,
                                  cfg.order, cfg.chunk_tokens, stream=cs,
                                  range_cost=cfg.range_cost,
                                  key_intervals=not args.no_key_intervals,
                                  pos=dev_tr[b][3] if pos_t is not None else None)
                ev_plan[b].record(cs)

            def d2h(ev_ready, pairs, ev_done=None):
                with torch.cuda.stream(cs_out):
                    cs_out.wait_event(ev_ready)
                    for dst, src in pairs:
                        dst.copy_(src, non_blocking=True)
                    if ev_done is not None:
                        ev_done.record(cs_out)

            h2d_and_plan(0)
            for i in range(K):
                b = i % 2
                p2 = plans[i]
                ob = outs[b]
                comp.wait_event(ev_plan[b])
                comp.wait_event(ev_qkv[b])
                q2, k2, v2 = [p2.permute(t) for t in dev_in[b][:3]]
                M.forward(p2, q2, k2, v2, st, o, lse, needed=needed)
                if i >= 2:
                    comp.wait_event(ev_d2h[b])      # step i - 2's results have left buffer b
                p2.permute(o, inverse=True, out=ob[0])
                ev_o[b].record(comp)
                if with_bwd:
                    d2h(ev_o[b], [(out_pin[b][0], ob[0])])   # O leaves while dK/dV run
                    comp.wait_event(ev_do[b])
                    do2 = p2.permute(dev_in[b][3])
                    dq.zero_()
                    dk.zero_()
                    dv.zero_()
                    M.backward(p2, q2, k2, v2, o, do2, lse, delta, dq, dk, dv, needed=needed)
                ev_used[b].record(comp)
                if with_bwd:
                    for g_, b_ in ((dq, ob[1]), (dk, ob[2]), (dv, ob[3])):
                        p2.permute_cast_bf16(g_, inverse=True, out=b_)
                ev_out[b].record(comp)
                pairs = list(zip(out_pin[b], ob))
                d2h(ev_out[b], pairs[1:] if with_bwd else pairs, ev_d2h[b])
                p2.close()                          # stream-ordered: no synchronisation
                plans[i] = None
                if i + 1 < K:
                    h2d_and_plan(i + 1)             # while step i computes
            torch.cuda.synchronize()

        # warm-up as long as the timed run, so that the memory pool already holds the
        # workspaces of the plans in flight
        e2e_run(max(4, args.warmup, args.e2e_steps))
        # the median of several timed runs of K steps each: on a shared host, single runs
        # now and then take a stall of tens of ms in the host thread (all runs are reported)
        runs = []
        for _ in range(max(1, args.e2e_runs)):
            torch.cuda.synchronize()
            t0 = time.perf_counter()
            e2e_run(args.e2e_steps)
            runs.append((time.perf_counter() - t0) / args.e2e_steps)
        e2e_s = max_over_ranks(statistics.median(runs), dist)
        h2d_b = sum(t.numel() * t.element_size() for t in hq_pin + htr)
        d2h_b = sum(t.numel() * t.element_size() for t in out_pin[0])
        e2e = {"value": world * flops / e2e_s / 1e12, "unit": UNIT,
               "h2d_bytes_per_step": h2d_b, "d2h_bytes_per_step": d2h_b,
               "ms_per_step": 1e3 * e2e_s,
               "runs_ms_per_step": [round(1e3 * r_, 3) for r_ in runs],
               "timing": f"median of {len(runs)} runs of {args.e2e_steps} pipelined steps, "
                         "host wall clock around each run",
               "includes": "H2D inputs+tracks, marble_plan, "
               "permute, fwd, finalize, " + ("bwd_prep, bwd, " if with_bwd else "") +
               "inverse permute" + (" (gradients: fused with the bf16 cast)" if with_bwd
                                    else "") + ", D2H, plan "
               "teardown; steps pipelined (copies and the next step's plan on copy streams "
               "overlap compute)"}

    # the forward with each merge of the ring steps: the carried fp32 state (the timed step
    # above), the merge of fp32 partials and the standard merge of bf16 partials
    merge_ms = {}
    for merge in ("carried", "fp32", "bf16"):
        M.attn_steps(pl, qp, kp, vp, sched, st, merge=merge)
        M.attn_finalize(pl, st, o, lse)
        evs = [(ev(), ev()) for _ in range(3)]
        for e0, e1 in evs:
            e0.record(stream)
            M.attn_steps(pl, qp, kp, vp, sched, st, merge=merge)
            M.attn_finalize(pl, st, o, lse)
            e1.record(stream)
        torch.cuda.synchronize()
        merge_ms[merge] = statistics.mean(e0.elapsed_time(e1) for e0, e1 in evs)
    pl.check()
    merge_variants = {"unit": "ms per forward pass (all ring steps + finalize), mean of 3",
                      **{k_: round(v_, 3) for k_, v_ in merge_ms.items()},
                      "tflops": {k_: flops_fwd / (v_ / 1e3) / 1e12 for k_, v_ in merge_ms.items()}}

    # The fused ring beside the per-step path: every forward ring step in one launch with the
    # state on chip between steps, then one dK/dV launch per kv shard over its ring (dK/dV on
    # chip across q shards) with the per-step dQ GEMMs; same inputs, same FLOPs, same
    # finalize and bwd_prep, device-timed over the same number of steps.
    fused = None
    if not needed:
        def fused_step():
            M.attn_fwd_fused(pl, qp, kp, vp, st)
            M.attn_finalize(pl, st, o, lse)
            if with_bwd:
                M.attn_bwd_prep(pl, o, dop, delta)
                dq.zero_()
                dk.zero_()
                dv.zero_()
                M.attn_bwd_fused(pl, qp, kp, vp, dop, lse, delta, dq, dk, dv)

        for _ in range(max(3, args.warmup)):
            fused_step()
        torch.cuda.synchronize()
        evs = [(ev(), ev(), ev()) for _ in range(args.steps)]
        M.timing_read()
        M.timing_enable(True)
        for e0, e1, e2 in evs:
            e0.record(stream)
            M.attn_fwd_fused(pl, qp, kp, vp, st)
            e1.record(stream)
            M.attn_finalize(pl, st, o, lse)
            if with_bwd:
                M.attn_bwd_prep(pl, o, dop, delta)
                dq.zero_()
                dk.zero_()
                dv.zero_()
                M.attn_bwd_fused(pl, qp, kp, vp, dop, lse, delta, dq, dk, dv)
            e2.record(stream)
        torch.cuda.synchronize()
        M.timing_enable(False)
        kt_f = M.timing_read()
        pl.check()
        f_ms = statistics.mean(a.elapsed_time(c) for a, b, c in evs)
        ff_ms = statistics.mean(a.elapsed_time(b) for a, b, c in evs)
        f_dev_s = max_over_ranks(f_ms * args.steps / 1e3, dist)
        fused = {"value": world * flops * args.steps / f_dev_s / 1e12, "unit": UNIT,
                 "ms_per_step": f_ms, "fwd_ms": ff_ms,
                 "fwd_tflops": flops_fwd / (ff_ms / 1e3) / 1e12,
                 "bwd_ms": f_ms - ff_ms,
                 "launches_per_step": {k_: kt_f[k_ + "_launches"] // args.steps
                                       for k_ in ("fwd", "dkdv", "dq")},
                 "what": "marble_attn_fwd_fused + finalize + bwd_prep + marble_attn_bwd_fused "
                         "(the same ring steps; state and dK/dV on chip between them)"}

    cpu = None
    if rank == 0 and args.cpu_budget > 0:
        r, el, ns, tok = oracle_sample_rate(cfg, tr, args.cpu_budget)
        cpu = {"value": r, "unit": UNIT, "cores": os.cpu_count(), "kind": "oracle",
               "sample": f"{ns} whole samples ({tok} tokens) of the pack, all {hq} q heads, "
                         f"fp64 dense {'fwd+bwd' if with_bwd else 'fwd'}, {el:.1f} s"}

    if rank == 0:
        line = {
            "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world,
            "steps": args.steps, "warmup": max(3, args.warmup), "ms_per_step": ms_per_step,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
            "data": "synthetic",
            "config": {"workload": cfg.name, "n_tokens": n, "heads": f"{hq}/{hkv}", "d": d,
                       "shards": P, "order": cfg.order, "window": cfg.window,
                       "range_cost": cfg.range_cost if cfg.order == "chunk_search" else None,
                       "key_intervals": not args.no_key_intervals,
                       "layout": args.layout or "as generated",
                       "schedule": "needed-blocks" if needed else "ring r-major P^2 steps",
                       "l2": "inputs larger than L2 (Q/K/V/dO 256 MiB each; state 512 MiB)",
                       "legal_pairs_per_head": pairs, "flops_per_step": flops,
                       "parallelism": f"replicas x{world}"},
            "pct_of_peak": 100.0 * value / world / peak,
            "pct_of_sustained_peak": (100.0 * value / world / peak_sus) if peak_sus else None,
            "phases_ms": {"fwd_steps": mf, "finalize+prep+zero": statistics.mean(mid_ms),
                          "bwd_steps": mb},
            "tile_tflops": (14.0 if with_bwd else 4.0) * d * hq * stats["nnz"] * 128 * 128
                           / (ms_per_step / 1e3) / 1e12,
            "fwd_tflops": flops_fwd / (mf / 1e3) / 1e12,
            "bwd_tflops": flops_bwd / (mb / 1e3) / 1e12 if with_bwd else None,
            "plan_ms": min(plan_ms), "plan_stats": stats,
            "wall_s_timed_region": t_wall,
            "roofline": roof,
            "roofline_in_situ": roof_situ,
            "hbm_helpers": helpers,
            "fwd_merge_variants": merge_variants,
            "fused": fused,
            "cpu_baseline": cpu,
            "e2e": e2e,
            # our kernels in the timed region: attention launches counted by the library,
            # plus finalize and bwd_prep once per step
            "gpu_launches": ktime["fwd_launches"] + ktime["dq_launches"] +
                            ktime["dkdv_launches"] + 2 * args.steps,
            "clocks": clk.summary(),
            "env": {"CUDA_DEVICE_MAX_CONNECTIONS": os.environ.get("CUDA_DEVICE_MAX_CONNECTIONS")},
        }
        print(json.dumps(line), flush=True)


def run_profile_pass(args):
    """Driver for ncu captures: plan + `--profile-pass` forward+backward passes of the
    workload (optionally a smaller pack of the same recipe, `--tokens`), untimed, no JSON."""
    import numpy as np
    import torch
    import context_attention_metadata_gb300 as M
    import workloads as wl
    cfg, tr = workload(args)
    trk = [torch.as_tensor(np.asarray(tr[x], np.int32)).cuda() for x in ("sample", "seg", "noise")]
    pos_t = torch.as_tensor(np.asarray(tr["pos"], np.int32)).cuda() if "pos" in tr else None
    pl = M.Plan(trk[0], trk[1], trk[2], cfg.window, cfg.shards, cfg.order, cfg.chunk_tokens,
                range_cost=cfg.range_cost, pos=pos_t)
    n, hq, hkv, d = cfg.n, cfg.hq, cfg.hkv, cfg.d
    q, k, v, do = wl.make_qkvdo(n, hq, hkv, d, device="cuda")
    qp, kp, vp, dop = (pl.permute(t) for t in (q, k, v, do))
    st = M.State(n, hq, d)
    o = torch.empty((n, hq, d), dtype=torch.bfloat16, device="cuda")
    lse = torch.empty((hq, n), dtype=torch.float32, device="cuda")
    delta = torch.empty_like(lse)
    dq = torch.zeros((n, hq, d), dtype=torch.float32, device="cuda")
    dk = torch.zeros((n, hkv, d), dtype=torch.float32, device="cuda")
    dv = torch.zeros((n, hkv, d), dtype=torch.float32, device="cuda")
    fused = args.profile_fused and not cfg.needed
    for _ in range(args.profile_pass):
        M.forward(pl, qp, kp, vp, st, o, lse, needed=cfg.needed, fused=fused)
        M.backward(pl, qp, kp, vp, o, dop, lse, delta, dq, dk, dv, needed=cfg.needed,
                   fused=fused)
    pl.check()
    torch.cuda.synchronize()
    print(f"profile pass ok: {cfg.name} n={n} passes={args.profile_pass}", flush=True)


def run_emulated_ring(args):
    """Side measurement for token layouts: every ring step (q shard r, kv shard j) timed on
    its own on an otherwise idle GPU (one GPU standing for one rank), then the time of a
    ring of P such GPUs: sum over steps s of the slowest rank's step, forward ring then
    backward ring.  Prints one JSON line with the plan's step cost in legal pairs beside it
    (the first term of the layout cost C of the chunked ring)."""
    import numpy as np
    import torch
    import context_attention_metadata_gb300 as M
    from context_attention_metadata_gb300 import _build

    _build.build()
    cfg, tr = workload(args)
    n, hq, hkv, d, P = cfg.n, cfg.hq, cfg.hkv, cfg.d, cfg.shards
    trk = [torch.as_tensor(np.asarray(tr[x], np.int32)).cuda() for x in ("sample", "seg", "noise")]
    pos_t = torch.as_tensor(np.asarray(tr["pos"], np.int32)).cuda() if "pos" in tr else None
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    pl = M.Plan(trk[0], trk[1], trk[2], cfg.window, P, cfg.order, cfg.chunk_tokens,
                range_cost=cfg.range_cost, pos=pos_t)
    torch.cuda.synchronize()
    plan_ms = 1e3 * (time.perf_counter() - t0)
    stats = pl.stats()
    import workloads as wl
    q, k, v, do = wl.make_qkvdo(n, hq, hkv, d, device="cuda", seed=0)
    qp, kp, vp, dop = (pl.permute(t) for t in (q, k, v, do))
    st = M.State(n, hq, d)
    o = torch.empty((n, hq, d), dtype=torch.bfloat16, device="cuda")
    lse = torch.empty((hq, n), dtype=torch.float32, device="cuda")
    delta = torch.empty_like(lse)
    dq = torch.zeros((n, hq, d), dtype=torch.float32, device="cuda")
    dk = torch.zeros((n, hkv, d), dtype=torch.float32, device="cuda")
    dv = torch.zeros((n, hkv, d), dtype=torch.float32, device="cuda")
    stream = torch.cuda.current_stream()
    tf = np.full((args.steps, P, P), np.inf)
    tb = np.full((args.steps, P, P), np.inf)
    for it in range(args.warmup + args.steps):
        for r in range(P):
            for s_ in range(P):
                j = (r - s_) % P
                e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                e0.record(stream)
                M.attn_step(pl, qp, kp, vp, r, j, st, first=(s_ == 0))
                e1.record(stream)
                torch.cuda.synchronize()
                if it >= args.warmup:
                    tf[it - args.warmup, r, j] = e0.elapsed_time(e1)
        M.attn_finalize(pl, st, o, lse)
        M.attn_bwd_prep(pl, o, dop, delta)
        for r in range(P):
            for s_ in range(P):
                j = (r - s_) % P
                e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                e0.record(stream)
                M.attn_bwd_steps(pl, qp, kp, vp, dop, lse, delta, [(r, j, False)], dq, dk, dv)
                e1.record(stream)
                torch.cuda.synchronize()
                if it >= args.warmup:
                    tb[it - args.warmup, r, j] = e0.elapsed_time(e1)
    pl.check()
    tf, tb = np.median(tf, axis=0), np.median(tb, axis=0)

    def ring(t):
        return float(sum(max(t[r, (r - s_) % P] for r in range(P)) for s_ in range(P)))

    line = {"measurement": "emulated ring of P GPUs, one rank per launch",
            "workload": cfg.name, "n_tokens": n, "heads": f"{hq}/{hkv}", "shards": P,
            "order": cfg.order, "chunk_tokens": cfg.chunk_tokens, "range_cost": cfg.range_cost,
            "steps": args.steps, "warmup": args.warmup,
            "ring_ms": {"fwd": ring(tf), "bwd": ring(tb), "total": ring(tf) + ring(tb)},
            "serial_ms": {"fwd": float(tf.sum()), "bwd": float(tb.sum())},
            "plan_ms": plan_ms,
            "step_cost_pairs": stats["step_cost_pairs"], "step_cost_tiles": stats["step_cost"],
            "chunks_per_rank": stats["chunks_per_rank"], "layout_cost": stats["layout_cost"],
            "legal_pairs": stats["legal_pairs"], "nnz": stats["nnz"]}
    print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=30)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", default="marble", choices=["marble", "reference"])
    ap.add_argument("--config", type=int, default=2)
    ap.add_argument("--e2e-steps", type=int, default=20)
    ap.add_argument("--e2e-runs", type=int, default=3)
    ap.add_argument("--cpu-budget", type=float, default=15.0,
                    help="seconds of oracle time for cpu_baseline (0 disables)")
    ap.add_argument("--ref-budget", type=float, default=5.0,
                    help="seconds of oracle time per reference-arm step")
    ap.add_argument("--profile-pass", type=int, default=0,
                    help="run this many untimed fwd+bwd passes for a profiler and exit")
    ap.add_argument("--profile-fused", action="store_true",
                    help="with --profile-pass: the fused ring entry points")
    ap.add_argument("--tokens", type=int, default=0,
                    help="a smaller pack of the same recipe (side measurements, profiling)")
    ap.add_argument("--order", default="",
                    help="token order instead of the workload's (side measurements)")
    ap.add_argument("--chunk-tokens", type=int, default=0, help="with --order ptrr_chunk")
    ap.add_argument("--range-cost", type=int, default=0,
                    help="with the chunk_search order: tau, legal pairs per range and step")
    ap.add_argument("--layout", default="", choices=["", "vision_groups"],
                    help="side measurement: run the workload in another token layout")
    ap.add_argument("--no-key-intervals", action="store_true",
                    help="side measurement: partial tiles always evaluate the four-track "
                         "predicate")
    ap.add_argument("--emulate-ring", action="store_true",
                    help="side measurement: time every ring step alone, report the ring time "
                         "of P GPUs (sum over steps of the slowest rank)")
    args = ap.parse_args()
    if args.profile_pass > 0:
        run_profile_pass(args)
        return
    if args.emulate_ring:
        run_emulated_ring(args)
        return
    rank, world, local, dist = _dist()
    if args.impl == "reference":
        run_reference(args, rank, world, dist)
    else:
        run_marble(args, rank, world, local, dist)
    if dist is not None:
        dist.barrier()
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
