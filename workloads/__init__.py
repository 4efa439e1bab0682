"""Seeded synthetic workloads shared by the CUDA path's tests/bench and the oracle.

This module only *builds inputs*: per-token metadata tracks for packed multimodal
sequences and seeded bf16 Q/K/V/dO tensors.  It contains none of the method's
arithmetic (no mask evaluation, no tile classification, no attention).

Track encoding (MARBLE post, section 01 "Packed multimodal masks"): every token carries
  sample  -- id of the sample it belongs to (non-decreasing along the pack),
  seg     -- id shared by the tokens of one bidirectional span or of one image group,
             -1 for causal tokens,
  noise   -- id of a generated (noise) span, -1 for every other token,
  pos     -- its original position, which is simply its index in the pack.

Span modes follow the mode table of the same section: ``causal``, ``full`` (bidirectional),
``noise`` (bidirectional, hidden from later spans), ``group`` (all spans of one group
of a sample attend jointly).  ``window`` is a per-layer property (W), not a span mode.
"""
from __future__ import annotations

import dataclasses
import math
from typing import Dict, List, Optional, Sequence, Tuple

import numpy as np

BLOCK = 128
WINDOW_INF = 2**31 - 1  # "infinite" window: every causal distance is < W


# --------------------------------------------------------------------------------------
# spans -> tracks
# --------------------------------------------------------------------------------------
@dataclasses.dataclass(frozen=True)
class Span:
    mode: str          # "causal" | "full" | "noise" | "group"
    length: int
    group: int = 0     # group key (only for mode == "group"; local to the sample)


def tracks_from_samples(samples: Sequence[Sequence[Span]]) -> Dict[str, np.ndarray]:
    """Encode a pack (list of samples, each a list of spans) into the four tracks.

    Segment ids are unique over the pack.  A group key maps to one segment id per
    sample.  A noise span gets a fresh segment id and the same value as its noise id.
    """
    n = sum(sp.length for s in samples for sp in s)
    sample = np.empty(n, np.int32)
    seg = np.full(n, -1, np.int32)
    noise = np.full(n, -1, np.int32)
    t = 0
    next_seg = 0
    for si, s in enumerate(samples):
        group_seg: Dict[int, int] = {}
        for sp in s:
            a, b = t, t + sp.length
            sample[a:b] = si
            if sp.mode == "causal":
                pass
            elif sp.mode == "full":
                seg[a:b] = next_seg
                next_seg += 1
            elif sp.mode == "noise":
                seg[a:b] = next_seg
                noise[a:b] = next_seg
                next_seg += 1
            elif sp.mode == "group":
                if sp.group not in group_seg:
                    group_seg[sp.group] = next_seg
                    next_seg += 1
                seg[a:b] = group_seg[sp.group]
            else:
                raise ValueError(f"unknown span mode {sp.mode!r}")
            t = b
    return {"sample": sample, "seg": seg, "noise": noise}


def _truncate(samples: List[List[Span]], n: int) -> List[List[Span]]:
    """Keep the first ``n`` tokens of a list of samples (the last one is cut)."""
    out: List[List[Span]] = []
    left = n
    for s in samples:
        if left <= 0:
            break
        cur: List[Span] = []
        for sp in s:
            if left <= 0:
                break
            L = min(sp.length, left)
            cur.append(Span(sp.mode, L, sp.group))
            left -= L
        out.append(cur)
    if left > 0:
        raise ValueError("not enough samples to fill the pack")
    return out


# --------------------------------------------------------------------------------------
# sample-mix recipes
# --------------------------------------------------------------------------------------
def _lognormal_len(rng: np.random.Generator, median: float = 650.0, sigma: float = 1.5,
                   lo: int = 16, hi: int = 16384) -> int:
    return int(np.clip(round(rng.lognormal(math.log(median), sigma)), lo, hi))


def packed_mix_samples(rng: np.random.Generator, n: int) -> List[List[Span]]:
    """60 % text / 30 % image / 10 % generated-image samples, lognormal text lengths.

    text:      one causal span of L tokens
    image:     a bidirectional image span of I ~ U[256, 4096] tokens, then a causal caption of L
    generated: a causal prompt of L, a noise image span of I ~ U[256, 4096], then a causal
               tail of max(16, L // 4) tokens that cannot see the noise span
    """
    samples: List[List[Span]] = []
    total = 0
    while total < n:
        L = _lognormal_len(rng)
        u = rng.random()
        if u < 0.6:
            s = [Span("causal", L)]
        elif u < 0.9:
            img = int(rng.integers(256, 4097))
            s = [Span("full", img), Span("causal", L)]
        else:
            img = int(rng.integers(256, 4097))
            s = [Span("causal", L), Span("noise", img), Span("causal", max(16, L // 4))]
        samples.append(s)
        total += sum(sp.length for sp in s)
    return _truncate(samples, n)


def grouped_image_samples(rng: np.random.Generator, n: int) -> List[List[Span]]:
    """Image-group samples: text U[1024, 8192], then 2..8 x (4096-token image + text).

    All images of a sample form one group (joint bidirectional attention); each image is,
    with probability 0.1, a generated image instead (own noise span, hidden from later).
    """
    samples: List[List[Span]] = []
    total = 0
    while total < n:
        s = [Span("causal", int(rng.integers(1024, 8193)))]
        for _ in range(int(rng.integers(2, 9))):
            if rng.random() < 0.1:
                s.append(Span("noise", 4096))
            else:
                s.append(Span("group", 4096, group=0))
            s.append(Span("causal", int(rng.integers(1024, 8193))))
        samples.append(s)
        total += sum(sp.length for sp in s)
    return _truncate(samples, n)


def video_generation_samples(rng: np.random.Generator, n: int,
                             sample_tokens: Tuple[int, int] = (131072, 1048576)
                             ) -> List[List[Span]]:
    """Long-video generation samples of interleaved noise and clean frames (the pack the
    MARBLE post's chunked ring attention is built for, section 03): a causal text prompt of
    U[64, 512] tokens, then frames of F ~ U{512, 1024, 2048} tokens (one F per sample), each
    frame as a noise span (the frame being generated: bidirectional within itself, sees
    the clean tokens before it, hidden from every later span) followed by the same frame
    clean (a bidirectional span that later frames see), until the sample holds about
    U[sample_tokens] tokens.
    """
    samples: List[List[Span]] = []
    total = 0
    while total < n:
        target = int(rng.integers(sample_tokens[0], sample_tokens[1] + 1))
        F = int(rng.choice([512, 1024, 2048]))
        s = [Span("causal", int(rng.integers(64, 513)))]
        size = s[0].length
        while size < target:
            s.append(Span("noise", F))
            s.append(Span("full", F))
            size += 2 * F
        samples.append(s)
        total += size
    return _truncate(samples, n)


def video_group_samples(rng: np.random.Generator, n: int) -> List[List[Span]]:
    """Video question-answer samples whose frames form one image group (the vision-group
    packs the MARBLE post's layout transform is built for, section 04): a causal prompt of
    U[64, 512] tokens, then 32..256 frames of F ~ U{64, 128, 192, 256} tokens (one F per
    sample, all frames one group: joint bidirectional attention) each followed by a causal
    timestamp of U[4, 16] tokens, then a causal answer of U[64, 1024] tokens.
    """
    samples: List[List[Span]] = []
    total = 0
    while total < n:
        F = int(rng.choice([64, 128, 192, 256]))
        s = [Span("causal", int(rng.integers(64, 513)))]
        for _ in range(int(rng.integers(32, 257))):
            s.append(Span("group", F, group=0))
            s.append(Span("causal", int(rng.integers(4, 17))))
        s.append(Span("causal", int(rng.integers(64, 1025))))
        samples.append(s)
        total += sum(sp.length for sp in s)
    return _truncate(samples, n)


# --------------------------------------------------------------------------------------
# configurations
# --------------------------------------------------------------------------------------
@dataclasses.dataclass(frozen=True)
class Config:
    cid: int
    name: str
    n: int
    hq: int
    hkv: int
    d: int
    shards: int          # P virtual shards
    order: str           # "contiguous" | "ptrr_block" | "ptrr_chunk"
    window: int = WINDOW_INF
    chunk_tokens: int = 0
    needed: bool = False  # run each q shard once over its needed KV blocks
    range_cost: int = 0   # chunk-layout search: tau, legal pairs per range and step
    bwd: bool = True
    description: str = ""


CONFIGS: Dict[int, Config] = {
    1: Config(1, "tiny_packed_fwd", 2048, 2, 2, 64, 4, "contiguous", bwd=False,
              description="N=2048, 2 heads, d=64; samples [768 causal text, 1024 bidirectional "
                          "image, 256 causal text]; P=4 contiguous; forward + LSE"),
    2: Config(2, "packed_multimodal_64k", 65536, 16, 16, 128, 8, "ptrr_block",
              description="N=65536, 16/16 heads, d=128; lognormal sample mix 60/30/10; P=8 PTRR"),
    3: Config(3, "sliding_window_256k", 262144, 32, 8, 128, 16, "contiguous", window=4096,
              needed=True,
              description="N=262144 single causal sample, GQA 32/8, d=128, W=4096; P=16 "
                          "contiguous shards, needed KV blocks only"),
    4: Config(4, "chunked_long_generation_1m", 1048576, 8, 8, 128, 16, "ptrr_chunk",
              chunk_tokens=16384,
              description="N=1048576: one 524288-token causal generation + packed mix; "
                          "PTRR over 16K-token chunks, P=16"),
    5: Config(5, "grouped_image_2m", 2097152, 8, 8, 128, 32, "ptrr_block",
              description="N=2097152 image-group samples (2-8 x 4096-token images in one group, "
                          "interleaved text, 10% generated); P=32 PTRR"),
}

# workloads beyond the five configurations above: not bench headline cases
EXTRA: Dict[int, Config] = {
    6: Config(6, "video_generation_1m", 1048576, 8, 8, 128, 16, "chunk_search",
              range_cost=167800,
              description="N=1048576 long-video generation samples (128K-1M tokens of "
                          "interleaved noise / clean frames); P=16, searched chunk layout, "
                          "tau = 167800 legal pairs (fitted to emulated ring times on GB300)"),
    7: Config(7, "video_group_512k", 524288, 8, 8, 128, 16, "ptrr_block",
              description="N=524288 video question-answer samples, frames of 64-256 tokens in "
                          "one image group with timestamps between; P=16 PTRR"),
    8: Config(8, "full_span", 262144, 8, 8, 128, 16, "contiguous",
              description="one bidirectional sample filling the pack: every tile full (the "
                          "dense reference for per-tile throughput); P=16 contiguous"),
}


def config_samples(cid: int, n: Optional[int] = None) -> List[List[Span]]:
    """Samples of configuration ``cid``; ``n`` shrinks the pack (mini variants)."""
    cfg = CONFIGS[cid] if cid in CONFIGS else EXTRA[cid]
    n = cfg.n if n is None else n
    rng = np.random.default_rng(100 + cid)
    if cid == 1:
        if n != 2048:
            raise ValueError("config 1 has a fixed layout")
        return [[Span("causal", 768)], [Span("full", 1024)], [Span("causal", 256)]]
    if cid == 2:
        return packed_mix_samples(rng, n)
    if cid == 3:
        return [[Span("causal", n)]]
    if cid == 4:
        gen = n // 2
        return [[Span("causal", gen)]] + packed_mix_samples(rng, n - gen)
    if cid == 5:
        return grouped_image_samples(rng, n)
    if cid == 6:
        return video_generation_samples(rng, n, (min(n, 131072), min(n, 1048576)))
    if cid == 7:
        return video_group_samples(rng, n)
    if cid == 8:
        return [[Span("full", n)]]
    raise KeyError(cid)


def config_tracks(cid: int, n: Optional[int] = None) -> Dict[str, np.ndarray]:
    return tracks_from_samples(config_samples(cid, n))


def mini_config(cid: int, n: int = 16384, hq: Optional[int] = None,
                hkv: Optional[int] = None) -> Config:
    """A small variant of config ``cid`` (same recipe, fewer tokens/heads)."""
    c = CONFIGS[cid] if cid in CONFIGS else EXTRA[cid]
    hq = hq if hq is not None else min(c.hq, 4)
    hkv = hkv if hkv is not None else (hq if c.hq == c.hkv else max(1, hq // (c.hq // c.hkv)))
    window = c.window if c.window == WINDOW_INF else min(c.window, n // 8)
    chunk = 0
    if c.order == "ptrr_chunk":
        chunk = max(BLOCK, n // (2 * c.shards)) // BLOCK * BLOCK
    return dataclasses.replace(c, name=c.name + f"_mini{n}", n=n, hq=hq, hkv=hkv,
                               window=window, chunk_tokens=chunk)


def random_samples(rng: np.random.Generator, n: int, max_samples: int = 6,
                   allow_groups: bool = True) -> List[List[Span]]:
    """A random small pack exercising every span mode (for fuzz / brute-force tests)."""
    samples: List[List[Span]] = []
    total = 0
    modes = ["causal", "full", "noise"] + (["group"] if allow_groups else [])
    while total < n:
        s: List[Span] = []
        for _ in range(int(rng.integers(1, 5))):
            L = int(rng.integers(1, max(2, n // max_samples)))
            m = modes[int(rng.integers(0, len(modes)))]
            s.append(Span(m, L, group=int(rng.integers(0, 2))))
        samples.append(s)
        total += sum(sp.length for sp in s)
    return _truncate(samples, n)


def random_pack(rng: np.random.Generator, n: int, max_samples: int = 6,
                allow_groups: bool = True) -> Dict[str, np.ndarray]:
    return tracks_from_samples(random_samples(rng, n, max_samples, allow_groups))


# --------------------------------------------------------------------------------------
# tensors
# --------------------------------------------------------------------------------------
def make_qkvdo(n: int, hq: int, hkv: int, d: int, device="cpu", seed: int = 0):
    """Q, K, V, dO ~ N(0, 1) in fp32 from one seeded torch generator (drawn in that order),
    rounded to bf16.  Layouts: Q, dO [n, hq, d]; K, V [n, hkv, d]; original token order."""
    import torch

    g = torch.Generator(device=device)
    g.manual_seed(seed)
    out = []
    for h in (hq, hkv, hkv, hq):
        out.append(torch.randn((n, h, d), generator=g, device=device,
                               dtype=torch.float32).to(torch.bfloat16))
    return tuple(out)
