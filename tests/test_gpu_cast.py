"""The gradient cast (marble_cast_bf16, fp32 -> bf16, round to nearest even) against the
oracle's rounding (oracle/ring.py round_bf16, pinned on ties and on the library's own
conversion), bit for bit: random values over the whole fp32 range, exact ties, signed
zeros, subnormals, infinities and values that round up to infinity."""
import numpy as np
import pytest
import torch

import context_attention_metadata_gb300 as M
from oracle import ring

pytestmark = pytest.mark.gpu


def _inputs(rng, n):
    bits = rng.integers(0, 2**32, size=n, dtype=np.uint64).astype(np.uint32)
    x = bits.view(np.float32).copy()
    x[np.isnan(x)] = 1.0  # NaN has no single rounded value: checked separately
    special = np.array([0.0, -0.0, np.inf, -np.inf, 1e-45, -1e-45, 1.1754942e-38,
                        -1.1754942e-38, 3.3961775e38, 3.4028235e38, -3.4028235e38,
                        1.0 + 2.0**-8, 1.0 + 3 * 2.0**-8, -(1.0 + 2.0**-8), 2.0**-130 * 1.5],
                       np.float32)
    # exact ties: the lower 16 bits of the encoding are 0x8000
    ties = (rng.integers(0, 2**16, size=4096, dtype=np.uint64).astype(np.uint32) << 16) | 0x8000
    ties = ties.view(np.float32)
    ties = ties[np.isfinite(ties)]
    # subnormals
    sub = (rng.integers(1, 2**23, size=4096, dtype=np.uint64).astype(np.uint32)
           | (rng.integers(0, 2, size=4096, dtype=np.uint64).astype(np.uint32) << 31)).view(np.float32)
    x = np.concatenate([special, ties, sub, x])
    pad = (-len(x)) % 4
    return np.concatenate([x, np.ones(pad, np.float32)])


@pytest.mark.parametrize("n", [4, 1 << 20, 3 * (1 << 20) + 52])
def test_cast_bf16_matches_oracle_rounding_bit_for_bit(n):
    rng = np.random.default_rng(n)
    x = _inputs(rng, n)
    src = torch.from_numpy(x).cuda()
    dst = torch.empty(len(x), dtype=torch.bfloat16, device="cuda")
    M.cast_bf16(src, dst)
    torch.cuda.synchronize()
    got = dst.cpu().view(torch.int16).numpy().view(np.uint16)
    want = ring.round_bf16(x).astype(np.float32).view(np.uint32) >> 16
    assert (got == want.astype(np.uint16)).all(), np.flatnonzero(got != want)[:8]


def test_cast_bf16_nan_stays_nan():
    x = np.array([np.nan, -np.nan, 1.0, 2.0], np.float32)
    src = torch.from_numpy(x).cuda()
    dst = torch.empty(4, dtype=torch.bfloat16, device="cuda")
    M.cast_bf16(src, dst)
    out = dst.float().cpu().numpy()
    assert np.isnan(out[:2]).all() and (out[2:] == [1.0, 2.0]).all()
