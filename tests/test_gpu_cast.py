"""The gradient cast (marble_cast_bf16, fp32 -> bf16, round to nearest even) and the
permutations that bring results back to original order (marble_permute, and
marble_permute_cast_bf16 which fuses the two), against the oracle planner's permutation
and the oracle's rounding (oracle/ring.py round_bf16, pinned on ties and on the library's
own conversion), bit for bit: random values over the whole fp32 range, exact ties, signed
zeros, subnormals, infinities and values that round up to infinity."""
import numpy as np
import pytest
import torch

import context_attention_metadata_gb300 as M
import workloads as wl
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


@pytest.mark.parametrize("n,row_elems,inverse,P", [(2048, 2048, 1, 4), (8192, 1024, 1, 8),
                                                    (4096, 4096, 0, 8), (1024, 12, 1, 2),
                                                    (1152, 260, 0, 3)])
def test_permute_cast_bf16_matches_oracle_order_and_rounding(n, row_elems, inverse, P):
    """marble_permute_cast_bf16: the oracle planner's token permutation (PTRR over blocks)
    applied to rows of fp32, each element rounded by the oracle's round_bf16, bit for bit.
    Rows of 12 and 260 elements leave a ragged last chunk group per block of threads."""
    from marble_testlib import make_plan
    from oracle import plan as oplan
    rng = np.random.default_rng(n + row_elems)
    tr = wl.random_pack(rng, n, max_samples=5)
    pl = make_plan(tr, wl.WINDOW_INF, P, "ptrr_block")
    perm = oplan.make_plan(tr, wl.WINDOW_INF, P, "ptrr_block").perm.astype(np.int64)
    x = _inputs(rng, n * row_elems)[: n * row_elems].reshape(n, row_elems)
    src = torch.from_numpy(np.ascontiguousarray(x)).cuda()
    got = pl.permute_cast_bf16(src, inverse=bool(inverse))
    torch.cuda.synchronize()
    got = got.cpu().view(torch.int16).numpy().view(np.uint16)
    r = (ring.round_bf16(x).astype(np.float32).view(np.uint32) >> 16).astype(np.uint16)
    want = np.empty_like(r)
    if inverse:
        want[perm] = r
    else:
        want[:] = r[perm]
    assert (got == want).all(), np.argwhere(got != want)[:8]


@pytest.mark.parametrize("row_bytes", [16, 4096, 8192, 48, 12])
def test_permute_rows_match_oracle_order(row_bytes):
    """marble_permute gathers and scatters whole rows by the oracle planner's permutation,
    for rows of 16-byte chunks (one to 512 per row) and rows of 4-byte words."""
    from marble_testlib import make_plan
    from oracle import plan as oplan
    n, P = 2048, 4
    rng = np.random.default_rng(row_bytes)
    tr = wl.random_pack(rng, n, max_samples=4)
    pl = make_plan(tr, wl.WINDOW_INF, P, "ptrr_block")
    perm = oplan.make_plan(tr, wl.WINDOW_INF, P, "ptrr_block").perm.astype(np.int64)
    x = rng.integers(-2**31, 2**31, size=(n, row_bytes // 4), dtype=np.int64).astype(np.int32)
    src = torch.from_numpy(x).cuda()
    fwd = pl.permute(src).cpu().numpy()
    back = pl.permute(src, inverse=True).cpu().numpy()
    assert (fwd == x[perm]).all()
    want = np.empty_like(x)
    want[perm] = x
    assert (back == want).all()
