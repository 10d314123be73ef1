"""Pins for the oracle's dtype conversions.

The oracle writes widening and round-to-nearest-even narrowing from the IEEE
definitions.  They are pinned here against (a) torch's CPU casts, exhaustively
over every bit pattern, and (b) the defining property of round-to-nearest
(no representable value is closer; ties go to the even pattern), evaluated in
exact binary64 arithmetic, which uses neither torch nor the oracle's code.
"""
from concurrent.futures import ThreadPoolExecutor

import numpy as np
import pytest
import torch

import oracle
from _util import decode64

TORCH = {oracle.BF16: torch.bfloat16, oracle.FP16: torch.float16}
NAME = {oracle.BF16: "bf16", oracle.FP16: "fp16"}


@pytest.mark.parametrize("dt", [oracle.BF16, oracle.FP16])
def test_widen_exhaustive(oracle_lib, dt):
    pats = np.arange(1 << 16, dtype=np.uint32).astype(np.uint16)
    ours = oracle.widen(pats, dt, oracle_lib)
    ref = torch.from_numpy(pats.view(np.int16)).view(TORCH[dt]).float().numpy()
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(ours), nan)
    assert np.array_equal(ours[~nan].view(np.uint32), ref[~nan].view(np.uint32))


def _chunk_mismatches(args):
    dt, start, count = args
    u = np.arange(start, start + count, dtype=np.uint64).astype(np.uint32)
    f = u.view(np.float32)
    ours = oracle.round_f32(f, dt)
    ref = torch.from_numpy(f).to(TORCH[dt]).view(torch.int16).numpy().view(np.uint16)
    nan = np.isnan(f)
    # NaN inputs: compare as a class (the result must be a NaN pattern)
    exp_all_ones = {oracle.BF16: 0x7F80, oracle.FP16: 0x7C00}[dt]
    frac_mask = {oracle.BF16: 0x007F, oracle.FP16: 0x03FF}[dt]
    ours_nan = ((ours & exp_all_ones) == exp_all_ones) & ((ours & frac_mask) != 0)
    bad = int(np.count_nonzero((ours != ref) & ~nan)) + int(np.count_nonzero(nan & ~ours_nan))
    return bad


@pytest.mark.parametrize("dt", [oracle.BF16, oracle.FP16])
def test_round_exhaustive_vs_torch(oracle_lib, dt):
    """Every one of the 2^32 binary32 patterns rounds as torch's CPU cast."""
    chunk = 1 << 24
    jobs = [(dt, s, chunk) for s in range(0, 1 << 32, chunk)]
    with ThreadPoolExecutor(max_workers=8) as ex:
        bad = sum(ex.map(_chunk_mismatches, jobs))
    assert bad == 0


def _neighbour_value(mag: np.ndarray, dt: int) -> np.ndarray:
    """Value of a magnitude pattern, with the infinity pattern standing for
    the next power of two (IEEE's overflow rule rounds as if the exponent
    range were unbounded)."""
    inf_pat = {oracle.BF16: 0x7F80, oracle.FP16: 0x7C00}[dt]
    inf_val = {oracle.BF16: 2.0 ** 128, oracle.FP16: 2.0 ** 16}[dt]
    v = decode64(mag.astype(np.uint16), NAME[dt])
    return np.where(mag == inf_pat, inf_val, v)


def _check_nearest(x: np.ndarray, y: np.ndarray, dt: int):
    """Assert y = RNE(x) by the definition, in exact binary64 arithmetic."""
    xs = x.astype(np.float64)
    sign_x = np.signbit(xs)
    y32 = y.astype(np.uint32)
    sign_y = (y32 >> 15) == 1
    mag = (y32 & 0x7FFF).astype(np.int64)
    ax = np.abs(xs)
    # the sign is kept (zero included)
    assert np.array_equal(sign_x, sign_y)
    vy = _neighbour_value(mag, dt)
    d0 = np.abs(ax - vy)
    lo = np.maximum(mag - 1, 0)
    hi = mag + 1
    inf_pat = {oracle.BF16: 0x7F80, oracle.FP16: 0x7C00}[dt]
    dlo = np.where(mag > 0, np.abs(ax - _neighbour_value(lo, dt)), np.inf)
    dhi = np.where(mag < inf_pat, np.abs(ax - _neighbour_value(np.minimum(hi, inf_pat), dt)), np.inf)
    assert np.all(d0 <= dlo), "a smaller neighbour is nearer"
    assert np.all(d0 <= dhi), "a larger neighbour is nearer"
    tie = (d0 == dlo) | (d0 == dhi)
    tie &= d0 > 0
    assert np.all((mag[tie] & 1) == 0), "a tie went to the odd pattern"


@pytest.mark.parametrize("dt", [oracle.BF16, oracle.FP16])
def test_round_is_nearest_even_by_definition(oracle_lib, dt):
    rng = np.random.default_rng(1234)
    pats = rng.integers(0, 1 << 32, size=1 << 21, dtype=np.uint64).astype(np.uint32)
    # every exactly-halfway pattern of every binade, and its two neighbours
    if dt == oracle.BF16:
        mids = (np.arange(1 << 15, dtype=np.uint32) << np.uint32(16)) | np.uint32(0x8000)
    else:
        # binary16 halfway points, written as binary32 patterns: value
        # (2q + 1) * 2^(Q - 1) for each quantum exponent Q of binary16
        qs = np.arange(0, 2048, dtype=np.float64)
        vals = np.concatenate([(2 * qs + 1) * 2.0 ** (Q - 1) for Q in range(-24, 6)])
        mids = vals.astype(np.float32).view(np.uint32)
    extra = np.concatenate([mids, mids - 1, mids + 1])
    pats = np.concatenate([pats, extra, extra | np.uint32(0x80000000)])
    f = pats.view(np.float32)
    f = f[np.isfinite(f)]
    y = oracle.round_f32(f, dt, oracle_lib)
    _check_nearest(f, y, dt)


def test_fp32_round_is_identity(oracle_lib):
    rng = np.random.default_rng(5)
    f = rng.integers(0, 1 << 32, size=1 << 16, dtype=np.uint64).astype(np.uint32).view(np.float32)
    y = oracle.round_f32(f, oracle.FP32, oracle_lib)
    assert np.array_equal(y.view(np.uint32), f.view(np.uint32))
