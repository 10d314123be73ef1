"""Pins for the oracle's all-reduce fold and its reduce-scatter step.

The first four kinds of check below do not restate the fold.  The last
restates it with independent host libraries (numpy's binary32 adds, torch's
narrowing casts) that share no code with the oracle's C arithmetic.  The
oracle is checked against:
  * hand-derived IEEE cases (tests/golden/fold_cases.json), which fix the rank
    order, binary32 accumulation, a single final rounding, the start from
    rank 0's value (signed zeros), subnormals and overflow;
  * exact closed forms: small integers and short dyadic fractions, whose
    partial sums are exact, so the result is the exact sum (Python integers
    or binary64) rounded once by torch's cast;
  * brute-force binary64 sums within the error bound of an (R-1)-add binary32
    fold plus one final rounding;
  * invariants: identical outputs, a single non-zero rank, x and -x,
    R = 1, rank permutation;
  * torch on the host: for R = 2, (a.float() + b.float()).to(dtype); for any
    R, an elementwise numpy binary32 left fold narrowed by torch's cast.
"""
import numpy as np
import pytest
import torch

import oracle
from all_reduce_reduction_gb300 import workload as wl
from _util import DT_CODE, as_uint, decode64, golden, hex_array, spacing

DTYPES = ["bf16", "fp16", "fp32"]


def _run(ins, dtype):
    return oracle.allreduce(ins, DT_CODE[dtype])


@pytest.mark.parametrize("case", golden("fold_cases.json")["cases"], ids=lambda c: c["name"])
def test_golden_cases(case):
    dt = case["dtype"]
    ins = [hex_array([h], dt) for h in case["inputs"]]
    outs = _run(ins, dt)
    want = int(case["expected"], 16)
    for o in outs:
        assert int(as_uint(o, dt)[0]) == want, case["derivation"]


def _inputs(dist, R, n, dtype, config=90):
    return [wl.bits(t) for t in wl.make_inputs(config, R, n, dtype, dist)]


@pytest.mark.parametrize("dtype", DTYPES)
@pytest.mark.parametrize("R", [1, 2, 3, 7, 8, 16, 32])
def test_integer_sums_are_exact(dtype, R):
    """Integers in [-8, 8]: every partial sum (|s| <= 256) is exact in binary32
    and in every dtype, so the output is the integer sum itself."""
    n = 1031
    ts = wl.make_inputs(91, R, n, dtype, "integer")
    ins = [wl.bits(t) for t in ts]
    exact = sum(t.to(torch.int64) for t in ts)           # Python-exact integers
    want = wl.bits(exact.to(torch.float64).to(wl.TORCH_DTYPE[dtype]))
    for o in _run(ins, dtype):
        assert np.array_equal(as_uint(o, dtype), as_uint(want, dtype))


@pytest.mark.parametrize("dtype", DTYPES)
@pytest.mark.parametrize("R", [2, 5, 8, 32])
def test_dyadic_sums_round_once(dtype, R):
    """Multiples of 2^-6 in (-1, 1): partial sums need < 24 bits, so binary32
    holds them exactly and the result is the exact binary64 sum rounded once
    (by torch's cast) to the dtype -- bits beyond the dtype's precision make
    the final rounding matter."""
    n = 2048
    rng = np.random.default_rng(R)
    q = rng.integers(-63, 64, size=(R, n)).astype(np.float64) / 64.0
    ts = [torch.from_numpy(q[r]).to(wl.TORCH_DTYPE[dtype]) for r in range(R)]
    # the inputs are representable (7 significant bits fit every dtype)
    assert all(np.array_equal(t.double().numpy(), q[r]) for r, t in enumerate(ts))
    exact = q.sum(axis=0)                                 # exact in binary64
    want = wl.bits(torch.from_numpy(exact).to(wl.TORCH_DTYPE[dtype]))
    outs = _run([wl.bits(t) for t in ts], dtype)
    for o in outs:
        assert np.array_equal(as_uint(o, dtype), as_uint(want, dtype))


def _bound_check(ins, outs, dtype):
    R = len(ins)
    x = np.stack([decode64(a, dtype) for a in ins])
    s = x.sum(axis=0)                                     # binary64
    abs_sum = np.abs(x).sum(axis=0)
    y = decode64(outs[0], dtype)
    tol = spacing(s, dtype) + R * 2.0 ** -24 * abs_sum
    finite = np.isfinite(y)
    # an infinite output is only allowed beyond the dtype's overflow threshold
    big = {"bf16": 3.3961775292304e38, "fp16": 65520.0, "fp32": 3.4028235677973366e38}[dtype]
    assert np.all(np.abs(s[~finite]) + R * 2.0 ** -24 * abs_sum[~finite] >= big)
    assert np.all(np.sign(y[~finite]) == np.sign(s[~finite]))
    err = np.abs(y[finite] - s[finite])
    assert np.all(err <= tol[finite]), float(np.max(err - tol[finite]))


@pytest.mark.parametrize("dtype", DTYPES)
@pytest.mark.parametrize("dist", ["uniform", "normal", "loguniform"])
@pytest.mark.parametrize("R", [1, 2, 4, 8, 16, 32])
def test_within_binary64_bound(dtype, dist, R):
    """|y - sum_fp64| <= ulp_dtype(sum) + R * 2^-24 * sum|x| (rounding-error
    bound of R-1 binary32 adds plus one final rounding)."""
    ins = _inputs(dist, R, 4099, dtype)
    outs = _run(ins, dtype)
    _bound_check(ins, outs, dtype)


@pytest.mark.parametrize("dtype", DTYPES)
def test_all_outputs_identical(dtype):
    ins = _inputs("loguniform", 9, 777, dtype)
    outs = _run(ins, dtype)
    for o in outs[1:]:
        assert np.array_equal(as_uint(o, dtype), as_uint(outs[0], dtype))


NEG_ZERO = {"bf16": 0x8000, "fp16": 0x8000, "fp32": 0x80000000}
UINT = {"bf16": np.uint16, "fp16": np.uint16, "fp32": np.uint32}


@pytest.mark.parametrize("dtype", DTYPES)
@pytest.mark.parametrize("R,who", [(2, 0), (2, 1), (8, 5), (32, 31), (32, 0)])
def test_single_nonzero_rank_is_exact(dtype, R, who):
    """Ranks filled with -0 leave the non-zero rank's value bit for bit
    (x + -0 = x for every x); with +0 filling only the sign of a zero input
    may change."""
    n = 1000
    x = _inputs("loguniform", 1, n, dtype, config=92)[0]
    x_u = as_uint(x, dtype).copy()
    x_u[:7] = [0, NEG_ZERO[dtype], 0, 0, NEG_ZERO[dtype], 0, 0]
    x = x_u.view(oracle.STORAGE[DT_CODE[dtype]])
    negz = np.full(n, NEG_ZERO[dtype], dtype=UINT[dtype]).view(x.dtype)
    ins = [x if r == who else negz.copy() for r in range(R)]
    out = _run(ins, dtype)[0]
    assert np.array_equal(as_uint(out, dtype), x_u)
    posz = np.zeros(n, dtype=x.dtype)
    ins = [x if r == who else posz.copy() for r in range(R)]
    out = decode64(_run(ins, dtype)[0], dtype)
    assert np.array_equal(out, decode64(x, dtype))        # equal as values


@pytest.mark.parametrize("dtype", DTYPES)
def test_x_and_minus_x_cancel(dtype):
    x = _inputs("loguniform", 1, 999, dtype, config=93)[0]
    neg = (as_uint(x, dtype) ^ UINT[dtype](NEG_ZERO[dtype])).view(x.dtype)
    for ins in ([x, neg], [x, neg, neg, x]):
        out = as_uint(_run(ins, dtype)[0], dtype)
        assert np.all(out == 0)                           # +0 exactly


@pytest.mark.parametrize("dtype", DTYPES)
def test_single_rank_is_copy(dtype):
    x = _inputs("normal", 1, 1234, dtype, config=94)[0]
    out = _run([x], dtype)[0]
    assert np.array_equal(as_uint(out, dtype), as_uint(x, dtype))


@pytest.mark.parametrize("dtype", DTYPES)
def test_rank_permutation_within_bound(dtype):
    ins = _inputs("loguniform", 16, 2000, dtype, config=95)
    perm = list(np.random.default_rng(3).permutation(16))
    a = _run(ins, dtype)
    b = _run([ins[p] for p in perm], dtype)
    _bound_check(ins, a, dtype)
    _bound_check([ins[p] for p in perm], b, dtype)
    if dtype == "fp32":
        # at binary32 output precision the order is observable
        assert not np.array_equal(as_uint(a[0], dtype), as_uint(b[0], dtype))


@pytest.mark.parametrize("dtype", DTYPES)
@pytest.mark.parametrize("R,n", [(1, 5), (3, 10), (4, 4097 * 3 + 3), (8, 64), (16, 1001), (32, 7), (32, 12345)])
def test_shard_bounds_partition(dtype, R, n):
    per_vec = 16 // wl.ELEM_SIZE[dtype]
    S = -(-n // R)
    S = -(-S // per_vec) * per_vec
    prev = 0
    for j in range(R):
        lo, hi = oracle.shard_bounds(R, n, DT_CODE[dtype], j)
        assert lo == min(n, j * S) and hi == min(n, (j + 1) * S)
        assert lo == prev and hi >= lo
        prev = hi
    assert prev == n


@pytest.mark.parametrize("dtype", DTYPES)
@pytest.mark.parametrize("R,n", [(4, 4097 * 3 + 3), (8, 64), (16, 1001), (5, 9)])
def test_reduce_scatter_writes_only_its_shard(dtype, R, n):
    ins = _inputs("normal", R, n, dtype, config=96)
    full = _run(ins, dtype)[0]
    sentinel = {"bf16": 0x7FC1, "fp16": 0x7E01, "fp32": 0x7FC00001}[dtype]
    outs = [np.full(n, sentinel, dtype=UINT[dtype]).view(ins[0].dtype) for _ in range(R)]
    oracle.reduce_scatter(ins, DT_CODE[dtype], outs)
    for j in range(R):
        lo, hi = oracle.shard_bounds(R, n, DT_CODE[dtype], j)
        o = as_uint(outs[j], dtype)
        assert np.array_equal(o[lo:hi], as_uint(full, dtype)[lo:hi])
        assert np.all(o[:lo] == sentinel) and np.all(o[hi:] == sentinel)


@pytest.mark.parametrize("dtype", DTYPES)
@pytest.mark.parametrize("dist", ["uniform", "normal", "loguniform"])
def test_two_ranks_equal_torch_add(dtype, dist):
    """R = 2: one binary32 add and one rounding, i.e. torch's own
    (a.float() + b.float()).to(dtype) on the host."""
    a, b = wl.make_inputs(60, 2, 20011, dtype, dist)
    want = wl.bits((a.float() + b.float()).to(wl.TORCH_DTYPE[dtype]))
    got = _run([wl.bits(a), wl.bits(b)], dtype)[0]
    assert np.array_equal(as_uint(got, dtype), as_uint(want, dtype))


@pytest.mark.parametrize("dtype", DTYPES)
@pytest.mark.parametrize("R", [3, 8, 32])
@pytest.mark.parametrize("dist", ["normal", "loguniform"])
def test_equals_numpy_binary32_left_fold(dtype, R, dist):
    """Any R: numpy's elementwise binary32 adds in rank order (IEEE round to
    nearest even, no contraction), narrowed once by torch's cast."""
    ins = wl.make_inputs(61, R, 7001, dtype, dist)
    acc = ins[0].float().numpy().copy()
    with np.errstate(over="ignore"):
        for t in ins[1:]:
            acc = acc + t.float().numpy()
    want = wl.bits(torch.from_numpy(acc).to(wl.TORCH_DTYPE[dtype]))
    got = _run([wl.bits(t) for t in ins], dtype)[0]
    assert np.array_equal(as_uint(got, dtype), as_uint(want, dtype))
