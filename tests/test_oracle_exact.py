"""The oracle's fold against a model of IEEE 754 arithmetic written with
exact rationals: no hardware floating point anywhere in the model.

Every binary32 add of the left fold is the exact rational sum rounded to
nearest, ties to even, at 24 bits with gradual underflow and overflow to
infinity; the final narrowing rounds the binary32 value the same way at the
buffer format's precision and exponent range (bfloat16: 8 bits, exponents of
binary32; binary16: 11 bits, exponents -14..15).  Signed zeros follow IEEE
754 section 6.3: an exact zero sum of two zeros keeps their common sign, any
other exact zero sum is +0 under round-to-nearest, and a nonzero result that
rounds to zero keeps its sign.  Inputs are drawn from the edge-of-format
pools (zeros, subnormals, smallest normals, ones, values near the largest
finite) and from the log-uniform workload recipe.  The weighted combine is
checked the same way, with IEEE binary32 multiplication in the model."""
from fractions import Fraction

import numpy as np
import pytest

import oracle
from all_reduce_reduction_gb300 import workload as wl

# (precision in bits including the leading one, emin, emax)
FORMATS = {"fp32": (24, -126, 127), "bf16": (8, -126, 127), "fp16": (11, -14, 15)}
NAN, INF, FIN = "nan", "inf", "fin"


def _floor_log2(a: Fraction) -> int:
    e = a.numerator.bit_length() - a.denominator.bit_length()
    while Fraction(2) ** e > a:
        e -= 1
    while Fraction(2) ** (e + 1) <= a:
        e += 1
    return e


def _round(value: Fraction, neg: bool, fmt: str):
    """Round a rational of sign `neg` to the format: (kind, neg, value)."""
    p, emin, emax = FORMATS[fmt]
    a = abs(value)
    if a == 0:
        return (FIN, neg, Fraction(0))
    q = max(_floor_log2(a), emin) - (p - 1)            # exponent of the quantum
    m = a / Fraction(2) ** q
    r = m.numerator // m.denominator
    rest = m - r
    if rest > Fraction(1, 2) or (rest == Fraction(1, 2) and r % 2 == 1):
        r += 1
    v = r * Fraction(2) ** q
    if v >= Fraction(2) ** (emax + 1):
        return (INF, neg, None)
    return (FIN, neg, v)


def _decode(bits: int, fmt: str):
    if fmt == "bf16":
        bits, fmt = bits << 16, "fp32"
    if fmt == "fp32":
        neg, e, f = bits >> 31, (bits >> 23) & 0xFF, bits & 0x7FFFFF
        if e == 0xFF:
            return (NAN, bool(neg), None) if f else (INF, bool(neg), None)
        v = Fraction(f, 1 << 149) if e == 0 else Fraction((1 << 23) + f) * Fraction(2) ** (e - 150)
        return (FIN, bool(neg), v)
    neg, e, f = bits >> 15, (bits >> 10) & 0x1F, bits & 0x3FF
    if e == 0x1F:
        return (NAN, bool(neg), None) if f else (INF, bool(neg), None)
    v = Fraction(f, 1 << 24) if e == 0 else Fraction(1024 + f) * Fraction(2) ** (e - 25)
    return (FIN, bool(neg), v)


def _add32(x, y):
    """IEEE binary32 addition, round to nearest even."""
    if x[0] == NAN or y[0] == NAN:
        return (NAN, False, None)
    if x[0] == INF and y[0] == INF:
        return x if x[1] == y[1] else (NAN, False, None)
    if x[0] == INF:
        return x
    if y[0] == INF:
        return y
    sx = -x[2] if x[1] else x[2]
    sy = -y[2] if y[1] else y[2]
    s = sx + sy
    if s == 0:
        if x[2] == 0 and y[2] == 0:
            return (FIN, x[1] and y[1], Fraction(0))
        return (FIN, False, Fraction(0))
    return _round(s, s < 0, "fp32")


def _model(columns, fmt):
    acc = _decode(columns[0], fmt)
    for b in columns[1:]:
        acc = _add32(acc, _decode(b, fmt))
    if fmt == "fp32" or acc[0] != FIN:
        return acc
    return _round(acc[2], acc[1], fmt)


def _same(got, want):
    if want[0] == NAN:
        return got[0] == NAN
    return got == want


def _case(dtype, R, n, inputs):
    u = np.uint32 if dtype == "fp32" else np.uint16
    bits = [np.ascontiguousarray(wl.bits(t)).view(u) for t in inputs]
    out = np.ascontiguousarray(oracle.allreduce([wl.bits(t) for t in inputs],
                                                wl.DTYPE_CODE[dtype])[0]).view(u)
    for i in range(n):
        want = _model([int(b[i]) for b in bits], dtype)
        got = _decode(int(out[i]), dtype)
        assert _same(got, want), (dtype, R, i, [hex(int(b[i])) for b in bits], got, want)


def test_model_rounding_examples():
    # the model itself, on values whose rounding is known by hand
    one = Fraction(1)
    assert _round(one + Fraction(1, 1 << 24), False, "fp32") == (FIN, False, one)      # tie, even
    # 1 + 1.5 quanta: a tie between 1 + 1 and 1 + 2 quanta (2^-23 each), even wins
    assert _round(one + Fraction(3, 1 << 24), False, "fp32") == (FIN, False, one + Fraction(2, 1 << 23))
    assert _round(one + Fraction(3, 1 << 25), False, "fp32") == (FIN, False, one + Fraction(1, 1 << 23))
    assert _round(Fraction(65520), False, "fp16")[0] == INF                        # fp16 overflow tie
    assert _round(Fraction(65519), False, "fp16") == (FIN, False, Fraction(65504))
    assert _round(Fraction(1, 1 << 25), True, "fp16") == (FIN, True, Fraction(0))  # half the quantum
    assert _round(Fraction(3, 1 << 26), False, "fp16") == (FIN, False, Fraction(1, 1 << 24))
    assert _decode(0x0001, "bf16") == (FIN, False, Fraction(1, 1 << 133))
    assert _decode(0x8001, "fp16") == (FIN, True, Fraction(1, 1 << 24))
    assert _add32((FIN, True, Fraction(0)), (FIN, True, Fraction(0))) == (FIN, True, Fraction(0))
    assert _add32((FIN, False, one), (FIN, True, one)) == (FIN, False, Fraction(0))


@pytest.mark.parametrize("dtype", ["bf16", "fp16", "fp32"])
@pytest.mark.parametrize("R", [1, 2, 3, 5, 8])
def test_fold_equals_exact_model_on_edge_values(dtype, R):
    n = 160
    _case(dtype, R, n, wl.special_inputs(300 + R, R, n, dtype))


@pytest.mark.parametrize("dtype", ["bf16", "fp16", "fp32"])
@pytest.mark.parametrize("R", [2, 7, 16])
def test_fold_equals_exact_model_on_loguniform(dtype, R):
    n = 96
    _case(dtype, R, n, wl.make_inputs(310 + R, R, n, dtype, "loguniform"))


def _mul32(x, y):
    """IEEE binary32 multiplication, round to nearest even."""
    neg = x[1] != y[1]
    if x[0] == NAN or y[0] == NAN:
        return (NAN, False, None)
    if x[0] == INF or y[0] == INF:
        other = y if x[0] == INF else x
        if other[0] == FIN and other[2] == 0:
            return (NAN, False, None)                    # infinity times zero
        return (INF, neg, None)
    return _round(x[2] * y[2], neg, "fp32")


def _combine_model(weights, columns, fmt):
    acc = _mul32(_decode(weights[0], "fp32"), _decode(columns[0], fmt))
    for wb, b in zip(weights[1:], columns[1:]):
        acc = _add32(acc, _mul32(_decode(wb, "fp32"), _decode(b, fmt)))
    if fmt == "fp32" or acc[0] != FIN:
        return acc
    return _round(acc[2], acc[1], fmt)


@pytest.mark.parametrize("dtype", ["bf16", "fp16", "fp32"])
@pytest.mark.parametrize("K", [1, 3, 8])
@pytest.mark.parametrize("special", [True, False])
def test_combine_equals_exact_model(dtype, K, special):
    """The weighted combine: every product w[t,k] * y_k[t,h] rounded to
    binary32 on its own, folded left to right from k = 0, rounded once."""
    T, H = 6, 24
    u = np.uint32 if dtype == "fp32" else np.uint16
    if special:
        ys = wl.special_inputs(320 + K, K, T * H, dtype)
        w = wl.special_weights(330 + K, T, K)
    else:
        ys = wl.make_inputs(340 + K, K, T * H, dtype, "loguniform")
        w = wl.gate_weights(350 + K, T, K)
    bits = [np.ascontiguousarray(wl.bits(t)).view(u) for t in ys]
    wbits = np.ascontiguousarray(w, dtype=np.float32).view(np.uint32)
    out = np.ascontiguousarray(oracle.combine([wl.bits(t) for t in ys], w, T, H,
                                              wl.DTYPE_CODE[dtype])).view(u)
    for t in range(T):
        for h in range(H):
            i = t * H + h
            want = _combine_model([int(wbits[t * K + k]) for k in range(K)],
                                  [int(b[i]) for b in bits], dtype)
            got = _decode(int(out[i]), dtype)
            assert _same(got, want), (dtype, K, t, h, got, want)
