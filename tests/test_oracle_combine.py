"""Pins for the oracle's weighted per-token combine."""
import numpy as np
import pytest

import oracle
from all_reduce_reduction_gb300 import workload as wl
from _util import DT_CODE, as_uint, decode64, golden, hex_array, spacing

DTYPES = ["bf16", "fp16", "fp32"]


def _ys(K, T, H, dtype, config=87, dist="loguniform"):
    return [wl.bits(t) for t in wl.make_inputs(config, K, T * H, dtype, dist)]


@pytest.mark.parametrize("case", golden("combine_cases.json")["cases"], ids=lambda c: c["name"])
def test_golden_cases(case):
    dt = case["dtype"]
    ys = [hex_array([h], dt) for h in case["y"]]
    w = np.array([int(x, 16) for x in case["w"]], dtype=np.uint32).view(np.float32)
    out = oracle.combine(ys, w, 1, 1, DT_CODE[dt])
    assert int(as_uint(out, dt)[0]) == int(case["expected"], 16), case["derivation"]


@pytest.mark.parametrize("dtype", DTYPES)
@pytest.mark.parametrize("K", [1, 3, 8])
def test_unit_weights_are_the_allreduce(dtype, K):
    T, H = 5, 67
    ys = _ys(K, T, H, dtype)
    out = oracle.combine(ys, np.ones(T * K, np.float32), T, H, DT_CODE[dtype])
    want = oracle.allreduce(ys, DT_CODE[dtype])[0]
    assert np.array_equal(as_uint(out, dtype), as_uint(want, dtype))


@pytest.mark.parametrize("dtype", DTYPES)
def test_power_of_two_weights_scale_exactly(dtype):
    """w[t][k] = 2^e(t,k): every product is exact, so the combine equals the
    all-reduce of inputs pre-scaled by those powers (scaled exactly here in
    binary64 and cast back, exact inside the dtype's range)."""
    K, T, H = 4, 6, 33
    ys = _ys(K, T, H, dtype, dist="uniform")
    rng = np.random.default_rng(9)
    e = rng.integers(-3, 4, size=(T, K))
    w = np.ldexp(1.0, e).astype(np.float32)
    scaled = []
    for k in range(K):
        x = decode64(ys[k], dtype).reshape(T, H) * np.ldexp(1.0, e[:, k])[:, None]
        t = wl.torch.from_numpy(x.reshape(-1)).to(wl.TORCH_DTYPE[dtype])
        assert np.array_equal(t.double().numpy(), x.reshape(-1))      # exact scaling
        scaled.append(wl.bits(t))
    want = oracle.allreduce(scaled, DT_CODE[dtype])[0]
    out = oracle.combine(ys, w.reshape(-1), T, H, DT_CODE[dtype])
    assert np.array_equal(as_uint(out, dtype), as_uint(want, dtype))


@pytest.mark.parametrize("dtype", DTYPES)
def test_one_hot_weights_select_a_source(dtype):
    K, T, H = 5, 7, 40
    ys = _ys(K, T, H, dtype)
    hot = np.arange(T) % K
    w = np.zeros((T, K), np.float32)
    w[np.arange(T), hot] = 1.0
    out = decode64(oracle.combine(ys, w.reshape(-1), T, H, DT_CODE[dtype]), dtype).reshape(T, H)
    for t in range(T):
        assert np.array_equal(out[t], decode64(ys[hot[t]], dtype).reshape(T, H)[t])


@pytest.mark.parametrize("dtype", DTYPES)
@pytest.mark.parametrize("K", [2, 8, 32])
def test_within_binary64_bound(dtype, K):
    """|y - sum w*x| <= ulp(sum) + (K + 1) * 2^-24 * sum|w*x|."""
    T, H = 9, 129
    ys = _ys(K, T, H, dtype, dist="normal")
    w = np.random.default_rng(K).random((T, K)).astype(np.float32)
    out = decode64(oracle.combine(ys, w.reshape(-1), T, H, DT_CODE[dtype]), dtype)
    x = np.stack([decode64(a, dtype) for a in ys]).reshape(K, T, H)
    terms = x * w.T.astype(np.float64)[:, :, None]
    s = terms.sum(axis=0).reshape(-1)
    tol = spacing(s, dtype) + (K + 1) * 2.0 ** -24 * np.abs(terms).sum(axis=0).reshape(-1)
    fin = np.isfinite(out)
    assert np.all(np.abs(out[fin] - s[fin]) <= tol[fin])
