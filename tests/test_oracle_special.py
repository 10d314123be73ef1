"""The oracle on edge-of-format inputs (signed zeros, subnormals, smallest
normals, sums that overflow), pinned against an independent restatement of
the fold: numpy binary32 adds in rank order (IEEE round to nearest even, no
flush to zero on the host) and torch's CPU narrowing to bf16/fp16.  These are
the inputs the GPU special-value parity cases use."""
import numpy as np
import pytest
import torch

import oracle
from all_reduce_reduction_gb300 import workload as wl


def numpy_fold(ins, dtype):
    with np.errstate(over="ignore", invalid="ignore"):
        acc = wl.bits(ins[0]).astype(np.float32) if dtype == "fp32" else ins[0].float().numpy()
        acc = acc.copy()
        for t in ins[1:]:
            acc = acc + (t.numpy() if dtype == "fp32" else t.float().numpy())
    return wl.bits(torch.from_numpy(acc).to(wl.TORCH_DTYPE[dtype]))


@pytest.mark.parametrize("dtype", ["bf16", "fp16", "fp32"])
@pytest.mark.parametrize("R", [2, 5, 16])
def test_oracle_special_values_match_numpy_fold(dtype, R):
    ins = wl.special_inputs(0x5E1 + R, R, 4099, dtype)
    got = oracle.allreduce([wl.bits(t) for t in ins], wl.DTYPE_CODE[dtype])[0]
    want = numpy_fold(ins, dtype)
    u = np.uint32 if dtype == "fp32" else np.uint16
    assert np.array_equal(np.ascontiguousarray(got).view(u), np.ascontiguousarray(want).view(u))


@pytest.mark.parametrize("dtype", ["bf16", "fp16", "fp32"])
def test_special_inputs_reach_subnormal_and_infinite_results(dtype):
    """The pool really exercises the edges: some results are subnormal and
    nonzero, some are infinite."""
    ins = wl.special_inputs(0x5E1 + 5, 5, 4099, dtype)
    y = oracle.allreduce([wl.bits(t) for t in ins], wl.DTYPE_CODE[dtype])[0]
    v = wl.from_bits(y, dtype).float()
    tiny = torch.finfo(wl.TORCH_DTYPE[dtype]).tiny
    assert bool(((v != 0) & (v.abs() < tiny)).any())
    assert bool(torch.isinf(v).any())


@pytest.mark.parametrize("dtype", ["bf16", "fp16", "fp32"])
@pytest.mark.parametrize("H", [72, 70])
def test_oracle_combine_special_values_match_numpy(dtype, H):
    """The weighted combine on the same pools: numpy binary32 products, each
    rounded on its own, folded in source order, then torch's narrowing."""
    K, T = 4, 7
    ys = wl.special_inputs(0x5E2, K, T * H, dtype)
    w = wl.special_weights(0x5E3, T, K)
    got = oracle.combine([wl.bits(t) for t in ys], w, T, H, wl.DTYPE_CODE[dtype])
    x = [(t.numpy() if dtype == "fp32" else t.float().numpy()).reshape(T, H) for t in ys]
    wk = w.reshape(T, K)
    with np.errstate(over="ignore", invalid="ignore", under="ignore"):
        acc = (wk[:, 0:1] * x[0]).astype(np.float32)
        for k in range(1, K):
            acc = acc + (wk[:, k:k + 1] * x[k]).astype(np.float32)
    assert not np.isnan(acc).any()
    want = wl.bits(torch.from_numpy(acc.reshape(-1).copy()).to(wl.TORCH_DTYPE[dtype]))
    u = np.uint32 if dtype == "fp32" else np.uint16
    assert np.array_equal(np.ascontiguousarray(got).view(u), np.ascontiguousarray(want).view(u))
