"""GPU parity on edge-of-format inputs: signed zeros, subnormals, smallest
normals and sums that overflow to infinity.  Nothing on the device may flush
subnormals to zero or round other than to nearest even; every path must give
the oracle's bits."""
import numpy as np
import pytest
import torch

import all_reduce_reduction_gb300 as ar
import oracle
from all_reduce_reduction_gb300 import workload as wl
from gpu_helpers import (ALL_PATHS, PATH_IDS, assert_bits_equal, check_guards, device_inputs,
                         expected, guarded_outputs, need_gpu)

pytestmark = pytest.mark.gpu

DTYPES = ["bf16", "fp16", "fp32"]


def _allreduce_case(R, n, dtype, algo, proto, inplace=False):
    need_gpu()
    cpu = wl.special_inputs(0x5E1 + R, R, n, dtype)
    want = expected(cpu, dtype)
    ins = device_inputs(cpu)
    bufs, outs = (None, ins) if inplace else guarded_outputs(R, n, dtype)
    with ar.Handle(R, n, dtype) as h:
        ar.ar_allreduce(h.h, ins, outs, algo, proto)
        st = ar.ar_status(h.h)
        assert st == ar.AR_OK, ar.ar_strerror(st)
    for r in range(R):
        assert_bits_equal(outs[r], want, dtype, "special R=%d n=%d %s rank %d" % (R, n, dtype, r))
    if bufs is not None:
        check_guards(bufs, n, dtype)


@pytest.mark.parametrize("path", ALL_PATHS, ids=PATH_IDS)
@pytest.mark.parametrize("dtype", DTYPES)
@pytest.mark.parametrize("R", [2, 5, 16])
def test_special_values_every_path(path, dtype, R):
    _allreduce_case(R, 4099, dtype, *path)


@pytest.mark.parametrize("path", ALL_PATHS, ids=PATH_IDS)
@pytest.mark.parametrize("dtype", DTYPES)
def test_special_values_many_tiles_in_place(path, dtype):
    """Large enough for the one-shot ring and many TMA tiles, in place."""
    _allreduce_case(5, (1 << 20) + 3, dtype, *path, inplace=True)


@pytest.mark.parametrize("algo", ["one_shot", "two_shot"])
@pytest.mark.parametrize("dtype", DTYPES)
def test_special_values_plans(algo, dtype):
    need_gpu()
    R, n = 5, 4099
    cpu = wl.special_inputs(0x5E1 + R, R, n, dtype)
    want = expected(cpu, dtype)
    ins = device_inputs(cpu)
    outs = [torch.empty(n, dtype=wl.TORCH_DTYPE[dtype], device="cuda") for _ in range(R)]
    with ar.Handle(R, n, dtype) as h:
        p = ar.ar_plan_builtin(h.h, algo, 0, 0)
        ar.ar_plan_execute(p, ins, outs)
        st = ar.ar_status(h.h)
        ar.ar_plan_destroy(p)
        assert st == ar.AR_OK, ar.ar_strerror(st)
    for r in range(R):
        assert_bits_equal(outs[r], want, dtype, "plan %s rank %d" % (algo, r))


@pytest.mark.parametrize("dtype", DTYPES)
@pytest.mark.parametrize("H", [72, 70])
def test_special_values_combine(dtype, H):
    """Products of special weights and special values (subnormal products
    included), folded and rounded once; H = 70 takes the element path."""
    need_gpu()
    K, T = 4, 7
    cpu = wl.special_inputs(0x5E2, K, T * H, dtype)
    w = wl.special_weights(0x5E3, T, K)
    want = oracle.combine([wl.bits(t) for t in cpu], w, T, H, wl.DTYPE_CODE[dtype])
    ys = device_inputs(cpu)
    out = torch.empty(T * H, dtype=wl.TORCH_DTYPE[dtype], device="cuda")
    with ar.Handle(K, T * H, dtype) as h:
        ar.ar_combine(h.h, ys, torch.from_numpy(np.ascontiguousarray(w)).cuda(), out, T, H)
        st = ar.ar_status(h.h)
        assert st == ar.AR_OK, ar.ar_strerror(st)
    assert_bits_equal(out, want, dtype, "combine special H=%d" % H)
