"""The weighted per-token combine on the GPU against the oracle, bit for bit."""
import numpy as np
import pytest
import torch

import all_reduce_reduction_gb300 as ar
import oracle
from all_reduce_reduction_gb300 import workload as wl
from gpu_helpers import assert_bits_equal, check_guards, device_inputs, guarded_outputs, need_gpu

pytestmark = pytest.mark.gpu


def _run(K, T, H, dtype, offset=0, out_is_source=None, dist="loguniform", seed=90):
    need_gpu()
    cpu = wl.make_inputs(seed, K, T * H, dtype, dist)
    w = wl.gate_weights(seed, T, K)
    want = oracle.combine([wl.bits(t) for t in cpu], w, T, H, wl.DTYPE_CODE[dtype])
    ys = device_inputs(cpu, offset)
    dw = torch.from_numpy(w).cuda()
    if out_is_source is None:
        bufs, outs = guarded_outputs(1, T * H, dtype, offset)
        out = outs[0]
    else:
        bufs, out = None, ys[out_is_source]
    with ar.Handle(K, T * H, dtype) as h:
        ar.ar_combine(h.h, ys, dw, out, T, H)
        assert ar.ar_status(h.h) == ar.AR_OK
    assert_bits_equal(out, want, dtype, "K=%d T=%d H=%d" % (K, T, H))
    if bufs is not None:
        check_guards(bufs, T * H, dtype, offset)


@pytest.mark.parametrize("dtype", ["bf16", "fp16", "fp32"])
@pytest.mark.parametrize("K", [1, 2, 3, 8, 32])
@pytest.mark.parametrize("T,H", [(1, 8), (3, 7), (16, 8192), (5, 1000), (128, 264)])
def test_combine_matrix(dtype, K, T, H):
    _run(K, T, H, dtype)


@pytest.mark.parametrize("dtype", ["bf16", "fp32"])
@pytest.mark.parametrize("offset", [1, 2])
def test_combine_misaligned(dtype, offset):
    _run(4, 9, 64, dtype, offset=offset)


def test_combine_in_place_into_a_source():
    _run(8, 16, 4096, "bf16", out_is_source=3)


@pytest.mark.parametrize("w", [w for w in wl.COMBINE], ids=lambda w: w.name)
def test_combine_workloads_full_size(w):
    need_gpu()
    cpu = w.inputs(threads=8)
    wts = w.weights()
    want = oracle.combine([wl.bits(t) for t in cpu], wts, w.T, w.H, wl.DTYPE_CODE[w.dtype])
    ys = [t.cuda() for t in cpu]
    out = torch.empty(w.T * w.H, dtype=wl.TORCH_DTYPE[w.dtype], device="cuda")
    with ar.Handle(w.K, w.T * w.H, w.dtype) as h:
        s = torch.cuda.Stream()
        dw = torch.from_numpy(wts).cuda()
        with torch.cuda.stream(s):
            ar.ar_combine(h.h, ys, dw, out, w.T, w.H, stream=s)
        s.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=s):
            for _ in range(10):
                ar.ar_combine(h.h, ys, dw, out, w.T, w.H, stream=s)
        out.fill_(float("nan"))
        g.replay()
        torch.cuda.synchronize()
        assert ar.ar_status(h.h) == ar.AR_OK
    assert_bits_equal(out, want, w.dtype, w.name)


def test_combine_rejections():
    need_gpu()
    K, T, H = 2, 4, 16
    ys = [torch.zeros(T * H, dtype=torch.bfloat16, device="cuda") for _ in range(K)]
    w = torch.ones(T * K, dtype=torch.float32, device="cuda")
    big = torch.zeros(2 * T * H, dtype=torch.bfloat16, device="cuda")
    with ar.Handle(K, T * H, "bf16") as h:
        with pytest.raises(ar.ArError):
            ar.ar_combine(h.h, ys, w, ys[0][1:], T, H - 1)    # out partly overlaps a source
        with pytest.raises(ar.ArError):
            ar.ar_combine(h.h, ys, w, ys[0], T, H + 1)        # T*H beyond N
        with pytest.raises(ar.ArError):
            ar.ar_combine(h.h, [big[:T * H], big[T * H // 2: T * H // 2 + T * H]], w, big[3:], T, H)
