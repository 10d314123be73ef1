"""ar_allreduce_host: the all-reduce with its buffers in page-locked host
memory, which the kernels read and write in place through the CPU-GPU link.

Every case compares every output element with the CPU oracle, bit for bit,
with canaries around every output: each schedule and protocol, AUTO, ragged
sizes, buffers off 16- and 8-byte alignment, in place, inputs on the host
with outputs on the device, the handle forced to the TMA staging or the
cluster LL transport (neither runs on host memory; the call must still give
the oracle's bits), a captured CUDA graph replayed on new host inputs, and
the refusals (pageable memory)."""
import numpy as np
import pytest
import torch

import all_reduce_reduction_gb300 as ar
from all_reduce_reduction_gb300 import workload as wl
from gpu_helpers import (GUARD, UINT_T, assert_bits_equal, canary_value, check_guards, expected,
                         need_gpu)

pytestmark = pytest.mark.gpu

PATHS = [(ar.AR_ONE_SHOT, ar.AR_LL), (ar.AR_TWO_SHOT, ar.AR_LL), (ar.AR_ONE_SHOT, ar.AR_HB),
         (ar.AR_TWO_SHOT, ar.AR_HB), (ar.AR_ALGO_AUTO, ar.AR_PROTO_AUTO),
         (ar.AR_ALGO_AUTO, ar.AR_LL), (ar.AR_ONE_SHOT, ar.AR_PROTO_AUTO)]
PATH_IDS = ["one_shot_ll", "two_shot_ll", "one_shot_hb", "two_shot_hb", "auto", "auto_ll",
            "one_shot_auto"]


def pinned_inputs(cpu, offset: int = 0):
    """Page-locked host copies of the inputs, `offset` elements into their
    buffers."""
    outs = []
    for t in cpu:
        b = torch.empty(offset + t.numel() + 8, dtype=t.dtype).pin_memory()
        v = b[offset: offset + t.numel()]
        v.copy_(t)
        outs.append(v)
    return outs


def pinned_outputs(R: int, n: int, dtype: str, offset: int = 0):
    """Page-locked host output views with canaries before and after."""
    bufs, views = [], []
    for _ in range(R):
        b = torch.empty(GUARD + offset + n + GUARD, dtype=wl.TORCH_DTYPE[dtype]).pin_memory()
        b.view(UINT_T[dtype]).fill_(canary_value(dtype))
        bufs.append(b)
        views.append(b[GUARD + offset: GUARD + offset + n])
    return bufs, views


def run_host(h, ins, outs, n, algo, proto):
    ar.ar_allreduce_host(h.h, ins, outs, n, algo, proto)
    torch.cuda.synchronize()
    assert ar.ar_status(h.h) == ar.AR_OK


@pytest.mark.parametrize("path", PATHS, ids=PATH_IDS)
@pytest.mark.parametrize("R,n,dtype", [(8, 1 << 18, "bf16"), (8, 1001, "bf16"), (2, 65539, "fp32"),
                                       (5, 4097, "fp16"), (32, 777, "bf16"), (1, 300, "fp32"),
                                       (4, (1 << 19) + 3, "bf16"), (16, (1 << 20) + 5, "bf16")],
                         ids=["r8_n262144_bf16", "r8_n1001_bf16", "r2_n65539_fp32",
                              "r5_n4097_fp16", "r32_n777_bf16", "r1_n300_fp32",
                              "r4_n524291_bf16", "r16_n1048581_bf16"])
@pytest.mark.parametrize("offset", [0, 1, 4], ids=["aligned", "off2or4", "off8or16"])
def test_host_buffers_match_oracle(path, R, n, dtype, offset):
    need_gpu()
    cpu = wl.make_inputs(80, R, n, dtype, "loguniform")
    want = expected(cpu, dtype)
    ins = pinned_inputs(cpu, offset)
    bufs, outs = pinned_outputs(R, n, dtype, offset)
    with ar.Handle(R, n, dtype) as h:
        run_host(h, ins, outs, n, *path)
    for r in range(R):
        assert_bits_equal(outs[r], want, dtype, "rank %d" % r)
    check_guards(bufs, n, dtype, offset)


@pytest.mark.parametrize("path", PATHS[:4], ids=PATH_IDS[:4])
def test_host_buffers_in_place(path):
    need_gpu()
    R, n, dtype = 8, 20001, "bf16"
    cpu = wl.make_inputs(81, R, n, dtype, "normal")
    want = expected(cpu, dtype)
    bufs = pinned_inputs(cpu)
    with ar.Handle(R, n, dtype) as h:
        run_host(h, bufs, bufs, n, *path)
    for r in range(R):
        assert_bits_equal(bufs[r], want, dtype, "in place, rank %d" % r)


@pytest.mark.parametrize("path", PATHS[:4], ids=PATH_IDS[:4])
def test_host_inputs_device_outputs(path):
    """Inputs in host memory, outputs in device memory (and the reverse)."""
    need_gpu()
    R, n, dtype = 4, 30000, "fp32"
    cpu = wl.make_inputs(82, R, n, dtype, "uniform")
    want = expected(cpu, dtype)
    with ar.Handle(R, n, dtype) as h:
        ins = pinned_inputs(cpu)
        outs = [torch.full((n,), float("nan"), device="cuda") for _ in range(R)]
        run_host(h, ins, outs, n, *path)
        for r in range(R):
            assert_bits_equal(outs[r], want, dtype, "device output, rank %d" % r)
        ins = [t.cuda() for t in cpu]
        bufs, outs = pinned_outputs(R, n, dtype)
        run_host(h, ins, outs, n, *path)
        for r in range(R):
            assert_bits_equal(outs[r], want, dtype, "host output, rank %d" % r)
        check_guards(bufs, n, dtype)


def test_host_buffers_with_tma_staging_and_cluster_transport_forced():
    """The handle's TMA staging and cluster LL transport do not run on host
    memory: the call takes the direct staging and the HBM packet slots and
    still gives the oracle's bits; with device buffers the same handle runs
    its settings as before."""
    need_gpu()
    R, n, dtype = 8, 1 << 17, "bf16"
    cpu = wl.make_inputs(83, R, n, dtype, "uniform")
    want = expected(cpu, dtype)
    ins = pinned_inputs(cpu)
    with ar.Handle(R, n, dtype) as h:
        ar.ar_set_hb_staging(h.h, ar.AR_HB_STAGING_TMA)
        ar.ar_set_ll_transport(h.h, ar.AR_LL_CLUSTER)
        for algo, proto in [(ar.AR_TWO_SHOT, ar.AR_HB), (ar.AR_ONE_SHOT, ar.AR_LL)]:
            bufs, outs = pinned_outputs(R, n, dtype)
            run_host(h, ins, outs, n, algo, proto)
            for r in range(R):
                assert_bits_equal(outs[r], want, dtype, "algo %d proto %d rank %d" % (algo, proto, r))
            check_guards(bufs, n, dtype)
            dins = [t.cuda() for t in cpu]
            douts = [torch.empty_like(t) for t in dins]
            run_host(h, dins, douts, n, algo, proto)
            for r in range(R):
                assert_bits_equal(douts[r], want, dtype, "device buffers rank %d" % r)


@pytest.mark.parametrize("path", [(ar.AR_ONE_SHOT, ar.AR_LL), (ar.AR_TWO_SHOT, ar.AR_HB)],
                         ids=["one_shot_ll", "two_shot_hb"])
def test_host_call_in_a_cuda_graph(path):
    """One captured call, replayed three times on new host inputs written
    between replays: every replay reads the host memory afresh."""
    need_gpu()
    R, n, dtype = 8, 4096, "bf16"
    ins = pinned_inputs(wl.make_inputs(84, R, n, dtype, "uniform"))
    bufs, outs = pinned_outputs(R, n, dtype)
    s = torch.cuda.Stream()
    with ar.Handle(R, n, dtype) as h:
        with torch.cuda.stream(s):
            ar.ar_allreduce_host(h.h, ins, outs, n, *path, stream=s)
        s.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=s):
            ar.ar_allreduce_host(h.h, ins, outs, n, *path, stream=s)
        for k in range(3):
            cpu = wl.make_inputs(85 + k, R, n, dtype, "normal")
            for t, c in zip(ins, cpu):
                t.copy_(c)
            g.replay()
            torch.cuda.synchronize()
            assert ar.ar_status(h.h) == ar.AR_OK
            want = expected(cpu, dtype)
            for r in range(R):
                assert_bits_equal(outs[r], want, dtype, "replay %d rank %d" % (k, r))
        check_guards(bufs, n, dtype)


def test_host_call_refusals():
    need_gpu()
    R, n = 2, 64
    pinned = [torch.zeros(n, dtype=torch.bfloat16).pin_memory() for _ in range(R)]
    pageable = [torch.zeros(n, dtype=torch.bfloat16) for _ in range(R)]
    with ar.Handle(R, n, "bf16") as h:
        for ins, outs in [(pageable, pinned), (pinned, pageable)]:
            with pytest.raises(ar.ArError) as e:
                ar.ar_allreduce_host(h.h, ins, outs, n)
            assert e.value.code == ar.AR_ERR_INVALID
        with pytest.raises(ar.ArError) as e:
            ar.ar_allreduce_host(h.h, pinned, pinned[:1], n)       # too few outputs
        assert e.value.code == ar.AR_ERR_INVALID
        with pytest.raises(ar.ArError) as e:
            ar.ar_allreduce_host(h.h, pinned, [t.clone().pin_memory() for t in pinned], n + 1)
        assert e.value.code == ar.AR_ERR_INVALID
        ar.ar_allreduce_host(h.h, pinned, [t.clone().pin_memory() for t in pinned], n)
        torch.cuda.synchronize()
        assert ar.ar_status(h.h) == ar.AR_OK
    assert np.array_equal(wl.bits(pinned[0]), np.zeros(n, dtype=np.uint16))
