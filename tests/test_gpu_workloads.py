"""GPU parity at the workloads' full sizes, element by element against the
oracle, in the launch configuration the benchmark times (CUDA graphs of 10
calls for the small messages, single calls for the large ones)."""
import ctypes

import numpy as np
import pytest
import torch

import all_reduce_reduction_gb300 as ar
import oracle
from all_reduce_reduction_gb300 import workload as wl
from gpu_helpers import ALL_PATHS, PATH_IDS, assert_bits_equal, need_gpu

pytestmark = pytest.mark.gpu


def oracle_single_output(cpu_inputs, dtype):
    """The oracle's result, written once (every rank's output is the same
    array, which the oracle fills R times with the same values)."""
    ins = [wl.bits(t) for t in cpu_inputs]
    out = np.empty_like(ins[0])
    lib = oracle.load()
    arr_in = (ctypes.c_void_p * len(ins))(*[a.ctypes.data for a in ins])
    arr_out = (ctypes.c_void_p * len(ins))(*([out.ctypes.data] * len(ins)))
    assert lib.oracle_allreduce(len(ins), ins[0].size, wl.DTYPE_CODE[dtype], arr_in, arr_out) == 0
    return out


def run_graph(w, algo, proto, cpu, calls=10, warm=2, transport=ar.AR_LL_AUTO,
              staging=ar.AR_HB_STAGING_AUTO):
    ins = [t.cuda() for t in cpu]
    outs = [torch.full_like(t, float("nan")) for t in ins]
    s = torch.cuda.Stream()
    with ar.Handle(w.R, w.n, w.dtype) as h:
        ar.ar_set_ll_transport(h.h, transport)
        ar.ar_set_hb_staging(h.h, staging)
        if algo == ar.AR_ALGO_AUTO or proto == ar.AR_PROTO_AUTO:
            ar.ar_tune(h.h, s)                           # as the decode benchmark does
        with torch.cuda.stream(s):
            ar.ar_allreduce(h.h, ins, outs, algo, proto, stream=s)
        s.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=s):
            for _ in range(calls):
                ar.ar_allreduce(h.h, ins, outs, algo, proto, stream=s)
        for _ in range(warm + 1):
            g.replay()
        torch.cuda.synchronize()
        assert ar.ar_status(h.h) == ar.AR_OK
    return outs


# every path with the default LL transport, and the LL paths again with the
# HBM-slot transport forced (the transport setting applies to LL only)
SWEEP_CASES = ([(p, ar.AR_LL_AUTO, i + "-auto") for p, i in zip(ALL_PATHS, PATH_IDS)]
               + [(p, ar.AR_LL_GLOBAL, i + "-global") for p, i in zip(ALL_PATHS, PATH_IDS)
                  if p[1] == ar.AR_LL])


@pytest.mark.parametrize("path,transport", [c[:2] for c in SWEEP_CASES],
                         ids=[c[2] for c in SWEEP_CASES])
def test_ll_sweep_sizes(path, transport):
    """R=8 bf16, N = 2^9..2^18, uniform [-1, 1), 10 calls per graph."""
    need_gpu()
    for w in wl.LL_SWEEP:
        cpu = w.inputs()
        want = oracle_single_output(cpu, w.dtype)
        outs = run_graph(w, *path, cpu, transport=transport)
        for r in range(w.R):
            assert_bits_equal(outs[r], want, w.dtype, "%s rank %d" % (w.name, r))


@pytest.mark.parametrize("path", ALL_PATHS + [(ar.AR_ALGO_AUTO, ar.AR_PROTO_AUTO)],
                         ids=PATH_IDS + ["auto_tuned"])
def test_decode_shapes(path):
    """R=8 bf16 [B, 8192], B in 1, 8, 32, 128, 256, N(0, 1)."""
    need_gpu()
    for w in wl.DECODE:
        cpu = w.inputs(threads=8)
        want = oracle_single_output(cpu, w.dtype)
        outs = run_graph(w, *path, cpu)
        for r in range(w.R):
            assert_bits_equal(outs[r], want, w.dtype, "%s rank %d" % (w.name, r))


@pytest.fixture(scope="module")
def prefill():
    need_gpu()
    w = wl.PREFILL
    cpu = w.inputs(threads=16)
    return w, cpu, oracle_single_output(cpu, w.dtype)


@pytest.mark.parametrize("algo,staging", [(ar.AR_TWO_SHOT, ar.AR_HB_STAGING_TMA),
                                          (ar.AR_TWO_SHOT, ar.AR_HB_STAGING_DIRECT),
                                          (ar.AR_ONE_SHOT, ar.AR_HB_STAGING_AUTO)],
                         ids=["two_shot_tma", "two_shot_direct", "one_shot"])
def test_prefill_full_size(prefill, algo, staging):
    """R=16 bf16 [8192, 8192] per rank (128 MiB), HB (two-shot with either
    staging)."""
    w, cpu, want = prefill
    outs = run_graph(w, algo, ar.AR_HB, cpu, calls=1, warm=1, staging=staging)
    for r in range(w.R):
        assert_bits_equal(outs[r], want, w.dtype, "prefill rank %d" % r)
    del outs
    torch.cuda.empty_cache()


@pytest.mark.parametrize("w", wl.EDGE, ids=lambda w: "R%d_%s" % (w.R, w.dtype))
def test_edge_full_size(w):
    """R in {4, 32}, bf16/fp16/fp32, N = 4097*4096+3, log-uniform values of
    both signs: every schedule; LL where the message is within its cap."""
    need_gpu()
    cpu = w.inputs(threads=16)
    want = oracle_single_output(cpu, w.dtype)
    ll_ok = w.bytes_per_rank <= ar.AR_LL_MAX_BYTES
    for algo, proto in ALL_PATHS:
        if proto == ar.AR_LL and not ll_ok:
            with ar.Handle(w.R, w.n, w.dtype) as h:
                assert ar.ar_get_info(h.h)["ll_capable"] == 0
            continue
        stagings = [ar.AR_HB_STAGING_AUTO]
        if algo == ar.AR_TWO_SHOT and proto == ar.AR_HB:
            stagings = [ar.AR_HB_STAGING_TMA, ar.AR_HB_STAGING_DIRECT]
        for staging in stagings:
            outs = run_graph(w, algo, proto, cpu, calls=1, warm=1, staging=staging)
            for r in range(w.R):
                assert_bits_equal(outs[r], want, w.dtype, "%s algo %d proto %d staging %d rank %d"
                                  % (w.name, algo, proto, staging, r))
            del outs
            torch.cuda.empty_cache()
