"""Compiled plans on the GPU against the oracle: the built-in one-shot and
two-shot all-reduce plans, and random copy/reduce programs whose cross-CTA
dependencies the compiler must synchronise."""
import numpy as np
import pytest
import torch

import all_reduce_reduction_gb300 as ar
import oracle
from all_reduce_reduction_gb300 import workload as wl
from gpu_helpers import assert_bits_equal, device_inputs, expected, need_gpu
from plan_helpers import random_steps, to_ops

pytestmark = pytest.mark.gpu


def _outs(R, n, dtype):
    return [torch.full((n,), float("nan"), dtype=wl.TORCH_DTYPE[dtype], device="cuda")
            for _ in range(R)]


@pytest.mark.parametrize("algo", ["one_shot", "two_shot"])
@pytest.mark.parametrize("dtype", ["bf16", "fp16", "fp32"])
@pytest.mark.parametrize("R,n,K,G", [(2, 1001, 2, 1), (3, 4097, 1, 2), (8, 1 << 18, 4, 4),
                                     (8, (1 << 20) + 5, 8, 8), (16, 70001, 2, 2), (32, 9999, 1, 1)])
def test_builtin_plans(algo, dtype, R, n, K, G):
    need_gpu()
    cpu = wl.make_inputs(81, R, n, dtype, "loguniform")
    ins = device_inputs(cpu)
    outs = _outs(R, n, dtype)
    with ar.Handle(R, n, dtype) as h:
        p = ar.ar_plan_builtin(h.h, algo, K, G)
        tasks, waits, signals = ar.ar_plan_stats(p)
        if algo == "one_shot":
            assert waits == 0 and signals == 0          # no dependencies at all
        else:
            assert waits > 0 and signals > 0
        for _ in range(2):                               # two runs: run index advances
            ar.ar_plan_execute(p, ins, outs)
        assert ar.ar_status(h.h) == ar.AR_OK
        ar.ar_plan_destroy(p)
    want = expected(cpu, dtype)
    for r in range(R):
        assert_bits_equal(outs[r], want, dtype, "rank %d" % r)


@pytest.mark.parametrize("seed", range(12))
@pytest.mark.parametrize("G", [1, 3])
def test_random_programs(seed, G):
    need_gpu()
    R, n, nch, dtype = 6, 50001, 7, ["bf16", "fp16", "fp32"][seed % 3]
    steps = random_steps(R, nch, 24, seed)
    cpu = wl.make_inputs(82, R, n, dtype, "uniform")
    start = [wl.bits(t) for t in wl.make_inputs(83, R, n, dtype, "uniform")]
    want_in = [wl.bits(t).copy() for t in cpu]
    want_out = oracle.plan_run(steps, want_in, [a.copy() for a in start],
                               wl.DTYPE_CODE[dtype], nch)
    ins = device_inputs(cpu)
    outs = [wl.from_bits(a, dtype).cuda() for a in start]
    with ar.Handle(R, n, dtype) as h:
        p = ar.ar_plan_compile(h.h, to_ops(steps, R), nch, G)
        ar.ar_plan_execute(p, ins, outs)
        assert ar.ar_status(h.h) == ar.AR_OK
        ar.ar_plan_destroy(p)
    for r in range(R):
        assert_bits_equal(outs[r], want_out[r], dtype, "seed %d out %d" % (seed, r))
        assert_bits_equal(ins[r], want_in[r], dtype, "seed %d in %d" % (seed, r))


def test_plan_in_a_captured_graph_with_new_inputs():
    need_gpu()
    R, n, dtype = 8, 65536 + 3, "bf16"
    ins = [torch.empty(n, dtype=torch.bfloat16, device="cuda") for _ in range(R)]
    outs = _outs(R, n, dtype)
    h = ar.Handle(R, n, dtype)
    p = ar.ar_plan_builtin(h.h, "two_shot", 4, 2)
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        for t in ins:
            t.zero_()
        ar.ar_plan_execute(p, ins, outs, stream=s)
    s.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        for _ in range(5):
            ar.ar_plan_execute(p, ins, outs, stream=s)
    for rep in range(3):
        cpu = wl.make_inputs(84 + rep, R, n, dtype, "uniform")
        for t, c in zip(ins, cpu):
            t.copy_(c)
        g.replay()
        torch.cuda.synchronize()
        assert ar.ar_status(h.h) == ar.AR_OK
        want = expected(cpu, dtype)
        for r in range(R):
            assert_bits_equal(outs[r], want, dtype, "replay %d rank %d" % (rep, r))
    ar.ar_plan_destroy(p)
    h.close()


def test_plan_misaligned_buffers_and_rejections():
    need_gpu()
    R, n, dtype = 4, 3001, "fp16"
    cpu = wl.make_inputs(85, R, n, dtype, "normal")
    ins = device_inputs(cpu, offset=1)
    outs = [torch.empty(n + 1, dtype=torch.float16, device="cuda")[1:] for _ in range(R)]
    with ar.Handle(R, n, dtype) as h:
        p = ar.ar_plan_builtin(h.h, "two_shot", 3, 2)
        ar.ar_plan_execute(p, ins, outs)
        assert ar.ar_status(h.h) == ar.AR_OK
        want = expected(cpu, dtype)
        for r in range(R):
            assert_bits_equal(outs[r], want, dtype, "rank %d" % r)
        with pytest.raises(ar.ArError):                  # in place is not allowed for plans
            ar.ar_plan_execute(p, ins, ins)
        bad = ar.make_op(ar.AR_OP_COPY, 0, (ar.AR_BUF_OUT, 0), [(ar.AR_BUF_IN, 1)], 0, 9)
        with pytest.raises(ar.ArError):                  # chunk range beyond nchunks
            ar.ar_plan_compile(h.h, [bad], 4, 1)
        huge = (1 << 20) + 1
        big = ar.make_op(ar.AR_OP_COPY, 0, (ar.AR_BUF_OUT, 0), [(ar.AR_BUF_IN, 1)], 0, huge)
        with pytest.raises(ar.ArError) as e:             # more tasks than a plan may hold
            ar.ar_plan_compile(h.h, [big], huge, 1)
        assert e.value.code == ar.AR_ERR_UNSUPPORTED
        with pytest.raises(ar.ArError) as e:             # R * chunks_per_rank beyond it too
            ar.ar_plan_builtin(h.h, "one_shot", 1 << 30, 2)
        assert e.value.code == ar.AR_ERR_UNSUPPORTED
        ar.ar_plan_destroy(p)


@pytest.mark.parametrize("algo", ["one_shot", "two_shot"])
def test_builtin_plan_fills_the_gpu_by_default(algo):
    need_gpu()
    R, n, dtype = 8, (1 << 19) + 3, "bf16"
    cpu = wl.make_inputs(86, R, n, dtype, "uniform")
    ins = device_inputs(cpu)
    outs = _outs(R, n, dtype)
    with ar.Handle(R, n, dtype) as h:
        p = ar.ar_plan_builtin(h.h, algo)                # chunks and CTAs chosen by the library
        tasks, _, _ = ar.ar_plan_stats(p)
        assert tasks >= R * 8                            # at least a few CTAs' worth per rank
        ar.ar_plan_execute(p, ins, outs)
        assert ar.ar_status(h.h) == ar.AR_OK
        ar.ar_plan_destroy(p)
    want = expected(cpu, dtype)
    for r in range(R):
        assert_bits_equal(outs[r], want, dtype, "rank %d" % r)
