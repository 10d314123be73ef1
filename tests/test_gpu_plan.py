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
        # one-shot: R ranks reduce every chunk, no dependencies at all;
        # two-shot: every all-gather copy fuses into its shard's reduction,
        # which leaves R * K reductions with R destinations and no waits
        assert tasks == (R * R * K if algo == "one_shot" else R * K)
        assert waits == 0 and signals == 0
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


@pytest.mark.parametrize("seed", range(8))
def test_random_copy_heavy_programs(seed):
    """Mostly copies between outputs: long chains the compiler fuses into
    earlier tasks, and copies it must not fuse."""
    need_gpu()
    R, n, nch, dtype = 5, 30001, 5, ["bf16", "fp16", "fp32"][seed % 3]
    steps = random_steps(R, nch, 40, 1000 + seed, copy_weight=3)
    _run_program(steps, R, n, nch, dtype, G=2, seed=seed)


def _run_program(steps, R, n, nch, dtype, G, seed, want_tasks=None):
    cpu = wl.make_inputs(87, R, n, dtype, "uniform")
    start = [wl.bits(t) for t in wl.make_inputs(88, R, n, dtype, "uniform")]
    want_in = [wl.bits(t).copy() for t in cpu]
    want_out = oracle.plan_run(steps, want_in, [a.copy() for a in start],
                               wl.DTYPE_CODE[dtype], nch)
    ins = device_inputs(cpu)
    outs = [wl.from_bits(a, dtype).cuda() for a in start]
    with ar.Handle(R, n, dtype) as h:
        p = ar.ar_plan_compile(h.h, to_ops(steps, R), nch, G)
        tasks, _, _ = ar.ar_plan_stats(p)
        ar.ar_plan_execute(p, ins, outs)
        assert ar.ar_status(h.h) == ar.AR_OK
        ar.ar_plan_destroy(p)
    if want_tasks is not None:
        assert tasks == want_tasks
    for r in range(R):
        assert_bits_equal(outs[r], want_out[r], dtype, "case %s out %d" % (seed, r))
        assert_bits_equal(ins[r], want_in[r], dtype, "case %s in %d" % (seed, r))


def _red(rank, dst, srcs, nch):
    return dict(kind="reduce", rank=rank, dst=dst, srcs=srcs, cbeg=0, cend=nch)


def _cp(rank, dst, src, nch):
    return dict(kind="copy", rank=rank, dst=dst, srcs=[src], cbeg=0, cend=nch)


# Buffer ids with R = 4: in[b] = b, out[r] = 4 + r.  Every case runs on 3
# chunks, so a step is 3 tasks; `fused` is how many copy steps the compiler
# may fold into earlier tasks.
FUSION_CASES = {
    # out1 is read between the reduce and the copy into it: no fusion
    "read_between": ([_red(0, 4, [0, 1], 3), _cp(1, 6, 5, 3), _cp(2, 5, 4, 3)], 0),
    # out1 is written between the reduce and the copy into it: no fusion
    "write_between": ([_red(0, 4, [0, 1], 3), _cp(1, 5, 3, 3), _cp(2, 5, 4, 3)], 0),
    # the copy's destination is one of the reduce's sources: no fusion
    "dst_is_source": ([_red(0, 4, [5, 6], 3), _cp(1, 5, 4, 3)], 0),
    # a chain out0 -> out1 -> out2 -> out3: all three copies fold into the reduce
    "chain": ([_red(0, 4, [0, 1, 2, 3], 3), _cp(1, 5, 4, 3), _cp(2, 6, 5, 3),
               _cp(3, 7, 6, 3)], 3),
    # the source is rewritten before the copy: it folds into the later writer
    "rewritten_source": ([_red(0, 4, [0, 1], 3), _red(1, 4, [2, 3], 3), _cp(2, 5, 4, 3)], 1),
    # two copies into one destination: each folds into its own producer
    "two_producers": ([_red(0, 4, [0, 1], 3), _cp(1, 6, 4, 3), _red(2, 5, [2, 3], 3),
                       _cp(3, 6, 5, 3)], 2),
    # copy from an input (never written by the plan): nothing to fold into
    "from_input": ([_cp(0, 4, 1, 3), _red(1, 5, [4, 6], 3)], 0),
}


@pytest.mark.parametrize("case", sorted(FUSION_CASES))
def test_fusion_rules(case):
    need_gpu()
    steps, fused = FUSION_CASES[case]
    _run_program(steps, 4, 5003, 3, "bf16", G=2, seed=case, want_tasks=3 * (len(steps) - fused))


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
def test_builtin_plan_default_chunks(algo):
    """With chunks_per_rank 0 a large two-shot message (R >= 8) is cut into a
    whole number of chunks per CTA, each about 8 KiB of a rank buffer; the
    one-shot plan keeps one chunk per CTA.  Both stay the oracle's bit for
    bit (ragged tail included)."""
    need_gpu()
    R, n, dtype = 8, (8 << 20) + 3, "bf16"
    with ar.Handle(R, 1000, dtype) as h:          # one chunk per CTA there: gives the CTA count
        p = ar.ar_plan_builtin(h.h, algo)
        tasks, _, _ = ar.ar_plan_stats(p)
        ar.ar_plan_destroy(p)
    per_chunk = R if algo == "one_shot" else 1     # tasks per chunk after fusion
    G = tasks // (R * per_chunk)
    assert G * R * per_chunk == tasks and G >= 1
    cpu = wl.make_inputs(87, R, n, dtype, "normal")
    ins = device_inputs(cpu)
    outs = _outs(R, n, dtype)
    with ar.Handle(R, n, dtype) as h:
        p = ar.ar_plan_builtin(h.h, algo)
        tasks, _, _ = ar.ar_plan_stats(p)
        K = tasks // (R * per_chunk)
        assert K * R * per_chunk == tasks
        if algo == "one_shot":
            assert K == G, (K, G)
        else:
            assert K % G == 0 and G < K <= 16 * G, (K, G)
            chunk_bytes = -(-n // (R * K)) * wl.ELEM_SIZE[dtype]
            assert 4096 <= chunk_bytes <= 12288, chunk_bytes
        ar.ar_plan_execute(p, ins, outs)
        assert ar.ar_status(h.h) == ar.AR_OK
        ar.ar_plan_destroy(p)
    want = expected(cpu, dtype)
    for r in range(R):
        assert_bits_equal(outs[r], want, dtype, "rank %d" % r)


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


@pytest.mark.parametrize("R", [16, 32])
def test_builtin_two_shot_plan_two_ctas_per_sm_from_r16(R):
    """From R = 16 the built-in two-shot plan runs two CTAs per SM by
    default (the one-shot plan and smaller R fill the resident capacity);
    the results stay the oracle's bit for bit."""
    need_gpu()
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    with ar.Handle(R, 1000, "bf16") as h:              # one chunk per CTA: gives the CTA count
        p = ar.ar_plan_builtin(h.h, "two_shot")
        tasks, _, _ = ar.ar_plan_stats(p)
        ar.ar_plan_destroy(p)
        assert tasks == R * (2 * sms // R)
        p = ar.ar_plan_builtin(h.h, "one_shot")
        tasks, _, _ = ar.ar_plan_stats(p)
        ar.ar_plan_destroy(p)
        assert tasks // (R * R) > 2 * sms // R          # more CTAs: the resident capacity
    n = (1 << 20) + 5
    cpu = wl.make_inputs(88, R, n, "bf16", "normal")
    ins = device_inputs(cpu)
    outs = _outs(R, n, "bf16")
    with ar.Handle(R, n, "bf16") as h:
        p = ar.ar_plan_builtin(h.h, "two_shot")
        ar.ar_plan_execute(p, ins, outs)
        assert ar.ar_status(h.h) == ar.AR_OK
        ar.ar_plan_destroy(p)
    want = expected(cpu, "bf16")
    for r in range(R):
        assert_bits_equal(outs[r], want, "bf16", "rank %d" % r)
