"""Pins for the oracle's plan interpreter (sequential execution of steps)."""
import numpy as np
import pytest

import oracle
from all_reduce_reduction_gb300 import workload as wl
from _util import DT_CODE, as_uint, decode64
from plan_helpers import builtin_steps

DTYPES = ["bf16", "fp16", "fp32"]


def _ins(R, n, dtype, config=80, dist="loguniform"):
    return [wl.bits(t) for t in wl.make_inputs(config, R, n, dtype, dist)]


def _sentinel_outs(R, n, dtype):
    v = {"bf16": 0x7FC3, "fp16": 0x7E03, "fp32": 0x7FC00003}[dtype]
    u = np.uint32 if dtype == "fp32" else np.uint16
    return [np.full(n, v, dtype=u).view(oracle.STORAGE[DT_CODE[dtype]]) for _ in range(R)]


@pytest.mark.parametrize("dtype", DTYPES)
@pytest.mark.parametrize("algo", ["one_shot", "two_shot"])
@pytest.mark.parametrize("R,n,K", [(1, 5, 1), (2, 1001, 3), (5, 4097, 2), (8, 100, 4), (16, 7, 1)])
def test_builtin_plans_are_the_allreduce(dtype, algo, R, n, K):
    ins = _ins(R, n, dtype)
    want = oracle.allreduce(ins, DT_CODE[dtype])
    outs = oracle.plan_run(builtin_steps(R, algo, K), [a.copy() for a in ins],
                           _sentinel_outs(R, n, dtype), DT_CODE[dtype], R * K)
    for r in range(R):
        assert np.array_equal(as_uint(outs[r], dtype), as_uint(want[r], dtype))


@pytest.mark.parametrize("dtype", DTYPES)
def test_copy_only_plan_moves_chunks(dtype):
    """A rotation out[r] = in[(r + 1) % R] on chunks 1..3 of 5: a plain copy
    of those element ranges, the rest untouched."""
    R, n, nch = 4, 1003, 5
    ins = _ins(R, n, dtype)
    per_vec = 16 // wl.ELEM_SIZE[dtype]
    C = -(-n // nch)
    C = -(-C // per_vec) * per_vec
    steps = [dict(kind="copy", rank=r, dst=R + r, srcs=[(r + 1) % R], cbeg=1, cend=4)
             for r in range(R)]
    start = _sentinel_outs(R, n, dtype)
    outs = oracle.plan_run(steps, ins, [a.copy() for a in start], DT_CODE[dtype], nch)
    lo, hi = C, min(4 * C, n)
    for r in range(R):
        want = as_uint(start[r], dtype).copy()
        want[lo:hi] = as_uint(ins[(r + 1) % R], dtype)[lo:hi]
        assert np.array_equal(as_uint(outs[r], dtype), want)


@pytest.mark.parametrize("dtype", DTYPES)
def test_single_source_reduce_is_a_copy(dtype):
    R, n = 3, 777
    ins = _ins(R, n, dtype)
    steps = [dict(kind="reduce", rank=0, dst=R + 2, srcs=[1], cbeg=0, cend=2)]
    outs = oracle.plan_run(steps, ins, _sentinel_outs(R, n, dtype), DT_CODE[dtype], 2)
    assert np.array_equal(as_uint(outs[2], dtype), as_uint(ins[1], dtype))


@pytest.mark.parametrize("dtype", DTYPES)
def test_steps_run_in_program_order(dtype):
    """out0 = sum(in); out1 = copy(out0); out2 = out0 + out1 = 2 * out0
    (doubling is exact), then out0 is overwritten by in[2]: later steps see
    earlier steps' results and nothing else."""
    R, n = 3, 2049
    ins = _ins(R, n, dtype, dist="uniform")
    steps = [dict(kind="reduce", rank=0, dst=R + 0, srcs=[0, 1, 2], cbeg=0, cend=4),
             dict(kind="copy", rank=1, dst=R + 1, srcs=[R + 0], cbeg=0, cend=4),
             dict(kind="reduce", rank=2, dst=R + 2, srcs=[R + 0, R + 1], cbeg=0, cend=4),
             dict(kind="copy", rank=1, dst=R + 0, srcs=[2], cbeg=0, cend=4)]
    outs = oracle.plan_run(steps, ins, _sentinel_outs(R, n, dtype), DT_CODE[dtype], 4)
    s = oracle.allreduce(ins, DT_CODE[dtype])[0]
    assert np.array_equal(as_uint(outs[1], dtype), as_uint(s, dtype))
    assert np.array_equal(decode64(outs[2], dtype), 2.0 * decode64(s, dtype))
    assert np.array_equal(as_uint(outs[0], dtype), as_uint(ins[2], dtype))


def test_bad_plan_rejected():
    ins = _ins(2, 10, "bf16")
    with pytest.raises(ValueError):
        oracle.plan_run([dict(kind="copy", rank=0, dst=9, srcs=[0], cbeg=0, cend=1)],
                        ins, _sentinel_outs(2, 10, "bf16"), DT_CODE["bf16"], 1)
    with pytest.raises(ValueError):
        oracle.plan_run([dict(kind="copy", rank=0, dst=2, srcs=[0, 1], cbeg=0, cend=1)],
                        ins, _sentinel_outs(2, 10, "bf16"), DT_CODE["bf16"], 1)


def _python_plan(steps, ins, outs, dtype, nchunks):
    """The plain meaning of a plan, restated with numpy and torch: steps one
    after another; chunk c is elements [c*C, min((c+1)*C, n)) with
    C = ceil(n / nchunks) rounded up to a whole 16-byte vector; a copy moves
    bits; a reduce is a binary32 left fold of its sources in the listed order,
    narrowed once by torch's cast."""
    import torch
    R, n = len(ins), ins[0].size
    per_vec = 16 // {"bf16": 2, "fp16": 2, "fp32": 4}[dtype]
    C = -(-(-(-n // nchunks)) // per_vec) * per_vec
    bufs = [a.copy() for a in ins] + [a.copy() for a in outs]
    for st in steps:
        for c in range(st["cbeg"], st["cend"]):
            lo, hi = min(c * C, n), min((c + 1) * C, n)
            if lo >= hi:
                continue
            if st["kind"] == "copy":
                bufs[st["dst"]][lo:hi] = bufs[st["srcs"][0]][lo:hi]
                continue
            with np.errstate(over="ignore"):
                acc = decode64(bufs[st["srcs"][0]][lo:hi], dtype).astype(np.float32)
                for b in st["srcs"][1:]:
                    acc = acc + decode64(bufs[b][lo:hi], dtype).astype(np.float32)
            y = wl.bits(torch.from_numpy(acc.copy()).to(wl.TORCH_DTYPE[dtype]))
            bufs[st["dst"]][lo:hi] = y
    return bufs[:R], bufs[R:]


def random_program(dtype, seed):
    """(steps, ins, outs, nchunks): 16 random copy/reduce steps over 4 ranks,
    writes into inputs included, on seeded inputs."""
    import random
    rng = random.Random(seed)
    R, n, nch = 4, 101 + seed * 37, 5
    steps = []
    for _ in range(16):
        cb = rng.randrange(nch)
        ce = rng.randrange(cb + 1, nch + 1)
        kind = rng.choice(["copy", "reduce"])
        sk = rng.choice([0, 1])
        srcs = [sk * R + rng.randrange(R)] if kind == "copy" else \
            [sk * R + rng.randrange(R) for _ in range(rng.randint(1, R))]
        steps.append(dict(kind=kind, rank=rng.randrange(R), dst=rng.randrange(2 * R),
                          srcs=srcs, cbeg=cb, cend=ce))
    ins = _ins(R, n, dtype, config=81, dist="normal")
    outs = [wl.bits(t) for t in wl.make_inputs(82, R, n, dtype, "normal")]
    return steps, ins, outs, nch


@pytest.mark.parametrize("dtype", DTYPES)
@pytest.mark.parametrize("seed", range(6))
def test_random_programs_match_a_python_restatement(dtype, seed):
    """Random copy/reduce programs (writes into inputs included): the oracle's
    plan interpreter against an independent restatement of the plan's
    meaning, bit for bit, on every buffer."""
    steps, ins, outs, nch = random_program(dtype, seed)
    R = len(ins)
    want_in, want_out = _python_plan(steps, ins, outs, dtype, nch)
    got_in, got_out = [a.copy() for a in ins], [a.copy() for a in outs]
    oracle.plan_run(steps, got_in, got_out, DT_CODE[dtype], nch)
    for r in range(R):
        assert np.array_equal(as_uint(got_in[r], dtype), as_uint(want_in[r], dtype))
        assert np.array_equal(as_uint(got_out[r], dtype), as_uint(want_out[r], dtype))
