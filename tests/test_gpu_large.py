"""Messages above 4 GiB per rank: byte offsets past 2^32 on every HB path.

A handle takes up to 2^40 bytes per rank, and every HB kernel indexes its
buffers in 64 bits.  These cases run each HB path (and the reduce-scatter and
all-gather steps, the built-in two-shot plan and the weighted combine) on a
message of a little more than 4 GiB per rank with a ragged tail, and compare
every element of every output with the CPU oracle, bit for bit.

Inputs: rank r's buffer repeats a seeded block of L = 2^20 + 7 elements drawn
by the workload generator.  L is odd, so an offset that wrapped at 2^32
bytes (or at any power of two) would read another position of the block and
show as a mismatch.  The oracle folds the R blocks once; element i of every
output must equal the oracle's element i mod L.  Canaries around the outputs
catch a store past either end.  Each case holds 12-36 GiB on the device."""
import numpy as np
import pytest
import torch

import all_reduce_reduction_gb300 as ar
import oracle
from all_reduce_reduction_gb300 import workload as wl
from gpu_helpers import UINT_T, check_guards, guarded_outputs, need_gpu

pytestmark = pytest.mark.gpu

L = (1 << 20) + 7
FOUR_GIB = 1 << 32


def periodic(block: torch.Tensor, n: int) -> torch.Tensor:
    """n elements on the device repeating the CPU tensor `block` (a view of
    a buffer holding whole periods)."""
    reps = -(-n // block.numel())
    return block.cuda().repeat(reps)[:n]


def assert_same_bits(got: torch.Tensor, want: torch.Tensor, dtype: str, what: str):
    """Bitwise equality of two device tensors of one dtype."""
    a, b = got.view(UINT_T[dtype]), want.view(UINT_T[dtype])
    if not torch.equal(a, b):
        i = int(torch.argmax((a != b).to(torch.uint8)))
        mask = 0xFFFFFFFF if dtype == "fp32" else 0xFFFF
        raise AssertionError("%s: first difference at element %d (byte %d): got %#x want %#x"
                             % (what, i, i * wl.ELEM_SIZE[dtype], int(a[i]) & mask,
                                int(b[i]) & mask))


CASES = [  # (R, dtype, n, distribution): more than 4 GiB per rank, ragged tails
    (2, "bf16", (1 << 31) + 13, "uniform"),
    (4, "fp32", (1 << 30) + 5, "loguniform"),
]


@pytest.mark.parametrize("R,dtype,n,dist", CASES, ids=["r2_bf16", "r4_fp32"])
def test_hb_paths_above_4_gib_per_rank(R, dtype, n, dist):
    """One-shot HB, two-shot HB with either staging (R = 4 above 1 GiB
    moved: the TMA one-stage form), the reduce-scatter and all-gather steps,
    the built-in two-shot plan, and one-shot HB in place."""
    need_gpu()
    assert n * wl.ELEM_SIZE[dtype] > FOUR_GIB
    blocks = wl.make_inputs(70 + R, R, L, dtype, dist)
    want_block = oracle.allreduce([wl.bits(t) for t in blocks], wl.DTYPE_CODE[dtype])[0]
    want = periodic(wl.from_bits(want_block, dtype), n)
    ins = [periodic(b, n) for b in blocks]
    bufs, outs = guarded_outputs(R, n, dtype)
    with ar.Handle(R, n, dtype) as h:
        runs = [("one-shot HB", ar.AR_ONE_SHOT, ar.AR_HB_STAGING_AUTO),
                ("two-shot HB, TMA staging", ar.AR_TWO_SHOT, ar.AR_HB_STAGING_TMA),
                ("two-shot HB, direct staging", ar.AR_TWO_SHOT, ar.AR_HB_STAGING_DIRECT)]
        for what, algo, staging in runs:
            for o in outs:
                o.view(UINT_T[dtype]).fill_(0x7FA5)
            ar.ar_set_hb_staging(h.h, staging)
            ar.ar_allreduce(h.h, ins, outs, algo, ar.AR_HB)
            torch.cuda.synchronize()
            assert ar.ar_status(h.h) == ar.AR_OK, what
            for r in range(R):
                assert_same_bits(outs[r], want, dtype, "%s, rank %d" % (what, r))
            check_guards(bufs, n, dtype)

        # reduce-scatter: shard j of out[j] only; the rest keeps its fill
        fill = 0x1234
        for o in outs:
            o.view(UINT_T[dtype]).fill_(fill)
        ar.ar_reduce_scatter(h.h, ins, outs)
        torch.cuda.synchronize()
        assert ar.ar_status(h.h) == ar.AR_OK
        for j in range(R):
            lo, hi = oracle.shard_bounds(R, n, wl.DTYPE_CODE[dtype], j)
            assert_same_bits(outs[j][lo:hi], want[lo:hi], dtype, "reduce-scatter shard %d" % j)
            rest = outs[j].view(UINT_T[dtype])
            assert bool((rest[:lo] == fill).all()) and bool((rest[hi:] == fill).all()), \
                "reduce-scatter wrote outside shard %d" % j
        ar.ar_all_gather(h.h, outs)
        torch.cuda.synchronize()
        assert ar.ar_status(h.h) == ar.AR_OK
        for r in range(R):
            assert_same_bits(outs[r], want, dtype, "all-gather, rank %d" % r)
        check_guards(bufs, n, dtype)

        p = ar.ar_plan_builtin(h.h, "two_shot")
        try:
            for o in outs:
                o.view(UINT_T[dtype]).fill_(0x7FA5)
            ar.ar_plan_execute(p, ins, outs)
            torch.cuda.synchronize()
            assert ar.ar_status(h.h) == ar.AR_OK
        finally:
            ar.ar_plan_destroy(p)
        for r in range(R):
            assert_same_bits(outs[r], want, dtype, "built-in two-shot plan, rank %d" % r)
        check_guards(bufs, n, dtype)

        del outs, bufs
        torch.cuda.empty_cache()
        ar.ar_allreduce(h.h, ins, ins, ar.AR_ONE_SHOT, ar.AR_HB)     # in place, last
        torch.cuda.synchronize()
        assert ar.ar_status(h.h) == ar.AR_OK
        for r in range(R):
            assert_same_bits(ins[r], want, dtype, "one-shot HB in place, rank %d" % r)
    del ins, want
    torch.cuda.empty_cache()


def test_combine_above_4_gib_per_source():
    """Weighted combine, K = 2 bf16 sources of T = 2^18 + 1 tokens x 8192
    (4 GiB + 16 KiB each).  Token 2^18 starts exactly at byte 2^32.  The
    oracle computes sampled tokens, one by one, from the same block and
    weights; the output's canaries are checked whole."""
    need_gpu()
    K, H, dtype = 2, 8192, "bf16"
    T = (1 << 18) + 1
    n = T * H
    assert n * 2 > FOUR_GIB
    blocks = wl.make_inputs(75, K, L, dtype, "normal")
    wts = wl.gate_weights(wl.seed_for(75, 1000), T, K)
    ys = [periodic(b, n) for b in blocks]
    bufs, (out,) = guarded_outputs(1, n, dtype)
    with ar.Handle(K, n, dtype) as h:
        ar.ar_combine(h.h, ys, torch.from_numpy(wts).cuda(), out, T, H)
        torch.cuda.synchronize()
        assert ar.ar_status(h.h) == ar.AR_OK
    check_guards(bufs, n, dtype)

    rng = np.random.default_rng(75)
    tokens = sorted({0, 1, (1 << 18) - 1, 1 << 18, T - 1,
                     *rng.integers(0, T, size=27).tolist()})
    block_bits = [wl.bits(b) for b in blocks]
    for t in tokens:
        pos = (np.arange(t * H, (t + 1) * H, dtype=np.int64)) % L
        rows = [np.ascontiguousarray(bb[pos]) for bb in block_bits]
        want = oracle.combine(rows, wts[t * K:(t + 1) * K], 1, H, wl.DTYPE_CODE[dtype])
        got = wl.bits(out[t * H:(t + 1) * H].cpu())
        bad = np.nonzero(got != want)[0]
        assert bad.size == 0, "token %d: %d of %d elements differ; first at %d: got %#x want %#x" % (
            t, bad.size, H, int(bad[0]), int(got[bad[0]]), int(want[bad[0]]))
    del ys, out, bufs
    torch.cuda.empty_cache()
