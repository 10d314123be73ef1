"""Messages shorter than the handle's N, and the AUTO choice of schedule and
protocol (before and after ar_tune), against the oracle."""
import numpy as np
import pytest
import torch

import all_reduce_reduction_gb300 as ar
from all_reduce_reduction_gb300 import workload as wl
from gpu_helpers import assert_bits_equal, check_guards, expected, guarded_outputs, need_gpu

pytestmark = pytest.mark.gpu

CHOICES = [(ar.AR_ALGO_AUTO, ar.AR_PROTO_AUTO), (ar.AR_ALGO_AUTO, ar.AR_LL),
           (ar.AR_ALGO_AUTO, ar.AR_HB), (ar.AR_ONE_SHOT, ar.AR_PROTO_AUTO),
           (ar.AR_TWO_SHOT, ar.AR_PROTO_AUTO), (ar.AR_ONE_SHOT, ar.AR_LL),
           (ar.AR_TWO_SHOT, ar.AR_HB)]
CHOICE_IDS = ["auto_auto", "auto_ll", "auto_hb", "one_auto", "two_auto", "one_ll", "two_hb"]


def _prefix_case(h, R, N, n, dtype, algo, proto, cpu):
    ins = [t.cuda() for t in cpu]
    bufs, outs = guarded_outputs(R, N, dtype)
    ar.ar_allreduce_n(h, ins, outs, n, algo, proto)
    assert ar.ar_status(h) == ar.AR_OK
    want = expected([t[:n] for t in cpu], dtype)
    for r in range(R):
        assert_bits_equal(outs[r][:n], want, dtype, "n=%d rank %d" % (n, r))
    # elements past n are untouched (they still hold the canary)
    check_guards(bufs, n, dtype)


@pytest.mark.parametrize("choice", CHOICES, ids=CHOICE_IDS)
@pytest.mark.parametrize("dtype", ["bf16", "fp32"])
def test_prefix_messages_before_tuning(choice, dtype):
    need_gpu()
    R, N = 8, (1 << 20) + 3
    cpu = wl.make_inputs(70, R, N, dtype, "loguniform")
    with ar.Handle(R, N, dtype) as h:
        for n in (1, 9, 512, 4097, 1 << 16, (1 << 18) + 1, (1 << 19) + 7, N):
            _prefix_case(h.h, R, N, n, dtype, *choice, cpu)


def test_n_out_of_range_rejected():
    need_gpu()
    x = [torch.zeros(100, dtype=torch.bfloat16, device="cuda") for _ in range(2)]
    y = [torch.zeros(100, dtype=torch.bfloat16, device="cuda") for _ in range(2)]
    with ar.Handle(2, 100, "bf16") as h:
        for n in (0, 101):
            with pytest.raises(ar.ArError) as e:
                ar.ar_allreduce_n(h.h, x, y, n)
            assert e.value.code == ar.AR_ERR_INVALID
        with pytest.raises(ar.ArError):
            ar.ar_allreduce_n(h.h, x, y, 10, 7, ar.AR_HB)


@pytest.mark.parametrize("R", [4, 8, 16, 32])
def test_untuned_rule(R):
    """Before ar_tune: HB, one-shot up to max(64 KiB, 512 KiB / R) per rank,
    two-shot above."""
    need_gpu()
    limit = max(64 << 10, (512 << 10) // R)
    with ar.Handle(R, 1 << 21, "bf16") as h:
        assert ar.ar_get_tuning(h.h, 4096)[:2] == (ar.AR_ONE_SHOT, ar.AR_HB)
        assert ar.ar_get_tuning(h.h, limit)[:2] == (ar.AR_ONE_SHOT, ar.AR_HB)
        assert ar.ar_get_tuning(h.h, limit + 2)[:2] == (ar.AR_TWO_SHOT, ar.AR_HB)
        assert ar.ar_get_tuning(h.h, 4 << 20)[2] == [0.0, 0.0, 0.0, 0.0]


@pytest.mark.parametrize("R,dtype", [(8, "bf16"), (4, "fp32"), (16, "fp16")])
def test_tune_picks_fastest_and_stays_exact(R, dtype):
    need_gpu()
    N = (1 << 21) + 1
    cpu = wl.make_inputs(71, R, N, dtype, "normal")
    with ar.Handle(R, N, dtype) as h:
        ar.ar_tune(h.h)
        esz = wl.ELEM_SIZE[dtype]
        # every tuned bucket: the AUTO choice is the fastest timed pair
        for lg in range(9, 24):
            a, p, us = ar.ar_get_tuning(h.h, 1 << lg)
            assert all(u > 0 for u in us), (lg, us)
            k = int(np.argmin(us))
            assert (a, p) == (k // 2, k % 2), (lg, us)
        # sizes round up to the next power of two
        assert ar.ar_get_tuning(h.h, 513)[2] == ar.ar_get_tuning(h.h, 1024)[2]
        assert ar.ar_get_tuning(h.h, 1)[2] == ar.ar_get_tuning(h.h, 512)[2]
        # above the largest tuned size the largest tuned bucket's choice holds
        assert ar.ar_get_tuning(h.h, 1 << 26)[:2] == ar.ar_get_tuning(h.h, 1 << 23)[:2]
        for n in (3, 1000, 70001, (1 << 20) // esz * 2 + 5, N):
            for choice in CHOICES[:5]:
                _prefix_case(h.h, R, N, n, dtype, *choice, cpu)


def test_auto_in_a_captured_graph():
    need_gpu()
    R, N = 8, 1 << 18
    h = ar.Handle(R, N, "bf16")
    ar.ar_tune(h.h)
    ins = [torch.empty(N, dtype=torch.bfloat16, device="cuda") for _ in range(R)]
    outs = [torch.empty_like(t) for t in ins]
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        for t in ins:
            t.zero_()
        for n in (512, 8192, N):
            ar.ar_allreduce_n(h.h, ins, outs, n, stream=s)
    s.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        for n in (512, 8192, N):
            for _ in range(3):
                ar.ar_allreduce_n(h.h, ins, outs, n, stream=s)
    for rep in range(2):
        cpu = wl.make_inputs(72 + rep, R, N, "bf16", "uniform")
        for t, c in zip(ins, cpu):
            t.copy_(c)
        g.replay()
        torch.cuda.synchronize()
        assert ar.ar_status(h.h) == ar.AR_OK
        want = expected(cpu, "bf16")
        for r in range(R):
            assert_bits_equal(outs[r], want, "bf16", "replay %d rank %d" % (rep, r))
    h.close()


@pytest.mark.parametrize("R", [2, 4, 8, 16, 32])
def test_untuned_staging_rule(R):
    """Before ar_tune, two-shot HB stages with TMA only in the band where it
    measured faster (R >= 16 and 16-64 MiB moved per call, or R >= 32 and
    256 KiB-64 MiB), directly elsewhere; a fixed setting overrides it."""
    need_gpu()
    MiB = 1 << 20
    with ar.Handle(R, 64 << 20, "bf16") as h:
        for nbytes in [1024, 4096, 65536, 1 << 20, 2 << 20, 4 << 20, 8 << 20, 32 << 20, 64 << 20]:
            T = 2 * R * nbytes
            band = (R >= 16 and 16 * MiB <= T <= 64 * MiB) or (R >= 32 and 256 * 1024 <= T <= 64 * MiB)
            want = ar.AR_HB_STAGING_TMA if band else ar.AR_HB_STAGING_DIRECT
            assert ar.ar_get_hb_staging(h.h, nbytes) == want, (R, nbytes)
        for fixed in (ar.AR_HB_STAGING_TMA, ar.AR_HB_STAGING_DIRECT):
            ar.ar_set_hb_staging(h.h, fixed)
            assert ar.ar_get_hb_staging(h.h, 4096) == fixed
            assert ar.ar_get_info(h.h)["hb_staging"] == fixed
        with pytest.raises(ar.ArError):
            ar.ar_set_hb_staging(h.h, 3)
        with pytest.raises(ar.ArError):
            ar.ar_get_hb_staging(h.h, 0)


@pytest.mark.parametrize("R,dtype", [(8, "bf16"), (32, "fp32")])
def test_tune_keeps_the_faster_staging(R, dtype):
    """ar_tune times two-shot HB with both stagings and keeps one per size;
    either way the results stay exact."""
    need_gpu()
    N = (1 << 20) + 3
    cpu = wl.make_inputs(73, R, N, dtype, "normal")
    with ar.Handle(R, N, dtype) as h:
        ar.ar_tune(h.h)
        esz = wl.ELEM_SIZE[dtype]
        seen = set()
        for lg in range(9, 24):
            if (1 << lg) > N * esz:
                break
            st = ar.ar_get_hb_staging(h.h, 1 << lg)
            assert st in (ar.AR_HB_STAGING_TMA, ar.AR_HB_STAGING_DIRECT), (lg, st)
            seen.add(st)
        assert seen
        for n in (1000, 70001, N):
            _prefix_case(h.h, R, N, n, dtype, ar.AR_TWO_SHOT, ar.AR_HB, cpu)
