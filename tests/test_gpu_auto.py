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


@pytest.mark.parametrize("R", [2, 3, 4, 6, 8, 16, 24, 32])
def test_untuned_rule(R):
    """Before ar_tune: LL only for the one-shot at R >= 24 up to 4 KiB per
    rank, HB otherwise; with HB one-shot for R <= 2 at every size, for R = 4
    up to 256 KiB, for R = 16 up to 128 KiB and for other 8 <= R <= 24 up to
    64 KiB, two-shot otherwise."""
    need_gpu()
    with ar.Handle(R, 1 << 23, "bf16") as h:
        for nbytes in (512, 4096, 4098, 64 << 10, (64 << 10) + 2, 128 << 10, (128 << 10) + 2,
                       256 << 10, (256 << 10) + 2, 1 << 20, 8 << 20, 16 << 20):
            if R >= 24 and nbytes <= 4 << 10:
                want = (ar.AR_ONE_SHOT, ar.AR_LL)
            else:
                if R <= 2:
                    one = True
                elif R == 4:
                    one = nbytes <= 256 << 10
                elif R == 16:
                    one = nbytes <= 128 << 10
                else:
                    one = 8 <= R <= 24 and nbytes <= 64 << 10
                want = (ar.AR_ONE_SHOT if one else ar.AR_TWO_SHOT, ar.AR_HB)
            assert ar.ar_get_tuning(h.h, nbytes)[:2] == want, (R, nbytes)
        assert ar.ar_get_tuning(h.h, 4 << 20)[2] == [0.0, 0.0, 0.0, 0.0]
    if R >= 24:
        with ar.Handle(R, (128 << 20) // 2, "bf16") as h:      # beyond the LL limit: HB's rule
            assert ar.ar_get_info(h.h)["ll_capable"] == 0
            want = ar.AR_ONE_SHOT if R <= 24 else ar.AR_TWO_SHOT
            assert ar.ar_get_tuning(h.h, 1024)[:2] == (want, ar.AR_HB)


@pytest.mark.parametrize("R", [2, 4, 8, 16, 32])
def test_untuned_staging_rule(R):
    """Before ar_tune, two-shot HB stages with TMA only in the bands where it
    measured faster (by bytes moved per call, T = 2 R n elem_size: 4 <= R <= 16
    and T >= 1 GiB; R >= 32 and 64 KiB-128 MiB; 16 <= R < 32 and 128 KiB-1 MiB or
    16-64 MiB; 8 <= R < 16 and 16-64 MiB), directly elsewhere; a fixed
    setting overrides it."""
    need_gpu()
    KiB, MiB = 1 << 10, 1 << 20

    def band(R, T):
        if 4 <= R <= 16 and T >= 1 << 30:
            return True
        if R >= 32:
            return 64 * KiB <= T <= 128 * MiB
        if R >= 16:
            return 128 * KiB <= T <= MiB or 16 * MiB <= T <= 64 * MiB
        if R >= 8:
            return 16 * MiB <= T <= 64 * MiB
        return False
    with ar.Handle(R, 64 << 20, "bf16") as h:          # 128 MiB per rank
        for nbytes in [1024, 4096, 16384, 65536, 1 << 20, 2 << 20, 4 << 20, 8 << 20, 32 << 20,
                       64 << 20, 128 << 20]:
            T = 2 * R * nbytes
            want = ar.AR_HB_STAGING_TMA if band(R, T) else ar.AR_HB_STAGING_DIRECT
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


PATHS = [(ar.AR_ONE_SHOT, ar.AR_HB), (ar.AR_TWO_SHOT, ar.AR_HB), (ar.AR_ONE_SHOT, ar.AR_LL),
         (ar.AR_TWO_SHOT, ar.AR_LL)]
PATH_IDS = ["one_shot_hb", "two_shot_hb", "one_shot_ll", "two_shot_ll"]


def _divided_case(R, n, dtype, algo, proto, divisor, offset=0, staging=None):
    from gpu_helpers import device_inputs
    cpu = wl.make_inputs(74, R, n, dtype, "loguniform")
    want = expected(cpu, dtype)
    ins = device_inputs(cpu, offset)
    bufs, outs = guarded_outputs(R, n, dtype, offset)
    with ar.Handle(R, n, dtype) as h:
        ar.ar_set_grid_divisor(h.h, divisor)
        if staging is not None:
            ar.ar_set_hb_staging(h.h, staging)
        assert ar.ar_get_grid_divisor(h.h, n * wl.ELEM_SIZE[dtype], algo, proto) == divisor
        ar.ar_allreduce(h.h, ins, outs, algo, proto)
        assert ar.ar_status(h.h) == ar.AR_OK
    for r in range(R):
        assert_bits_equal(outs[r], want, dtype, "R=%d n=%d div=%d rank %d" % (R, n, divisor, r))
    check_guards(bufs, n, dtype, offset)


@pytest.mark.parametrize("divisor", [2, 4, 8])
@pytest.mark.parametrize("path", PATHS, ids=PATH_IDS)
def test_grid_divisor_every_path(path, divisor):
    """Every path with its CTA cap divided (each CTA serving more of the
    message): sizes large enough to reach the caps, a ragged tail, and
    buffers off 16- and 8-byte alignment (the element-wise and per-rank
    kernels); the same bits as the oracle."""
    need_gpu()
    algo, proto = path
    _divided_case(8, (1 << 18) + 3, "bf16", algo, proto, divisor)
    _divided_case(5, (1 << 17) + 1, "bf16", algo, proto, divisor, offset=1)
    if proto == ar.AR_HB:
        _divided_case(16, (1 << 20) + 5, "fp16", algo, proto, divisor)


@pytest.mark.parametrize("divisor", [2, 4])
@pytest.mark.parametrize("staging", [ar.AR_HB_STAGING_TMA, ar.AR_HB_STAGING_DIRECT],
                         ids=["tma", "direct"])
def test_grid_divisor_two_shot_stagings(staging, divisor):
    """Two-shot HB with each staging and a divided grid, up to the binary32
    wide form (more than 64 MiB moved, 384-thread CTAs)."""
    need_gpu()
    _divided_case(8, (4 << 20) + 1, "fp32", ar.AR_TWO_SHOT, ar.AR_HB, divisor, staging=staging)
    _divided_case(32, (1 << 16) + 7, "bf16", ar.AR_TWO_SHOT, ar.AR_HB, divisor, staging=staging)


def test_grid_divisor_setting_and_tuning():
    """The forced divisor is reported for every path and rejected outside
    0, 1, 2, 4, 8; ar_tune picks 1, 2 or 4 per size and path, and calls
    after tuning (forced paths and AUTO) stay exact."""
    need_gpu()
    R, N, dtype = 8, (1 << 20) + 3, "bf16"
    cpu = wl.make_inputs(75, R, N, dtype, "normal")
    with ar.Handle(R, N, dtype) as h:
        for a, p in PATHS:
            assert ar.ar_get_grid_divisor(h.h, 4096, a, p) == 1
        for bad in (-1, 3, 16):
            with pytest.raises(ar.ArError):
                ar.ar_set_grid_divisor(h.h, bad)
        for a, p, nbytes in ((ar.AR_ALGO_AUTO, ar.AR_HB, 16), (ar.AR_ONE_SHOT, 5, 16),
                             (ar.AR_ONE_SHOT, ar.AR_HB, 0), (ar.AR_ONE_SHOT, ar.AR_HB, 2 * N + 1)):
            with pytest.raises(ar.ArError):
                ar.ar_get_grid_divisor(h.h, nbytes, a, p)
        ar.ar_set_grid_divisor(h.h, 4)
        assert ar.ar_get_grid_divisor(h.h, 4096, ar.AR_TWO_SHOT, ar.AR_LL) == 4
        ar.ar_set_grid_divisor(h.h, 0)
        ar.ar_tune(h.h)
        for lg in range(9, 22):
            for a, p in PATHS:
                assert ar.ar_get_grid_divisor(h.h, 1 << lg, a, p) in (1, 2, 4), (lg, a, p)
        for choice in [(ar.AR_ALGO_AUTO, ar.AR_PROTO_AUTO)] + PATHS:
            for n in (1000, 70001, (1 << 19) + 7, N):
                _prefix_case(h.h, R, N, n, dtype, *choice, cpu)


@pytest.mark.parametrize("R,sizes", [
    (8, [128 << 10, 256 << 10, 512 << 10, 1 << 20, 2 << 20]),
    (16, [64 << 10, 128 << 10, 256 << 10, 512 << 10, 1 << 20]),
    (4, [256 << 10, 512 << 10, 1 << 20, 2 << 20, 4 << 20]),
    (32, [64 << 10, 256 << 10])], ids=["r8", "r16", "r4", "r32"])
def test_one_shot_hb_untuned_divisor(R, sizes):
    """Before ar_tune, one-shot HB runs a quarter of its CTA cap where the
    full cap would give every CTA at most two runs of a mid-sized message
    (R <= 16: more runs than a quarter of the cap, at most twice the cap; a
    run is 32 16-byte units of every rank for one CTA of 8 warps, or R warps
    above 8 ranks, and the cap fills 2048 threads per SM), the full cap
    elsewhere; a forced divisor overrides it.  On 152 SMs the middle three
    sizes of R = 4, 8 and 16 take the quarter."""
    need_gpu()
    with ar.Handle(R, 2 << 20, "bf16") as h:
        sms = ar.ar_get_info(h.h)["num_sms"]
        warps = R * ((8 + R - 1) // R) if R <= 8 else R
        cap = sms * (2048 // (32 * warps))
        per_run = (warps // R) * 32
        for nbytes in sizes:
            runs = -(-(nbytes // 16) // per_run)
            want = 4 if R <= 16 and cap // 4 < runs <= 2 * cap else 1
            got = ar.ar_get_grid_divisor(h.h, nbytes, ar.AR_ONE_SHOT, ar.AR_HB)
            assert got == want, (R, nbytes, got)
            assert ar.ar_get_grid_divisor(h.h, nbytes, ar.AR_TWO_SHOT, ar.AR_HB) == 1
        ar.ar_set_grid_divisor(h.h, 1)
        for nbytes in sizes:
            assert ar.ar_get_grid_divisor(h.h, nbytes, ar.AR_ONE_SHOT, ar.AR_HB) == 1
