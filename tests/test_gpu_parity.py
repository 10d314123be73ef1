"""GPU parity: every schedule and protocol against the CPU oracle, bit for bit.

Inputs come from the seeded generator; the expected values from the oracle
alone.  Outputs sit between canary zones that must stay untouched.
"""
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


def run_case(R, n, dtype, algo, proto, dist="loguniform", config=40, offset=0, inplace=False,
             transport=None, staging=None):
    need_gpu()
    cpu = wl.make_inputs(config, R, n, dtype, dist)
    want = expected(cpu, dtype)
    ins = device_inputs(cpu, offset)
    if inplace:
        outs, bufs = ins, None
    else:
        bufs, outs = guarded_outputs(R, n, dtype, offset)
    with ar.Handle(R, n, dtype) as h:
        if transport is not None:
            ar.ar_set_ll_transport(h.h, transport)
        if staging is not None:
            ar.ar_set_hb_staging(h.h, staging)
        ar.ar_allreduce(h.h, ins, outs, algo, proto)
        st = ar.ar_status(h.h)
        assert st == ar.AR_OK, ar.ar_strerror(st)
    for r in range(R):
        assert_bits_equal(outs[r], want, dtype, "R=%d n=%d %s rank %d" % (R, n, dtype, r))
    if bufs is not None:
        check_guards(bufs, n, dtype, offset)


def test_small_config_every_path():
    """8 ranks x 512 bf16, uniform [-1, 1): the small workload."""
    w = wl.SMALL
    for algo, proto in ALL_PATHS:
        run_case(w.R, w.n, w.dtype, algo, proto, dist=w.dist, config=w.config)


@pytest.mark.parametrize("path", ALL_PATHS, ids=PATH_IDS)
@pytest.mark.parametrize("dtype", DTYPES)
@pytest.mark.parametrize("R", [1, 2, 3, 8, 16, 32])
@pytest.mark.parametrize("n", [1, 3, 8, 9, 100, 4097, 70001])
def test_parity_matrix(path, dtype, R, n):
    run_case(R, n, dtype, *path)


TRANSPORTS = [ar.AR_LL_GLOBAL, ar.AR_LL_CLUSTER]
TRANSPORT_IDS = ["global", "cluster"]


@pytest.mark.parametrize("transport", TRANSPORTS, ids=TRANSPORT_IDS)
@pytest.mark.parametrize("dtype", DTYPES)
@pytest.mark.parametrize("R", [1, 2, 3, 5, 8, 12, 16])
@pytest.mark.parametrize("n", [1, 7, 8, 9, 100, 4097, 70001, (1 << 20) + 3])
def test_ll_one_shot_transports(transport, dtype, R, n):
    """One-shot LL through HBM slots and through cluster shared memory."""
    run_case(R, n, dtype, ar.AR_ONE_SHOT, ar.AR_LL, transport=transport)


def test_cluster_transport_available_up_to_eight_ranks():
    need_gpu()
    for R in (1, 2, 3, 4, 5, 6, 7, 8):
        with ar.Handle(R, 4096, "bf16") as h:
            info = ar.ar_get_info(h.h)
            assert info["ll_cluster_ok"] == 1 and info["ll_cluster_max"] > 0, (R, info)


def test_info_reports_launch_capacities():
    need_gpu()
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    for R in (1, 8, 32):
        with ar.Handle(R, 4096, "fp32") as h:
            info = ar.ar_get_info(h.h)
            assert info["num_sms"] == sms
            # the staged kernel: at least one CTA per SM, at most one epoch word
            # each (2048 words)
            assert sms <= info["ll_staged_ctas_max"] <= 2048, info
            assert info["ll_ctas_per_rank_max"] >= 1, info


@pytest.mark.parametrize("transport", TRANSPORTS, ids=TRANSPORT_IDS)
@pytest.mark.parametrize("offset", [0, 1])
def test_ll_transports_in_place(transport, offset):
    run_case(8, 70001, "bf16", ar.AR_ONE_SHOT, ar.AR_LL, transport=transport, offset=offset,
             inplace=True)


@pytest.mark.parametrize("path", ALL_PATHS, ids=PATH_IDS)
@pytest.mark.parametrize("dtype", DTYPES)
@pytest.mark.parametrize("R", [4, 16])
def test_many_tiles_ragged_tail(path, dtype, R):
    """Over a million elements: many TMA tiles / LL units, plus a ragged tail."""
    run_case(R, (1 << 20) + 5, dtype, *path, dist="normal")


@pytest.mark.parametrize("R,n,dtype", [(8, (4 << 20) + 3, "bf16"), (16, (2 << 20) + 5, "fp16"),
                                       (32, (1 << 20) + 7, "fp32"), (3, 3 << 20, "bf16"),
                                       (5, (2 << 20) + 1, "fp32")],
                         ids=["r8_bf16", "r16_fp16", "r32_fp32", "r3_bf16", "r5_fp32"])
def test_two_shot_tma_many_items_per_cta(R, n, dtype):
    """Two-shot HB with every CTA folding 5 to 14 items, so each shared-memory
    stage is refilled by the producer many times while the consumers fold and
    store the items before it: R fixed at compile time (8, 16, 32) and a
    runtime R (3, 5), each with a ragged tail."""
    run_case(R, n, dtype, ar.AR_TWO_SHOT, ar.AR_HB, dist="normal", staging=ar.AR_HB_STAGING_TMA)
    with ar.Handle(R, n, dtype) as h:
        info = ar.ar_get_info(h.h)
    body = n * wl.ELEM_SIZE[dtype] // 16 * 16
    items = -(-body // info["tma_tile_bytes"])
    assert items >= 5 * info["num_sms"], (items, info["tma_tile_bytes"])


STAGINGS = [ar.AR_HB_STAGING_TMA, ar.AR_HB_STAGING_DIRECT]
STAGING_IDS = ["tma", "direct"]


@pytest.mark.parametrize("staging", STAGINGS, ids=STAGING_IDS)
@pytest.mark.parametrize("dtype", DTYPES)
@pytest.mark.parametrize("R", [1, 3, 8, 16, 32])
@pytest.mark.parametrize("n", [1, 9, 100, 4097, 70001, (1 << 20) + 5])
def test_two_shot_hb_stagings(staging, dtype, R, n):
    """Two-shot HB with each staging forced: the same bits as the oracle
    (buffers 16-byte aligned, so the chosen staging runs)."""
    run_case(R, n, dtype, ar.AR_TWO_SHOT, ar.AR_HB, staging=staging)


@pytest.mark.parametrize("staging", STAGINGS, ids=STAGING_IDS)
@pytest.mark.parametrize("offset", [0, 1])
def test_two_shot_hb_stagings_in_place(staging, offset):
    """In place, aligned (the chosen staging) and one element off (element by
    element whatever the setting)."""
    run_case(8, 300001, "bf16", ar.AR_TWO_SHOT, ar.AR_HB, offset=offset, inplace=True,
             staging=staging)


@pytest.mark.parametrize("R,n,dtype,inplace", [(5, (1 << 26) + 3, "bf16", False),
                                               (4, (1 << 25) + 1, "fp32", False),
                                               (4, (1 << 25) + 1, "fp32", True)],
                         ids=["r5_bf16", "r4_fp32", "r4_fp32_in_place"])
def test_two_shot_tma_one_stage_form(R, n, dtype, inplace):
    """Two-shot HB with TMA staging on calls moving 1 GiB or more (one stage
    of 128 KiB per CTA, two CTAs per SM in turn): a runtime rank count and
    R = 4 (32 KiB tiles), each with a ragged tail, and in place; the same
    bits as the oracle."""
    assert 2 * R * n * wl.ELEM_SIZE[dtype] >= 1 << 30
    run_case(R, n, dtype, ar.AR_TWO_SHOT, ar.AR_HB, dist="normal", inplace=inplace,
             staging=ar.AR_HB_STAGING_TMA)


def wide_threshold_units():
    """16-byte vectors per rank from which a binary32 two-shot HB call moving
    more than 64 MiB runs its direct staging in 384-thread CTAs: the grid of
    those reaches the thread count of the 256-thread grid (8 CTAs per SM)."""
    with ar.Handle(1, 1, "fp32") as h:
        sms = ar.ar_get_info(h.h)["num_sms"]
    cap = sms * 8 * 256 // 384
    return (cap - 1) * 384 + 1


@pytest.mark.parametrize("R,extra", [(8, -1), (8, 0), (32, 0), (3, None)],
                         ids=["r8_below", "r8_from", "r32_from", "r3_many_waves"])
def test_two_shot_direct_fp32_wide_form(R, extra):
    """binary32, direct staging, more than 64 MiB moved: one vector below the
    384-thread form's threshold (256-thread CTAs), from it with a ragged tail
    of 3 elements, and far above it (every thread folding several vectors);
    the same bits as the oracle."""
    units = wide_threshold_units() + extra if extra is not None else 2 << 20
    n = units * 4 + (3 if extra == 0 else 0)
    assert 2 * R * n * 4 > (64 << 20)
    run_case(R, n, "fp32", ar.AR_TWO_SHOT, ar.AR_HB, dist="normal", staging=ar.AR_HB_STAGING_DIRECT)


@pytest.mark.parametrize("path", ALL_PATHS, ids=PATH_IDS)
@pytest.mark.parametrize("dtype", DTYPES)
@pytest.mark.parametrize("offset", [1, 2, 3])
def test_misaligned_buffers(path, dtype, offset):
    """Buffers off 16-byte alignment take the element-wise paths."""
    if dtype == "fp32" and offset == 3:
        offset = 1
    run_case(5, 3001, dtype, *path, offset=offset)


@pytest.mark.parametrize("path", ALL_PATHS, ids=PATH_IDS)
@pytest.mark.parametrize("dtype", DTYPES)
@pytest.mark.parametrize("n", [7, 4099, 300001])
def test_in_place(path, dtype, n):
    run_case(8, n, dtype, *path, inplace=True)


@pytest.mark.parametrize("path", ALL_PATHS, ids=PATH_IDS)
def test_in_place_misaligned(path):
    run_case(3, 999, "bf16", *path, offset=1, inplace=True)


def one_shot_hb_span(R, dtype):
    """Elements the one-shot HB grid covers with one run per CTA on this GPU:
    R warps per run of 32 vectors, at least 8 warps per CTA, 2048 threads
    per SM.  One more vector makes some CTA take a second run (the ring)."""
    W = R * -(-8 // R) if R <= 8 else R
    ctas = torch.cuda.get_device_properties(0).multi_processor_count * (2048 // (32 * W))
    return ctas * (W // R) * 32 * (16 // wl.ELEM_SIZE[dtype])


@pytest.mark.parametrize("inplace", [False, True], ids=["out", "inplace"])
@pytest.mark.parametrize("dtype", ["bf16", "fp32"])
@pytest.mark.parametrize("R", [3, 8, 17, 32])
@pytest.mark.parametrize("extra", ["exact", "tail", "one_more_vector", "runs_and_tail"])
def test_one_shot_hb_single_and_ring(extra, R, dtype, inplace):
    """Both sides of the switch from one run per CTA (folded from global, or
    staged once above 16 ranks) to the shared-memory ring, with and without
    a ragged tail, in place and not."""
    need_gpu()
    pv = 16 // wl.ELEM_SIZE[dtype]
    add = {"exact": 0, "tail": pv - 1, "one_more_vector": pv,
           "runs_and_tail": 3 * 32 * pv + pv - 1}[extra]
    run_case(R, one_shot_hb_span(R, dtype) + add, dtype, ar.AR_ONE_SHOT, ar.AR_HB,
             dist="normal", inplace=inplace)


@pytest.mark.parametrize("dtype", DTYPES)
@pytest.mark.parametrize("R,n", [(4, 4097 * 3 + 3), (16, 1001), (5, 9), (32, 70001), (8, 1 << 20)])
def test_reduce_scatter_then_all_gather(dtype, R, n):
    need_gpu()
    cpu = wl.make_inputs(41, R, n, dtype, "normal")
    ins = device_inputs(cpu)
    bufs, outs = guarded_outputs(R, n, dtype)
    # oracle reduce-scatter on the same starting outputs (canary-filled)
    start = [wl.bits(o.cpu()).copy() for o in outs]
    want_rs = oracle.reduce_scatter([wl.bits(t) for t in cpu], wl.DTYPE_CODE[dtype], start)
    with ar.Handle(R, n, dtype) as h:
        ar.ar_reduce_scatter(h.h, ins, outs)
        assert ar.ar_status(h.h) == ar.AR_OK
        for r in range(R):
            assert_bits_equal(outs[r], want_rs[r], dtype, "reduce-scatter rank %d" % r)
        ar.ar_all_gather(h.h, outs)
        assert ar.ar_status(h.h) == ar.AR_OK
    want = expected(cpu, dtype)
    for r in range(R):
        assert_bits_equal(outs[r], want, dtype, "all-gather rank %d" % r)
    check_guards(bufs, n, dtype)


@pytest.mark.parametrize("dtype", DTYPES)
@pytest.mark.parametrize("n", [1, 2, 3, 5, 64, 1001, 1 << 18])
@pytest.mark.parametrize("offset", [0, 1])
def test_ll_pack_unpack_vs_oracle(dtype, n, offset):
    need_gpu()
    x = wl.make_inputs(42, 1, n, dtype, "loguniform")[0]
    flag = 0xC0FFEE00 + n
    want = oracle.ll_pack(wl.bits(x), wl.DTYPE_CODE[dtype], flag)
    src = device_inputs([x], offset)[0]
    P = want.size
    pk_buf = torch.zeros(P + 2, dtype=torch.int64, device="cuda")
    pk = pk_buf[offset: offset + P]
    with ar.Handle(1, n, dtype) as h:
        ar.ar_ll_pack(h.h, src, pk, n, flag)
        got = pk.cpu().numpy().view(np.uint64)
        assert np.array_equal(got, want)
        dst = torch.zeros(n + offset, dtype=x.dtype, device="cuda")[offset:]
        ar.ar_ll_unpack(h.h, pk, dst, n, flag)
        assert ar.ar_status(h.h) == ar.AR_OK
        assert_bits_equal(dst, wl.bits(x), dtype, "unpack")
        # a wrong flag: nothing written, mismatch reported
        dst.zero_()
        ar.ar_ll_unpack(h.h, pk, dst, n, flag + 1)
        assert ar.ar_status(h.h) == ar.AR_ERR_FLAG_MISMATCH
        assert int(dst.view(torch.int16 if dtype != "fp32" else torch.int32).abs().sum()) == 0
        assert ar.ar_status(h.h) == ar.AR_OK        # cleared by the read


@pytest.mark.parametrize("dtype", DTYPES)
def test_ll_unpack_partial_mismatch(dtype):
    need_gpu()
    n = 37
    x = wl.make_inputs(43, 1, n, dtype, "normal")[0]
    pk = oracle.ll_pack(wl.bits(x), wl.DTYPE_CODE[dtype], 9)
    pk[3] = (pk[3] & np.uint64(0xFFFFFFFF)) | (np.uint64(8) << np.uint64(32))
    want = np.zeros(n, dtype=oracle.STORAGE[wl.DTYPE_CODE[dtype]])
    want, bad = oracle.ll_unpack(pk, wl.DTYPE_CODE[dtype], n, 9, dst=want)
    assert bad == 1
    dpk = torch.from_numpy(pk.view(np.int64)).cuda()
    dst = torch.zeros(n, dtype=x.dtype, device="cuda")
    with ar.Handle(1, n, dtype) as h:
        ar.ar_ll_unpack(h.h, dpk, dst, n, 9)
        assert ar.ar_status(h.h) == ar.AR_ERR_FLAG_MISMATCH
    assert_bits_equal(dst, want, dtype, "partial unpack")


@pytest.mark.parametrize("transport", TRANSPORTS, ids=TRANSPORT_IDS)
@pytest.mark.parametrize("path", ALL_PATHS, ids=PATH_IDS)
def test_graph_replays_see_new_inputs(path, transport):
    """10 calls captured in one CUDA graph; the inputs change between replays.
    A flag frozen at capture time would let LL receivers accept the previous
    replay's packets; the device epoch must prevent that."""
    need_gpu()
    R, n, dtype = 8, 4096 + 3, "bf16"
    algo, proto = path
    ins = [torch.empty(n, dtype=torch.bfloat16, device="cuda") for _ in range(R)]
    outs = [torch.empty_like(t) for t in ins]
    h = ar.Handle(R, n, dtype)
    ar.ar_set_ll_transport(h.h, transport)
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        for t in ins:
            t.zero_()
        ar.ar_allreduce(h.h, ins, outs, algo, proto, stream=s)   # warm up outside capture
    s.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        for _ in range(10):
            ar.ar_allreduce(h.h, ins, outs, algo, proto, stream=s)
    for rep in range(4):
        cpu = wl.make_inputs(50 + rep, R, n, dtype, "uniform")
        for t, c in zip(ins, cpu):
            t.copy_(c)
        for o in outs:
            o.fill_(float("nan"))
        g.replay()
        torch.cuda.synchronize()
        assert ar.ar_status(h.h) == ar.AR_OK
        want = expected(cpu, dtype)
        for r in range(R):
            assert_bits_equal(outs[r], want, dtype, "replay %d rank %d" % (rep, r))
    h.close()


@pytest.mark.parametrize("algo,transport", [(ar.AR_ONE_SHOT, ar.AR_LL_GLOBAL),
                                             (ar.AR_ONE_SHOT, ar.AR_LL_CLUSTER),
                                             (ar.AR_TWO_SHOT, ar.AR_LL_GLOBAL)],
                         ids=["one_shot_global", "one_shot_cluster", "two_shot"])
def test_ll_timeout_then_recovery(algo, transport):
    """A rank that never writes its packets: the peers' bounded polls give up,
    AR_ERR_TIMEOUT is reported, and the next normal call is correct."""
    need_gpu()
    R, n, dtype = 4, 10000, "bf16"
    cpu = wl.make_inputs(44, R, n, dtype, "uniform")
    ins = device_inputs(cpu)
    outs = [torch.empty_like(t) for t in ins]
    with ar.Handle(R, n, dtype) as h:
        ar.ar_set_ll_transport(h.h, transport)
        ar.ar_set_timeout(h.h, 20_000_000)      # 20 ms
        ar.ar_debug_drop_rank(h.h, 2)
        ar.ar_allreduce(h.h, ins, outs, algo, ar.AR_LL)
        assert ar.ar_status(h.h) == ar.AR_ERR_TIMEOUT
        ar.ar_debug_drop_rank(h.h, -1)
        ar.ar_allreduce(h.h, ins, outs, algo, ar.AR_LL)
        assert ar.ar_status(h.h) == ar.AR_OK
    want = expected(cpu, dtype)
    for r in range(R):
        assert_bits_equal(outs[r], want, dtype, "after recovery rank %d" % r)


def test_ll_rejected_above_cap():
    need_gpu()
    n = ar.AR_LL_MAX_BYTES // 2 + 1
    x = [torch.zeros(n, dtype=torch.bfloat16, device="cuda") for _ in range(2)]
    with ar.Handle(2, n, "bf16") as h:
        assert ar.ar_get_info(h.h)["ll_capable"] == 0
        with pytest.raises(ar.ArError) as e:
            ar.ar_allreduce(h.h, x, x, ar.AR_ONE_SHOT, ar.AR_LL)
        assert e.value.code == ar.AR_ERR_UNSUPPORTED
        ar.ar_allreduce(h.h, x, x, ar.AR_TWO_SHOT, ar.AR_HB)   # HB still serves it


@pytest.mark.parametrize("algo", [ar.AR_ONE_SHOT, ar.AR_TWO_SHOT], ids=["one_shot", "two_shot"])
def test_ll_at_the_cap(algo):
    """The largest message LL accepts: exactly AR_LL_MAX_BYTES per rank."""
    need_gpu()
    R, n = 2, ar.AR_LL_MAX_BYTES // 2
    run_case(R, n, "bf16", algo, ar.AR_LL, dist="normal", config=44)


def test_too_few_buffers_rejected():
    """The binding pads pointer arrays with NULL: fewer buffers than ranks is
    an argument error, never a read past the array."""
    need_gpu()
    R, n = 4, 1000
    ins = [torch.zeros(n, dtype=torch.bfloat16, device="cuda") for _ in range(R)]
    outs = [torch.empty_like(t) for t in ins]
    with ar.Handle(R, n, "bf16") as h:
        for a, b in [(ins[:3], outs), (ins, outs[:2]), ([], [])]:
            with pytest.raises(ar.ArError) as e:
                ar.ar_allreduce(h.h, a, b, ar.AR_TWO_SHOT, ar.AR_HB)
            assert e.value.code == ar.AR_ERR_INVALID
        with pytest.raises(ValueError):
            ar.ar_allreduce(h.h, ins * 9, outs, ar.AR_ONE_SHOT, ar.AR_HB)


def test_invalid_aliasing_rejected():
    need_gpu()
    R, n = 3, 100
    a = [torch.zeros(n, dtype=torch.bfloat16, device="cuda") for _ in range(R)]
    big = torch.zeros(3 * n, dtype=torch.bfloat16, device="cuda")
    with ar.Handle(R, n, "bf16") as h:
        # two outputs overlapping
        outs = [big[0:n], big[n // 2: n // 2 + n], big[2 * n:]]
        with pytest.raises(ar.ArError):
            ar.ar_allreduce(h.h, a, outs, ar.AR_ONE_SHOT, ar.AR_HB)
        # rank 0's input is rank 1's output
        with pytest.raises(ar.ArError):
            ar.ar_allreduce(h.h, [a[0], a[1], a[2]], [a[1], big[:n], big[n:2 * n]],
                            ar.AR_ONE_SHOT, ar.AR_HB)


@pytest.mark.parametrize("dtype", ["bf16", "fp16"])
def test_round_exhaustive_vs_oracle(dtype):
    """The kernels' rounding (cvt.rn) on all 2^32 binary32 patterns equals
    the oracle's definition-based rounding."""
    need_gpu()
    chunk = 1 << 28
    dst = torch.empty(chunk, dtype=wl.TORCH_DTYPE[dtype], device="cuda")
    for start in range(0, 1 << 32, chunk):
        pats = torch.arange(start, start + chunk, dtype=torch.int64, device="cuda")
        src = (pats - (1 << 32) * (pats >= (1 << 31)).long()).to(torch.int32).view(torch.float32)
        ar.ar_round(dtype, src, dst, chunk)
        got = wl.bits(dst.cpu())
        f = src.cpu().numpy()
        want = oracle.round_f32(f, wl.DTYPE_CODE[dtype])
        nan = np.isnan(f)
        assert np.array_equal(got[~nan], want[~nan]), "chunk at %#x" % start


@pytest.mark.parametrize("pdl", [1, 0], ids=["pdl", "no_pdl"])
@pytest.mark.parametrize("captured", [False, True], ids=["eager", "graph"])
def test_chained_calls_wait_for_their_inputs(pdl, captured):
    """Each call reads the previous call's outputs.  With programmatic
    dependent launch a kernel may start before the previous one ends; it
    must still see that kernel's results (it waits before reading)."""
    need_gpu()
    R, n, dtype = 8, 70001, "bf16"
    cpu = wl.make_inputs(45, R, n, dtype, "uniform")
    bufs = [device_inputs(cpu)] + [[torch.empty(n, dtype=torch.bfloat16, device="cuda")
                                    for _ in range(R)] for _ in range(len(ALL_PATHS))]
    for b in bufs[1:]:
        for t in b:
            t.fill_(float("nan"))
    h = ar.Handle(R, n, dtype)
    ar.ar_set_pdl(h.h, pdl)
    s = torch.cuda.Stream()

    def chain():
        for i, (algo, proto) in enumerate(ALL_PATHS):
            ar.ar_allreduce(h.h, bufs[i], bufs[i + 1], algo, proto, stream=s)

    with torch.cuda.stream(s):
        if captured:
            chain()                          # warm-up outside capture
            s.synchronize()
            for b in bufs[1:]:
                for t in b:
                    t.fill_(float("nan"))
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=s):
                chain()
            g.replay()
        else:
            chain()
    torch.cuda.synchronize()
    assert ar.ar_status(h.h) == ar.AR_OK
    h.close()
    want = [wl.bits(t) for t in cpu]
    for i in range(len(ALL_PATHS)):
        want = [oracle.allreduce(want, wl.DTYPE_CODE[dtype])[0]] * R
        for r in range(R):
            assert_bits_equal(bufs[i + 1][r], want[0], dtype, "step %d rank %d" % (i, r))


@pytest.mark.parametrize("path", ALL_PATHS, ids=PATH_IDS)
@pytest.mark.parametrize("n", [9, 4097, (1 << 20) + 5])
def test_parity_without_pdl(path, n):
    need_gpu()
    R, dtype = 8, "fp16"
    cpu = wl.make_inputs(46, R, n, dtype, "normal")
    ins = device_inputs(cpu)
    outs = [torch.empty_like(t) for t in ins]
    with ar.Handle(R, n, dtype) as h:
        ar.ar_set_pdl(h.h, 0)
        assert ar.ar_get_info(h.h)["pdl"] == 0
        ar.ar_allreduce(h.h, ins, outs, *path)
        assert ar.ar_status(h.h) == ar.AR_OK
    want = expected(cpu, dtype)
    for r in range(R):
        assert_bits_equal(outs[r], want, dtype, "rank %d" % r)
