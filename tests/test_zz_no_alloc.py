"""ar_allreduce_ll_static: the one-shot LL all-reduce for callers that cannot
allocate device memory where they run it (an engine that has reserved all of
the GPU's memory for its own pool, or a hook on a latency-critical path that
must not pay the device-wide synchronisation cudaMalloc and cudaFree can
imply).  Its packet scratch is the library's static device array.

Every case makes two calls in a row, with new inputs each time, and checks
both against the CPU oracle and against the handle-based one-shot LL call
(ar_allreduce), bit for bit: the tolerance of every parity test here.  The
cases cover 8-byte-aligned buffers (the staged kernel), buffers one element
off that alignment (the per-rank kernel), in place, and a message whose
packets fill the static scratch exactly.

This file is collected last on purpose: if it fails, a run that stops at the
first failure has already run every other test."""
import pytest
import torch

import all_reduce_reduction_gb300 as ar
from all_reduce_reduction_gb300 import workload as wl
from gpu_helpers import (assert_bits_equal, check_guards, device_inputs, expected,
                         guarded_outputs, need_gpu)

pytestmark = pytest.mark.gpu


def static_packet_bytes(R: int, n: int, dtype: str) -> int:
    """Packet scratch a call needs, as the library sizes it: R slots of
    ceil(n * elem_size / 4) packets, rounded up to a multiple of 4, 8 bytes
    each."""
    packets = -(-(n * wl.ELEM_SIZE[dtype]) // 4)
    return R * (-(-packets // 4) * 4) * 8


def limit_n(R: int, dtype: str) -> int:
    """Elements per rank whose packets fill the static scratch exactly."""
    return ar.AR_NOALLOC_SCRATCH_BYTES // (R * 8) * 4 // wl.ELEM_SIZE[dtype]


def test_limit_helpers_mirror_the_library():
    for dtype in ("bf16", "fp16", "fp32"):
        n = limit_n(8, dtype)
        assert static_packet_bytes(8, n, dtype) == ar.AR_NOALLOC_SCRATCH_BYTES
        assert static_packet_bytes(8, n + 1, dtype) > ar.AR_NOALLOC_SCRATCH_BYTES
    assert limit_n(8, "bf16") == 1 << 18          # the largest size of the LL sweep


CASES = [  # (R, n, element offset, in place)
    (8, 512, 0, False),
    (8, "limit", 0, False),
    (3, 1001, 0, False),
    (32, 4097, 0, False),
    (8, 4097, 1, False),
    (5, 1001, 1, True),
    (8, "limit", 1, False),
]


@pytest.mark.parametrize("dtype", ["bf16", "fp16", "fp32"])
@pytest.mark.parametrize("R,n,offset,inplace", CASES,
                         ids=["r8_n512", "r8_at_limit", "r3_n1001", "r32_n4097",
                              "r8_n4097_offset", "r5_n1001_offset_inplace",
                              "r8_at_limit_offset"])
def test_static_scratch_two_calls_match_oracle_and_handle_path(dtype, R, n, offset, inplace):
    need_gpu()
    if n == "limit":
        n = limit_n(R, dtype)
    assert static_packet_bytes(R, n, dtype) <= ar.AR_NOALLOC_SCRATCH_BYTES
    outs_ref = [torch.empty(n, dtype=wl.TORCH_DTYPE[dtype], device="cuda") for _ in range(R)]
    with ar.Handle(R, n, dtype) as h:
        for call in range(2):           # two calls in a row, new inputs each time
            cpu = wl.make_inputs(60 + call, R, n, dtype, "loguniform")
            want = expected(cpu, dtype)
            ref_ins = [t.cuda() for t in cpu]
            ar.ar_allreduce(h.h, ref_ins, outs_ref, ar.AR_ONE_SHOT, ar.AR_LL)
            ins = device_inputs(cpu, offset)
            if inplace:
                bufs, outs = None, ins
            else:
                bufs, outs = guarded_outputs(R, n, dtype, offset)
            ar.ar_allreduce_ll_static(R, n, dtype, ins, outs)
            torch.cuda.synchronize()
            assert ar.ar_status(h.h) == ar.AR_OK
            for r in range(R):
                what = "call %d rank %d" % (call, r)
                assert_bits_equal(outs[r], want, dtype, what + " vs the oracle")
                assert_bits_equal(outs[r], wl.bits(outs_ref[r].cpu()), dtype,
                                  what + " vs ar_allreduce")
            if bufs is not None:
                check_guards(bufs, n, dtype, offset)


@pytest.mark.parametrize("dtype", ["bf16", "fp32"])
def test_static_scratch_rejects_one_element_past_the_limit(dtype):
    need_gpu()
    R = 8
    n = limit_n(R, dtype) + 1
    x = [torch.zeros(n, dtype=wl.TORCH_DTYPE[dtype], device="cuda") for _ in range(R)]
    y = [torch.zeros_like(t) for t in x]
    with pytest.raises(ar.ArError) as e:
        ar.ar_allreduce_ll_static(R, n, dtype, x, y)
    assert e.value.code == ar.AR_ERR_UNSUPPORTED
