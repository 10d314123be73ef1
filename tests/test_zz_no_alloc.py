"""ar_allreduce_ll_static: the all-reduce for callers that cannot allocate
device memory where they run it (an engine's plugin hook during graph
capture, or an engine that owns every byte of device memory).  It must give
the same bits as the handle-based one-shot LL call, call after call, with
its scratch in the library's static device array.

This file is collected last on purpose: if it fails, a run that stops at the
first failure has already run every other test."""
import pytest
import torch

import all_reduce_reduction_gb300 as ar
from all_reduce_reduction_gb300 import workload as wl
from gpu_helpers import assert_bits_equal, need_gpu

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("dtype", ["bf16", "fp16", "fp32"])
@pytest.mark.parametrize("R,n", [(8, 512), (8, 1 << 18), (3, 1001), (32, 4097)])
def test_static_scratch_matches_handle_path_two_calls(dtype, R, n):
    need_gpu()
    if R * ((n * wl.ELEM_SIZE[dtype] + 3) // 4 + 3) // 4 * 32 > ar.AR_NOALLOC_SCRATCH_BYTES:
        pytest.skip("beyond the static scratch")
    outs_ref = [torch.empty(n, dtype=wl.TORCH_DTYPE[dtype], device="cuda") for _ in range(R)]
    outs = [torch.empty_like(o) for o in outs_ref]
    with ar.Handle(R, n, dtype) as h:
        for call in range(2):           # two calls in a row, new inputs each time
            cpu = wl.make_inputs(60 + call, R, n, dtype, "loguniform")
            ins = [t.cuda() for t in cpu]
            for o in outs:
                o.fill_(float("nan"))
            ar.ar_allreduce(h.h, ins, outs_ref, ar.AR_ONE_SHOT, ar.AR_LL)
            ar.ar_allreduce_ll_static(R, n, dtype, ins, outs)
            torch.cuda.synchronize()
            assert ar.ar_status(h.h) == ar.AR_OK
            for r in range(R):
                assert_bits_equal(outs[r], wl.bits(outs_ref[r].cpu()), dtype,
                                  "call %d rank %d" % (call, r))


def test_static_scratch_rejects_too_large():
    need_gpu()
    R = 8
    n = ar.AR_NOALLOC_SCRATCH_BYTES // (2 * R) + 8      # > 512 KiB of bf16 per rank
    x = [torch.zeros(n, dtype=torch.bfloat16, device="cuda") for _ in range(R)]
    with pytest.raises(ar.ArError) as e:
        ar.ar_allreduce_ll_static(R, n, "bf16", x, x)
    assert e.value.code == ar.AR_ERR_UNSUPPORTED
