"""Several handles in flight at once, and handle life cycles.

Two tensor-parallel groups on one GPU would run their all-reduces on two
streams with no ordering between them: each handle has its own scratch,
epoch and status words, and the LL kernels are cooperative launches, so
concurrent calls must neither mix data nor time out."""
import pytest
import torch

import all_reduce_reduction_gb300 as ar
from all_reduce_reduction_gb300 import workload as wl
from gpu_helpers import ALL_PATHS, PATH_IDS, assert_bits_equal, expected, need_gpu

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("path", ALL_PATHS, ids=PATH_IDS)
def test_two_handles_on_two_streams(path):
    need_gpu()
    R, n, dtype = 8, (1 << 18) + 3, "bf16"
    groups = []
    for g in range(2):
        cpu = wl.make_inputs(100 + g, R, n, dtype, "uniform")
        ins = [t.cuda() for t in cpu]
        outs = [torch.empty_like(t) for t in ins]
        groups.append((ar.Handle(R, n, dtype), torch.cuda.Stream(), cpu, ins, outs))
    torch.cuda.synchronize()
    for _ in range(20):                       # interleaved, never synchronised in between
        for h, s, _, ins, outs in groups:
            ar.ar_allreduce(h.h, ins, outs, *path, stream=s)
    torch.cuda.synchronize()
    for h, s, cpu, ins, outs in groups:
        assert ar.ar_status(h.h, s) == ar.AR_OK
        want = expected(cpu, dtype)
        for r in range(R):
            assert_bits_equal(outs[r], want, dtype, "rank %d" % r)
        h.close()


def test_create_destroy_does_not_leak():
    need_gpu()
    torch.cuda.synchronize()
    free0, _ = torch.cuda.mem_get_info()
    for i in range(50):
        with ar.Handle(32, (1 << 20) + i, "fp32") as h:      # ~270 MB of LL scratch each
            assert ar.ar_get_info(h.h)["ll_capable"] == 1
    torch.cuda.synchronize()
    free1, _ = torch.cuda.mem_get_info()
    assert free0 - free1 < (64 << 20)


def test_handle_survives_many_calls_and_epoch_wrap_region():
    """A few thousand LL calls in graphs: the device epoch keeps advancing and
    every replay stays exact."""
    need_gpu()
    R, n = 4, 4096
    cpu = wl.make_inputs(102, R, n, "fp16", "normal")
    ins = [t.cuda() for t in cpu]
    outs = [torch.empty_like(t) for t in ins]
    h = ar.Handle(R, n, "fp16")
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        ar.ar_allreduce(h.h, ins, outs, ar.AR_TWO_SHOT, ar.AR_LL, stream=s)
    s.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        for _ in range(100):
            ar.ar_allreduce(h.h, ins, outs, ar.AR_ONE_SHOT, ar.AR_LL, stream=s)
            ar.ar_allreduce(h.h, ins, outs, ar.AR_TWO_SHOT, ar.AR_LL, stream=s)
    for _ in range(20):
        g.replay()
    torch.cuda.synchronize()
    assert ar.ar_status(h.h) == ar.AR_OK
    want = expected(cpu, "fp16")
    for r in range(R):
        assert_bits_equal(outs[r], want, "fp16", "rank %d" % r)
    h.close()
