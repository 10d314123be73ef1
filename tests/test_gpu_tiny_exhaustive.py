"""Every tiny message on every path: N = 1..67 elements per rank for every
R in 1..32 and every dtype, through one-shot/two-shot x HB/LL, checked bit
for bit against the oracle with canary zones on both sides of each output.
These sizes cover every split of a message into whole 16-byte vectors, LL
packet pairs, single packets and element tails, and every shard layout of
the two-shot schedule with empty and short shards.  Each size runs with
every buffer 16-byte aligned, 8-byte aligned only (the staged LL kernels,
element-wise HB) and element aligned only (the per-rank LL kernel)."""
import numpy as np
import pytest
import torch

import all_reduce_reduction_gb300 as ar
import oracle
from all_reduce_reduction_gb300 import workload as wl
from gpu_helpers import ALL_PATHS, GUARD, UINT_T, canary_value, device_inputs, need_gpu

pytestmark = pytest.mark.gpu

NMAX = 67
# each rank's output row: GUARD canaries, a 72-element slot (a whole number of
# 16-byte vectors, so every row starts 16-byte aligned), GUARD canaries
ROW = GUARD + 72 + GUARD
# byte offset of every input and output from a 16-byte boundary (None: one
# element)
ALIGNMENTS = {"a16": 0, "a8": 8, "elem": None}


@pytest.mark.parametrize("align", list(ALIGNMENTS))
@pytest.mark.parametrize("dtype", ["bf16", "fp16", "fp32"])
def test_every_tiny_size_every_rank_count(dtype, align):
    need_gpu()
    u = np.uint32 if dtype == "fp32" else np.uint16
    cv = canary_value(dtype)
    failures = []
    for R in range(1, 33):
        cpu = wl.make_inputs(120 + R, R, NMAX, dtype, "loguniform")
        # the fold is elementwise: the result for a prefix of n elements is the
        # prefix of the result for all NMAX elements
        want = np.ascontiguousarray(oracle.allreduce([wl.bits(t) for t in cpu],
                                                     wl.DTYPE_CODE[dtype])[0]).view(u)
        esz = wl.ELEM_SIZE[dtype]
        off = 1 if ALIGNMENTS[align] is None else ALIGNMENTS[align] // esz
        ins = device_inputs(cpu, off)
        block = torch.empty((R, ROW), dtype=wl.TORCH_DTYPE[dtype], device="cuda")
        outs = [block[r, GUARD + off:GUARD + off + NMAX] for r in range(R)]
        want_align = {"a16": 16, "a8": 8, "elem": esz}[align]
        for t in ins + outs:
            assert t.data_ptr() % want_align == 0
            assert want_align == 16 or t.data_ptr() % (2 * want_align) != 0
        with ar.Handle(R, NMAX, dtype) as h:
            for n in range(1, NMAX + 1):
                for algo, proto in ALL_PATHS:
                    block.view(UINT_T[dtype]).fill_(cv)
                    ar.ar_allreduce_n(h.h, ins, outs, n, algo, proto)
                    got = block.view(UINT_T[dtype]).cpu().numpy().view(u)
                    st = ar.ar_status(h.h)
                    if st != ar.AR_OK:
                        failures.append((R, n, algo, proto, "status " + ar.ar_strerror(st)))
                        continue
                    canary = np.array(cv, dtype=np.int64).astype(u)
                    body = got[:, GUARD + off:GUARD + off + n]
                    if not (body == want[:n]).all():
                        r, i = np.argwhere(body != want[:n])[0]
                        failures.append((R, n, algo, proto, "rank %d element %d" % (r, i)))
                    if not ((got[:, :GUARD + off] == canary).all()
                            and (got[:, GUARD + off + n:] == canary).all()):
                        failures.append((R, n, algo, proto, "write outside the message"))
    assert not failures, "%d failures, first: %s" % (len(failures), failures[:5])
