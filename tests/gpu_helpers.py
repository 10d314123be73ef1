"""Helpers for the GPU parity tests: seeded inputs, guarded output buffers,
and element-by-element comparison with the CPU oracle."""
from __future__ import annotations

import numpy as np
import pytest
import torch

import all_reduce_reduction_gb300 as ar
import oracle
from all_reduce_reduction_gb300 import workload as wl

GUARD = 64          # elements of canary before and after every output
CANARY = {"bf16": 0x7FA5, "fp16": 0x7E5A, "fp32": 0x7FA5A5A5}
UINT_T = {"bf16": torch.int16, "fp16": torch.int16, "fp32": torch.int32}

ALL_PATHS = [(ar.AR_ONE_SHOT, ar.AR_HB), (ar.AR_TWO_SHOT, ar.AR_HB),
             (ar.AR_ONE_SHOT, ar.AR_LL), (ar.AR_TWO_SHOT, ar.AR_LL)]
PATH_IDS = ["one_shot_hb", "two_shot_hb", "one_shot_ll", "two_shot_ll"]


def need_gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")


def canary_value(dtype: str) -> int:
    v = CANARY[dtype]
    return v - (1 << 16) if dtype != "fp32" and v >= 1 << 15 else v


def guarded_outputs(R: int, n: int, dtype: str, offset: int = 0):
    """R output views of n elements inside buffers whose GUARD elements
    before and after hold a canary pattern.  `offset` extra elements shift
    the view off 16-byte alignment."""
    bufs, views = [], []
    for _ in range(R):
        b = torch.empty(GUARD + offset + n + GUARD, dtype=wl.TORCH_DTYPE[dtype], device="cuda")
        b.view(UINT_T[dtype]).fill_(canary_value(dtype))
        bufs.append(b)
        views.append(b[GUARD + offset: GUARD + offset + n])
    return bufs, views


def check_guards(bufs, n: int, dtype: str, offset: int = 0):
    for b in bufs:
        u = b.view(UINT_T[dtype])
        head = u[: GUARD + offset]
        tail = u[GUARD + offset + n:]
        cv = canary_value(dtype)
        assert bool((head == cv).all()) and bool((tail == cv).all()), "write outside the output"


def device_inputs(cpu_inputs, offset: int = 0):
    """Copy CPU inputs to the device, optionally at an element offset."""
    outs = []
    for t in cpu_inputs:
        b = torch.empty(offset + t.numel() + 8, dtype=t.dtype, device="cuda")
        v = b[offset: offset + t.numel()]
        v.copy_(t)
        outs.append(v)
    return outs


def expected(cpu_inputs, dtype: str) -> np.ndarray:
    return oracle.allreduce([wl.bits(t) for t in cpu_inputs], wl.DTYPE_CODE[dtype])[0]


def assert_bits_equal(got_t: torch.Tensor, want: np.ndarray, dtype: str, what: str):
    got = wl.bits(got_t.cpu())
    gu = got.view(np.uint32 if dtype == "fp32" else np.uint16)
    wu = np.ascontiguousarray(want).view(np.uint32 if dtype == "fp32" else np.uint16)
    if not np.array_equal(gu, wu):
        bad = np.nonzero(gu != wu)[0]
        i = int(bad[0])
        raise AssertionError("%s: %d of %d elements differ; first at %d: got %#x want %#x"
                             % (what, bad.size, gu.size, i, int(gu[i]), int(wu[i])))
