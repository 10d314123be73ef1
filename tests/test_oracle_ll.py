"""Pins for the oracle's LL packet encode/decode.

The packet layout is a reading (the pages name the LL protocol but print no
layout); the hand-derived packets in tests/golden/ll_packets.json fix it, and
the round trip and flag checks pin the decode side.
"""
import numpy as np
import pytest

import oracle
from all_reduce_reduction_gb300 import workload as wl
from _util import DT_CODE, as_uint, golden, hex_array

DTYPES = ["bf16", "fp16", "fp32"]


@pytest.mark.parametrize("case", golden("ll_packets.json")["cases"], ids=lambda c: c["name"])
def test_golden_packets(case):
    dt = case["dtype"]
    x = hex_array(case["elements"], dt)
    flag = int(case["flag"], 16)
    pk = oracle.ll_pack(x, DT_CODE[dt], flag)
    assert [hex(int(p)) for p in pk] == [hex(int(h, 16)) for h in case["packets"]]
    back, bad = oracle.ll_unpack(pk, DT_CODE[dt], x.size, flag)
    assert bad == 0 and np.array_equal(as_uint(back, dt), as_uint(x, dt))


@pytest.mark.parametrize("dtype", DTYPES)
@pytest.mark.parametrize("n", list(range(1, 68)) + [4097 * 4096 // 1024 + 3])
def test_round_trip(dtype, n):
    x = wl.bits(wl.make_inputs(97, 1, n, dtype, "loguniform")[0])
    flag = 0x9E37_79B9 ^ n
    pk = oracle.ll_pack(x, DT_CODE[dtype], flag)
    assert pk.size == -(-n * wl.ELEM_SIZE[dtype] // 4)
    assert np.all((pk >> np.uint64(32)) == flag)
    back, bad = oracle.ll_unpack(pk, DT_CODE[dtype], n, flag)
    assert bad == 0
    assert np.array_equal(as_uint(back, dtype), as_uint(x, dtype))
    # payloads are the message bytes in order, zero padded
    raw = np.zeros(pk.size * 4, dtype=np.uint8)
    raw[: n * wl.ELEM_SIZE[dtype]] = np.ascontiguousarray(x).view(np.uint8)
    assert np.array_equal((pk & np.uint64(0xFFFFFFFF)).astype(np.uint32), raw.view("<u4"))


@pytest.mark.parametrize("dtype", DTYPES)
def test_wrong_flag_is_reported_and_not_written(dtype):
    n = 37
    x = wl.bits(wl.make_inputs(98, 1, n, dtype, "normal")[0])
    pk = oracle.ll_pack(x, DT_CODE[dtype], 5)
    dst = np.zeros(n, dtype=x.dtype)
    _, bad = oracle.ll_unpack(pk, DT_CODE[dtype], n, 6, dst=dst)
    assert bad == pk.size
    assert np.all(as_uint(dst, dtype) == 0)
    # a stale packet in the middle: only its bytes stay unwritten
    pk2 = pk.copy()
    pk2[3] = (pk2[3] & np.uint64(0xFFFFFFFF)) | (np.uint64(4) << np.uint64(32))
    dst = np.zeros(n, dtype=x.dtype)
    _, bad = oracle.ll_unpack(pk2, DT_CODE[dtype], n, 5, dst=dst)
    assert bad == 1
    got = np.ascontiguousarray(dst).view(np.uint8)
    want = np.ascontiguousarray(x).view(np.uint8).copy()
    want[12:16] = 0
    assert np.array_equal(got, want)
