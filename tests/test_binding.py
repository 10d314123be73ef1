"""The Python binding's argument marshalling, on the CPU: pointer arrays,
plan steps and errors (no device call)."""
import ctypes

import pytest

import all_reduce_reduction_gb300 as ar


class FakeTensor:
    def __init__(self, ptr):
        self.ptr = ptr

    def data_ptr(self):
        return self.ptr


def test_pointer_array_is_padded_with_nulls():
    arr = ar._ptr_array([FakeTensor(0x1000), 0x2000, None])
    assert len(arr) == ar.AR_MAX_RANKS
    assert [arr[i] for i in range(3)] == [0x1000, 0x2000, None]
    assert all(arr[i] is None for i in range(3, ar.AR_MAX_RANKS))   # NULL
    full = ar._ptr_array([FakeTensor(16 * (i + 1)) for i in range(ar.AR_MAX_RANKS)])
    assert [full[i] for i in range(ar.AR_MAX_RANKS)] == [16 * (i + 1)
                                                          for i in range(ar.AR_MAX_RANKS)]
    with pytest.raises(ValueError):
        ar._ptr_array([0x10] * (ar.AR_MAX_RANKS + 1))


def test_stream_handles():
    assert ar._stream(0) == 0
    assert ar._stream(0xABC) == 0xABC

    class S:
        cuda_stream = 0x1234
    assert ar._stream(S()) == 0x1234


def test_make_op_fields():
    o = ar.make_op(ar.AR_OP_REDUCE, 3, (ar.AR_BUF_OUT, 2),
                   [(ar.AR_BUF_IN, 5), (ar.AR_BUF_IN, 0), (ar.AR_BUF_IN, 7)], 4, 9)
    assert (o.kind, o.rank, o.dst_buf, o.dst_rank) == (ar.AR_OP_REDUCE, 3, ar.AR_BUF_OUT, 2)
    assert (o.src_buf, o.nsrc) == (ar.AR_BUF_IN, 3)
    assert list(o.src_rank)[:3] == [5, 0, 7] and not any(list(o.src_rank)[3:])
    assert (o.chunk_begin, o.chunk_end) == (4, 9)
    with pytest.raises(ValueError):
        ar.make_op(ar.AR_OP_REDUCE, 0, (ar.AR_BUF_OUT, 0),
                   [(ar.AR_BUF_IN, 0), (ar.AR_BUF_OUT, 1)], 0, 1)
    # a step array as the library receives it
    arr = (ar.ar_op * 2)(o, o)
    assert ctypes.sizeof(arr) == 2 * ctypes.sizeof(ar.ar_op)


def test_error_carries_its_code():
    e = ar.ArError(ar.AR_ERR_UNSUPPORTED, "ar_allreduce")
    assert e.code == ar.AR_ERR_UNSUPPORTED
    assert str(e).startswith("ar_allreduce: AR_ERR_UNSUPPORTED")


def _header_constants():
    import os
    import re
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    text = open(os.path.join(root, "include", "ar.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    consts = {}
    for body in re.findall(r"enum\s+\w+\s*\{(.*?)\}", text, re.S):
        for name, value in re.findall(r"(AR_\w+)\s*=\s*(\d+)", body):
            consts[name] = int(value)
    for name, expr in re.findall(r"^#define\s+(AR_\w+)\s+(.+)$", text, re.M):
        expr = re.sub(r"(\d+)u?l?l?", r"\1", expr.strip())
        if re.fullmatch(r"[\d\s()<]+", expr):
            consts[name] = eval(expr)                 # digits, shifts, parentheses only
    return consts


def test_binding_constants_match_the_header():
    consts = _header_constants()
    assert {"AR_MAX_RANKS", "AR_LL_MAX_BYTES", "AR_NOALLOC_SCRATCH_BYTES", "AR_OK",
            "AR_ERR_FLAG_MISMATCH", "AR_LL_CLUSTER", "AR_BUF_OUT"} <= set(consts)
    for name, value in consts.items():
        if hasattr(ar, name):
            assert getattr(ar, name) == value, name
    # every enumerator the calls take or return is exposed by the binding
    for name in consts:
        if name.startswith(("AR_ERR_", "AR_OK", "AR_BF16", "AR_FP", "AR_ONE", "AR_TWO",
                            "AR_ALGO", "AR_PROTO", "AR_LL", "AR_HB", "AR_OP_", "AR_BUF_")):
            if name != "AR_LL_MAX_BYTES":
                assert hasattr(ar, name), name
