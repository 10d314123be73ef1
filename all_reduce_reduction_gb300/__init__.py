"""GB300-native sum all-reduce over R virtual ranks held in one GPU's HBM.

This module is a thin ctypes binding of the C ABI declared in
``include/ar.h`` (library ``libar_gb300.so``, built in-tree by
``all_reduce_reduction_gb300.build``).  Every function has the name of the C
entry point it calls and only marshals arguments: device buffers may be given
as integers (device addresses) or as objects with ``data_ptr()`` (torch CUDA
tensors); a stream as an integer ``cudaStream_t``, an object with
``cuda_stream`` (``torch.cuda.Stream``), or ``None`` for torch's current
stream.  All work runs in the library's CUDA kernels; there is no CPU path.
If the library is missing, the first call raises ``RuntimeError``.
"""
from __future__ import annotations

import ctypes
import os
import threading

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "libar_gb300.so")

# enum ar_dtype / ar_algo / ar_proto / ar_status_code (include/ar.h)
AR_BF16, AR_FP16, AR_FP32 = 0, 1, 2
AR_ONE_SHOT, AR_TWO_SHOT, AR_ALGO_AUTO = 0, 1, 2
AR_LL, AR_HB, AR_PROTO_AUTO = 0, 1, 2
AR_OK = 0
AR_ERR_INVALID = 1
AR_ERR_UNSUPPORTED = 2
AR_ERR_CUDA = 3
AR_ERR_NOMEM = 4
AR_ERR_TIMEOUT = 5
AR_ERR_FLAG_MISMATCH = 6
AR_LL_AUTO, AR_LL_GLOBAL, AR_LL_CLUSTER = 0, 1, 2
AR_HB_STAGING_AUTO, AR_HB_STAGING_TMA, AR_HB_STAGING_DIRECT = 0, 1, 2
AR_MAX_RANKS = 32
AR_LL_MAX_BYTES = 64 << 20

DTYPES = {"bf16": AR_BF16, "fp16": AR_FP16, "fp32": AR_FP32}
ALGOS = {"one_shot": AR_ONE_SHOT, "two_shot": AR_TWO_SHOT, "auto": AR_ALGO_AUTO}
PROTOS = {"ll": AR_LL, "hb": AR_HB, "auto": AR_PROTO_AUTO}


class ArError(RuntimeError):
    """A nonzero ar_status_code returned by the library."""

    def __init__(self, code: int, where: str):
        self.code = code
        super().__init__("%s: %s" % (where, ar_strerror(code)))


class ar_info(ctypes.Structure):
    _fields_ = [
        ("R", ctypes.c_int),
        ("dtype", ctypes.c_int),
        ("N", ctypes.c_size_t),
        ("elem_size", ctypes.c_size_t),
        ("ll_capable", ctypes.c_int),
        ("ll_packets_per_rank", ctypes.c_size_t),
        ("scratch_bytes", ctypes.c_size_t),
        ("num_sms", ctypes.c_int),
        ("ll_ctas_per_rank_max", ctypes.c_int),
        ("tma_tile_bytes", ctypes.c_int),
        ("tma_stages", ctypes.c_int),
        ("timeout_ns", ctypes.c_uint64),
        ("ll_transport", ctypes.c_int),
        ("ll_cluster_ok", ctypes.c_int),
        ("ll_cluster_units", ctypes.c_int),
        ("ll_cluster_max", ctypes.c_int),
        ("pdl", ctypes.c_int),
        ("ll_staged_ctas_max", ctypes.c_int),
        ("hb_staging", ctypes.c_int),
    ]

    def as_dict(self) -> dict:
        return {name: getattr(self, name) for name, _ in self._fields_}


AR_OP_COPY, AR_OP_REDUCE = 0, 1
AR_BUF_IN, AR_BUF_OUT = 0, 1


class ar_op(ctypes.Structure):
    _fields_ = [
        ("kind", ctypes.c_int),
        ("rank", ctypes.c_int),
        ("dst_buf", ctypes.c_int),
        ("dst_rank", ctypes.c_int),
        ("src_buf", ctypes.c_int),
        ("nsrc", ctypes.c_int),
        ("src_rank", ctypes.c_int * AR_MAX_RANKS),
        ("chunk_begin", ctypes.c_int),
        ("chunk_end", ctypes.c_int),
    ]


_lock = threading.Lock()
_lib = None

# exported entry points: name -> (argtypes, restype)
_VP, _SZ, _I, _U32, _U64 = ctypes.c_void_p, ctypes.c_size_t, ctypes.c_int, ctypes.c_uint32, ctypes.c_uint64
_VPP = ctypes.POINTER(ctypes.c_void_p)
SIGNATURES = {
    "ar_create": ([_I, _SZ, _I, ctypes.POINTER(_VP)], _I),
    "ar_destroy": ([_VP], _I),
    "ar_allreduce": ([_VP, _VPP, _VPP, _I, _I, _VP], _I),
    "ar_allreduce_n": ([_VP, _VPP, _VPP, _SZ, _I, _I, _VP], _I),
    "ar_allreduce_host": ([_VP, _VPP, _VPP, _SZ, _I, _I, _VP], _I),
    "ar_tune": ([_VP, _VP], _I),
    "ar_combine": ([_VP, _VPP, _VP, _VP, _SZ, _SZ, _VP], _I),
    "ar_get_tuning": ([_VP, _SZ, ctypes.POINTER(_I), ctypes.POINTER(_I),
                       ctypes.POINTER(ctypes.c_float)], _I),
    "ar_reduce_scatter": ([_VP, _VPP, _VPP, _VP], _I),
    "ar_all_gather": ([_VP, _VPP, _VP], _I),
    "ar_ll_pack": ([_VP, _VP, _VP, _SZ, _U32, _VP], _I),
    "ar_ll_unpack": ([_VP, _VP, _VP, _SZ, _U32, _VP], _I),
    "ar_status": ([_VP, _VP], _I),
    "ar_set_timeout": ([_VP, _U64], _I),
    "ar_debug_drop_rank": ([_VP, _I], _I),
    "ar_set_ll_transport": ([_VP, _I], _I),
    "ar_set_hb_staging": ([_VP, _I], _I),
    "ar_get_hb_staging": ([_VP, _SZ, ctypes.POINTER(_I)], _I),
    "ar_set_grid_divisor": ([_VP, _I], _I),
    "ar_get_grid_divisor": ([_VP, _SZ, _I, _I, ctypes.POINTER(_I)], _I),
    "ar_set_pdl": ([_VP, _I], _I),
    "ar_round": ([_I, _VP, _VP, _SZ, _VP], _I),
    "ar_get_info": ([_VP, ctypes.POINTER(ar_info)], _I),
    "ar_strerror": ([_I], ctypes.c_char_p),
    "ar_allreduce_ll_static": ([_I, _SZ, _I, _VPP, _VPP, _VP], _I),
    "ar_plan_compile": ([_VP, ctypes.POINTER(ar_op), _I, _I, _I, ctypes.POINTER(_VP)], _I),
    "ar_plan_builtin": ([_VP, _I, _I, _I, ctypes.POINTER(_VP)], _I),
    "ar_plan_execute": ([_VP, _VPP, _VPP, _VP], _I),
    "ar_plan_stats": ([_VP, ctypes.POINTER(_I), ctypes.POINTER(_I), ctypes.POINTER(_I)], _I),
    "ar_plan_destroy": ([_VP], _I),
}


def load_library(path: str = LIB_PATH) -> ctypes.CDLL:
    """Load the CUDA library (no GPU call is made).  Raises if it is absent."""
    global _lib
    with _lock:
        if _lib is not None and path == LIB_PATH:
            return _lib
        if not os.path.exists(path):
            raise RuntimeError(
                "libar_gb300.so is not built (expected at %s); run "
                "`python -c 'import __graft_entry__ as g; g.build()'`" % path)
        lib = ctypes.CDLL(path)
        for name, (args, res) in SIGNATURES.items():
            fn = getattr(lib, name)
            fn.argtypes, fn.restype = args, res
        if path == LIB_PATH:
            _lib = lib
        return lib


def _ptr(x) -> int:
    if x is None:
        return 0
    if isinstance(x, int):
        return x
    return int(x.data_ptr())


def _stream(s) -> int:
    if s is None:
        import torch
        return int(torch.cuda.current_stream().cuda_stream)
    if isinstance(s, int):
        return s
    return int(s.cuda_stream)


def _ptr_array(bufs):
    """Host array of device pointers, always AR_MAX_RANKS long: entries past
    the given buffers are NULL, so passing fewer buffers than the handle's
    ranks is rejected by the library (AR_ERR_INVALID) instead of reading past
    the end of the array."""
    if len(bufs) > AR_MAX_RANKS:
        raise ValueError("at most %d buffers" % AR_MAX_RANKS)
    arr = (ctypes.c_void_p * AR_MAX_RANKS)()
    for i, b in enumerate(bufs):
        arr[i] = _ptr(b)
    return arr


def _check(code: int, where: str) -> None:
    if code != AR_OK:
        raise ArError(code, where)


def ar_strerror(code: int) -> str:
    return load_library().ar_strerror(code).decode()


def ar_create(R: int, N: int, dtype) -> int:
    """Create a handle for R ranks of N elements; returns it as an integer."""
    dt = DTYPES[dtype] if isinstance(dtype, str) else dtype
    h = ctypes.c_void_p()
    _check(load_library().ar_create(R, N, dt, ctypes.byref(h)), "ar_create")
    return h.value


def ar_destroy(h: int) -> None:
    _check(load_library().ar_destroy(h), "ar_destroy")


def ar_allreduce(h: int, ins, outs, algo=AR_ONE_SHOT, proto=AR_HB, stream=None) -> None:
    algo = ALGOS[algo] if isinstance(algo, str) else algo
    proto = PROTOS[proto] if isinstance(proto, str) else proto
    _check(load_library().ar_allreduce(h, _ptr_array(ins), _ptr_array(outs), algo, proto,
                                       _stream(stream)), "ar_allreduce")


def ar_allreduce_n(h: int, ins, outs, n: int, algo=AR_ALGO_AUTO, proto=AR_PROTO_AUTO,
                   stream=None) -> None:
    algo = ALGOS[algo] if isinstance(algo, str) else algo
    proto = PROTOS[proto] if isinstance(proto, str) else proto
    _check(load_library().ar_allreduce_n(h, _ptr_array(ins), _ptr_array(outs), n, algo, proto,
                                         _stream(stream)), "ar_allreduce_n")


def ar_allreduce_host(h: int, ins, outs, n: int, algo=AR_ALGO_AUTO, proto=AR_PROTO_AUTO,
                      stream=None) -> None:
    algo = ALGOS[algo] if isinstance(algo, str) else algo
    proto = PROTOS[proto] if isinstance(proto, str) else proto
    _check(load_library().ar_allreduce_host(h, _ptr_array(ins), _ptr_array(outs), n, algo, proto,
                                            _stream(stream)), "ar_allreduce_host")


def ar_combine(h: int, ys, w, out, T: int, H: int, stream=None) -> None:
    _check(load_library().ar_combine(h, _ptr_array(ys), _ptr(w), _ptr(out), T, H,
                                      _stream(stream)), "ar_combine")


def ar_tune(h: int, stream=None) -> None:
    _check(load_library().ar_tune(h, _stream(stream)), "ar_tune")


def ar_get_tuning(h: int, nbytes: int):
    """(algo, proto, [µs one-shot LL, one-shot HB, two-shot LL, two-shot HB])."""
    a, p = ctypes.c_int(), ctypes.c_int()
    us = (ctypes.c_float * 4)()
    _check(load_library().ar_get_tuning(h, nbytes, ctypes.byref(a), ctypes.byref(p), us),
           "ar_get_tuning")
    return a.value, p.value, list(us)


def ar_reduce_scatter(h: int, ins, outs, stream=None) -> None:
    _check(load_library().ar_reduce_scatter(h, _ptr_array(ins), _ptr_array(outs), _stream(stream)),
           "ar_reduce_scatter")


def ar_all_gather(h: int, outs, stream=None) -> None:
    _check(load_library().ar_all_gather(h, _ptr_array(outs), _stream(stream)), "ar_all_gather")


def ar_ll_pack(h: int, src, pkts, n: int, flag: int, stream=None) -> None:
    _check(load_library().ar_ll_pack(h, _ptr(src), _ptr(pkts), n, flag & 0xFFFFFFFF,
                                     _stream(stream)), "ar_ll_pack")


def ar_ll_unpack(h: int, pkts, dst, n: int, flag: int, stream=None) -> None:
    _check(load_library().ar_ll_unpack(h, _ptr(pkts), _ptr(dst), n, flag & 0xFFFFFFFF,
                                       _stream(stream)), "ar_ll_unpack")


def ar_status(h: int, stream=None) -> int:
    """Wait for the stream; return (and clear) the handle's device status."""
    return load_library().ar_status(h, _stream(stream))


def ar_set_timeout(h: int, ns: int) -> None:
    _check(load_library().ar_set_timeout(h, ns), "ar_set_timeout")


def ar_set_pdl(h: int, enable: int) -> None:
    _check(load_library().ar_set_pdl(h, enable), "ar_set_pdl")


def ar_set_ll_transport(h: int, transport: int) -> None:
    _check(load_library().ar_set_ll_transport(h, transport), "ar_set_ll_transport")


def ar_set_hb_staging(h: int, staging: int) -> None:
    _check(load_library().ar_set_hb_staging(h, staging), "ar_set_hb_staging")


def ar_get_hb_staging(h: int, nbytes: int) -> int:
    """AR_HB_STAGING_TMA or AR_HB_STAGING_DIRECT: what a two-shot HB call of
    `nbytes` per rank (16-byte-aligned buffers) would use now."""
    out = ctypes.c_int(0)
    _check(load_library().ar_get_hb_staging(h, nbytes, ctypes.byref(out)), "ar_get_hb_staging")
    return out.value


def ar_set_grid_divisor(h: int, divisor: int) -> None:
    """Force the CTA-cap divisor of later calls (1, 2, 4, 8; 0 = tuned)."""
    _check(load_library().ar_set_grid_divisor(h, divisor), "ar_set_grid_divisor")


def ar_get_grid_divisor(h: int, nbytes: int, algo, proto) -> int:
    """The CTA-cap divisor a call of `nbytes` per rank with this algo and
    proto would use now."""
    algo = ALGOS[algo] if isinstance(algo, str) else algo
    proto = PROTOS[proto] if isinstance(proto, str) else proto
    out = ctypes.c_int(0)
    _check(load_library().ar_get_grid_divisor(h, nbytes, algo, proto, ctypes.byref(out)),
           "ar_get_grid_divisor")
    return out.value


def ar_debug_drop_rank(h: int, rank: int) -> None:
    _check(load_library().ar_debug_drop_rank(h, rank), "ar_debug_drop_rank")


def ar_round(dtype, src, dst, n: int, stream=None) -> None:
    dt = DTYPES[dtype] if isinstance(dtype, str) else dtype
    _check(load_library().ar_round(dt, _ptr(src), _ptr(dst), n, _stream(stream)), "ar_round")


def ar_get_info(h: int) -> dict:
    info = ar_info()
    _check(load_library().ar_get_info(h, ctypes.byref(info)), "ar_get_info")
    return info.as_dict()


def ar_allreduce_ll_static(R: int, N: int, dtype, ins, outs, stream=None) -> None:
    """One-shot LL all-reduce with no handle and no allocation, for callers
    that may not allocate device memory where they run it: an engine whose
    own pool holds nearly all of the GPU's memory, or a latency-critical
    hook that cannot pay for cudaMalloc's device-wide synchronisation.  The
    packet scratch is a static array inside the library (at most
    AR_NOALLOC_SCRATCH_BYTES of packets, else AR_ERR_UNSUPPORTED); the first
    call on a device sets it up and waits for that to finish; calls that
    overlap on the GPU race on the shared array."""
    dt = DTYPES[dtype] if isinstance(dtype, str) else dtype
    _check(load_library().ar_allreduce_ll_static(R, N, dt, _ptr_array(ins), _ptr_array(outs),
                                                 _stream(stream)), "ar_allreduce_ll_static")


AR_NOALLOC_SCRATCH_BYTES = 8 << 20


def make_op(kind, rank, dst, srcs, chunk_begin, chunk_end) -> ar_op:
    """One plan step.  dst = (buf, rank); srcs = [(buf, rank), ...] (all of
    one buffer kind)."""
    o = ar_op()
    o.kind = kind
    o.rank = rank
    o.dst_buf, o.dst_rank = dst
    o.src_buf = srcs[0][0]
    o.nsrc = len(srcs)
    for i, (b, r) in enumerate(srcs):
        if b != o.src_buf:
            raise ValueError("the sources of one step share a buffer kind")
        o.src_rank[i] = r
    o.chunk_begin, o.chunk_end = chunk_begin, chunk_end
    return o


def ar_plan_compile(h: int, ops, nchunks: int, ctas_per_rank: int = 1) -> int:
    arr = (ar_op * len(ops))(*ops)
    p = ctypes.c_void_p()
    _check(load_library().ar_plan_compile(h, arr, len(ops), nchunks, ctas_per_rank,
                                          ctypes.byref(p)), "ar_plan_compile")
    return p.value


def ar_plan_builtin(h: int, algo, chunks_per_rank: int = 0, ctas_per_rank: int = 0) -> int:
    algo = ALGOS[algo] if isinstance(algo, str) else algo
    p = ctypes.c_void_p()
    _check(load_library().ar_plan_builtin(h, algo, chunks_per_rank, ctas_per_rank,
                                          ctypes.byref(p)), "ar_plan_builtin")
    return p.value


def ar_plan_execute(p: int, ins, outs, stream=None) -> None:
    _check(load_library().ar_plan_execute(p, _ptr_array(ins), _ptr_array(outs), _stream(stream)),
           "ar_plan_execute")


def ar_plan_stats(p: int):
    t, w, s = ctypes.c_int(), ctypes.c_int(), ctypes.c_int()
    _check(load_library().ar_plan_stats(p, ctypes.byref(t), ctypes.byref(w), ctypes.byref(s)),
           "ar_plan_stats")
    return t.value, w.value, s.value


def ar_plan_destroy(p: int) -> None:
    _check(load_library().ar_plan_destroy(p), "ar_plan_destroy")


class Handle:
    """Owns one handle: ``with Handle(R, N, "bf16") as h: ar_allreduce(h.h, ...)``."""

    def __init__(self, R: int, N: int, dtype):
        self.R, self.N = R, N
        self.dtype = dtype
        self.h = ar_create(R, N, dtype)

    def close(self) -> None:
        if self.h:
            ar_destroy(self.h)
            self.h = 0

    def __enter__(self):
        return self

    def __exit__(self, *exc):
        self.close()

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass
