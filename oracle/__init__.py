"""CPU oracle for the virtual-rank sum all-reduce (test infrastructure only).

Only the tests, ``__graft_entry__.smoke()`` and the benchmark's CPU-baseline
leg may import this package.  The product path (the CUDA library and its
Python binding) never loads it and fails loudly when its own extension is
missing.

The arithmetic lives in ``ar_oracle.c`` (plain C11, compiled here with gcc,
no fast-math, no FP contraction); this module only builds it, loads it with
ctypes and moves numpy arrays in and out.  See the header of ``ar_oracle.c``
for what every function computes and which passage of the pages it follows.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(HERE, "ar_oracle.c")
LIB = os.path.join(HERE, "liboracle.so")

BF16, FP16, FP32 = 0, 1, 2
ELEM_SIZE = {BF16: 2, FP16: 2, FP32: 4}
# numpy storage type of each dtype's bit patterns
STORAGE = {BF16: np.uint16, FP16: np.uint16, FP32: np.float32}

CFLAGS = ["-O2", "-std=c11", "-fPIC", "-shared", "-ffp-contract=off",
          "-fno-fast-math", "-fno-unsafe-math-optimizations", "-Wall", "-Wextra"]

_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile liboracle.so next to its source if it is missing or stale."""
    if (not force and os.path.exists(LIB)
            and os.path.getmtime(LIB) >= os.path.getmtime(SRC)):
        return LIB
    tmp = LIB + ".tmp.%d" % os.getpid()
    subprocess.check_call(["gcc", *CFLAGS, "-o", tmp, SRC, "-lm"])
    os.replace(tmp, LIB)
    return LIB


def load(path: str | None = None) -> ctypes.CDLL:
    """Load (building first if needed) the oracle library."""
    global _lib
    with _lock:
        if path is not None:
            return _bind(ctypes.CDLL(path))
        if _lib is None:
            build()
            _lib = _bind(ctypes.CDLL(LIB))
        return _lib


def _bind(lib: ctypes.CDLL) -> ctypes.CDLL:
    vp, sz, i32, u32 = ctypes.c_void_p, ctypes.c_size_t, ctypes.c_int, ctypes.c_uint32
    vpp = ctypes.POINTER(ctypes.c_void_p)
    lib.oracle_elem_size.argtypes, lib.oracle_elem_size.restype = [i32], sz
    lib.oracle_bf16_to_f32.argtypes, lib.oracle_bf16_to_f32.restype = [ctypes.c_uint16], ctypes.c_float
    lib.oracle_fp16_to_f32.argtypes, lib.oracle_fp16_to_f32.restype = [ctypes.c_uint16], ctypes.c_float
    lib.oracle_f32_to_bf16.argtypes, lib.oracle_f32_to_bf16.restype = [ctypes.c_float], ctypes.c_uint16
    lib.oracle_f32_to_fp16.argtypes, lib.oracle_f32_to_fp16.restype = [ctypes.c_float], ctypes.c_uint16
    lib.oracle_allreduce.argtypes, lib.oracle_allreduce.restype = [i32, sz, i32, vpp, vpp], i32
    lib.oracle_reduce_scatter.argtypes, lib.oracle_reduce_scatter.restype = [i32, sz, i32, vpp, vpp], i32
    lib.oracle_shard_bounds.argtypes = [i32, sz, i32, i32, ctypes.POINTER(sz), ctypes.POINTER(sz)]
    lib.oracle_shard_bounds.restype = None
    lib.oracle_ll_packets.argtypes, lib.oracle_ll_packets.restype = [i32, sz], sz
    lib.oracle_ll_pack.argtypes, lib.oracle_ll_pack.restype = [i32, vp, sz, u32, vp], i32
    lib.oracle_ll_unpack.argtypes, lib.oracle_ll_unpack.restype = [i32, vp, sz, u32, vp], sz
    ip = ctypes.POINTER(ctypes.c_int)
    lib.oracle_plan_run.argtypes = [i32, sz, i32, i32, i32, ip, ip, ip, ip, ip, ip, vpp, vpp]
    lib.oracle_plan_run.restype = i32
    lib.oracle_combine.argtypes = [i32, sz, sz, i32, vpp, vp, vp]
    lib.oracle_combine.restype = i32
    lib.oracle_round_f32.argtypes, lib.oracle_round_f32.restype = [i32, vp, sz, vp], None
    lib.oracle_widen.argtypes, lib.oracle_widen.restype = [i32, vp, sz, vp], None
    return lib


def _ptr(a: np.ndarray) -> int:
    assert a.flags["C_CONTIGUOUS"]
    return a.ctypes.data


def _ptr_array(arrs) -> ctypes.Array:
    return (ctypes.c_void_p * len(arrs))(*[_ptr(a) for a in arrs])


def allreduce(ins, dtype: int, outs=None, lib=None):
    """out[r] = round_dtype(fold of ins[0..R-1] in binary32) for every r.

    ``ins`` is a list of R equal-length numpy arrays holding the dtype's bit
    patterns (uint16 for bf16/fp16, float32 for fp32).  Returns the R outputs
    (new arrays unless ``outs`` is given)."""
    lib = lib or load()
    R = len(ins)
    n = ins[0].size
    if outs is None:
        outs = [np.empty_like(ins[0]) for _ in range(R)]
    rc = lib.oracle_allreduce(R, n, dtype, _ptr_array(ins), _ptr_array(outs))
    if rc != 0:
        raise ValueError("oracle_allreduce rejected its arguments")
    return outs


def reduce_scatter(ins, dtype: int, outs, lib=None):
    """Shard j of outs[j] receives the reduced shard j; nothing else changes."""
    lib = lib or load()
    rc = lib.oracle_reduce_scatter(len(ins), ins[0].size, dtype, _ptr_array(ins), _ptr_array(outs))
    if rc != 0:
        raise ValueError("oracle_reduce_scatter rejected its arguments")
    return outs


def shard_bounds(R: int, n: int, dtype: int, j: int, lib=None):
    lib = lib or load()
    lo, hi = ctypes.c_size_t(), ctypes.c_size_t()
    lib.oracle_shard_bounds(R, n, dtype, j, ctypes.byref(lo), ctypes.byref(hi))
    return lo.value, hi.value


def ll_packets(dtype: int, n: int, lib=None) -> int:
    return (lib or load()).oracle_ll_packets(dtype, n)


def ll_pack(src: np.ndarray, dtype: int, flag: int, lib=None) -> np.ndarray:
    lib = lib or load()
    pk = np.empty(ll_packets(dtype, src.size, lib), dtype=np.uint64)
    lib.oracle_ll_pack(dtype, _ptr(src), src.size, flag, _ptr(pk))
    return pk


def ll_unpack(pkts: np.ndarray, dtype: int, n: int, flag: int, dst=None, lib=None):
    """Returns (dst, mismatch_count); mismatched packets leave dst untouched."""
    lib = lib or load()
    if dst is None:
        dst = np.zeros(n, dtype=STORAGE[dtype])
    bad = lib.oracle_ll_unpack(dtype, _ptr(np.ascontiguousarray(pkts)), n, flag, _ptr(dst))
    return dst, bad


def round_f32(x: np.ndarray, dtype: int, lib=None) -> np.ndarray:
    """Round binary32 values to the dtype (RNE); returns bit patterns."""
    lib = lib or load()
    x = np.ascontiguousarray(x, dtype=np.float32)
    out = np.empty(x.size, dtype=STORAGE[dtype])
    lib.oracle_round_f32(dtype, _ptr(x), x.size, _ptr(out))
    return out


def widen(bits: np.ndarray, dtype: int, lib=None) -> np.ndarray:
    """Exact widening of dtype bit patterns to binary32."""
    lib = lib or load()
    bits = np.ascontiguousarray(bits, dtype=STORAGE[dtype])
    out = np.empty(bits.size, dtype=np.float32)
    lib.oracle_widen(dtype, _ptr(bits), bits.size, _ptr(out))
    return out


def plan_run(steps, ins, outs, dtype: int, nchunks: int, lib=None):
    """Run a plan sequentially (see oracle_plan_run).  `steps` is a list of
    dicts with keys kind ('copy'|'reduce'), dst, srcs (buffer ids: b < R is
    in[b], R <= b < 2R is out[b - R]), cbeg, cend.  Modifies ins/outs in
    place and returns outs."""
    lib = lib or load()
    R = len(ins)
    n = len(steps)
    arr = lambda vals: (ctypes.c_int * max(1, len(vals)))(*vals)
    src = []
    for st in steps:
        src += list(st["srcs"]) + [0] * (32 - len(st["srcs"]))
    rc = lib.oracle_plan_run(
        R, ins[0].size, dtype, nchunks, n,
        arr([0 if st["kind"] == "copy" else 1 for st in steps]), arr([st["dst"] for st in steps]),
        arr([len(st["srcs"]) for st in steps]), arr(src), arr([st["cbeg"] for st in steps]),
        arr([st["cend"] for st in steps]), _ptr_array(ins), _ptr_array(outs))
    if rc != 0:
        raise ValueError("oracle_plan_run rejected the plan")
    return outs


def combine(ys, w: np.ndarray, T: int, H: int, dtype: int, lib=None) -> np.ndarray:
    """out[t*H+h] = round(fold_k w[t,k] * ys[k][t*H+h]) (see oracle_combine).
    ``w`` is a float32 array of T*K weights, row-major."""
    lib = lib or load()
    w = np.ascontiguousarray(w, dtype=np.float32)
    out = np.empty(T * H, dtype=STORAGE[dtype])
    rc = lib.oracle_combine(len(ys), T, H, dtype, _ptr_array(ys), _ptr(w), _ptr(out))
    if rc != 0:
        raise ValueError("oracle_combine rejected its arguments")
    return out
