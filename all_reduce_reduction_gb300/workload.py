"""Seeded synthetic inputs for the all-reduce workloads.

This module only draws numbers.  It holds none of the all-reduce's arithmetic
(no sums, no rounding of sums, no packets); the final cast of each drawn
binary64 value to the buffer dtype is torch's own CPU cast.  Both the tests'
oracle side and the CUDA side take their inputs from here.

Generator: SplitMix64 (Steele, Lea and Flood, "Fast splittable pseudorandom
number generators", OOPSLA 2014; the 64-bit finaliser with Stafford's
"Mix13" constants as published by Vigna).  It is used as a counter-based
generator: draw ``c`` of a stream with seed ``s`` is
``mix(s + (c + 1) * 0x9E3779B97F4A7C15)``, so any element of any rank can be
recomputed on its own, and a prefix of a longer buffer equals the shorter
buffer with the same seed.

Seeds: ``0xA11ED000 + 97 * config + rank``.

Distributions (the workloads' value recipes):
  * ``uniform``     U[-1, 1): ``2u - 1`` with ``u = (draw >> 11) * 2^-53``
  * ``normal``      N(0, 1) by Box-Muller from draws 2i and 2i+1
  * ``loguniform``  ``+-10^(-4 + 8u)``, |x| in [1e-4, 1e4), the sign from a
                    second draw
"""
from __future__ import annotations

import math
from concurrent.futures import ThreadPoolExecutor
from dataclasses import dataclass

import numpy as np
import torch

GAMMA = np.uint64(0x9E3779B97F4A7C15)
MIX1 = np.uint64(0xBF58476D1CE4E5B9)
MIX2 = np.uint64(0x94D049BB133111EB)

TORCH_DTYPE = {"bf16": torch.bfloat16, "fp16": torch.float16, "fp32": torch.float32}
DTYPE_CODE = {"bf16": 0, "fp16": 1, "fp32": 2}
ELEM_SIZE = {"bf16": 2, "fp16": 2, "fp32": 4}

_CHUNK = 1 << 22


def seed_for(config: int, rank: int) -> int:
    return (0xA11ED000 + 97 * config + rank) & 0xFFFFFFFFFFFFFFFF


def splitmix64(seed: int, counters: np.ndarray) -> np.ndarray:
    """Draws ``counters`` (uint64 array) of the SplitMix64 stream ``seed``."""
    with np.errstate(over="ignore"):
        z = np.uint64(seed) + (counters.astype(np.uint64) + np.uint64(1)) * GAMMA
        z = (z ^ (z >> np.uint64(30))) * MIX1
        z = (z ^ (z >> np.uint64(27))) * MIX2
        return z ^ (z >> np.uint64(31))


def _unit(draws: np.ndarray) -> np.ndarray:
    """[0, 1) from the top 53 bits of each draw (exact in binary64)."""
    return (draws >> np.uint64(11)).astype(np.float64) * (2.0 ** -53)


def values_at(dist: str, seed: int, idx: np.ndarray) -> np.ndarray:
    """binary64 values of elements ``idx`` of the stream ``seed``."""
    idx = np.asarray(idx, dtype=np.uint64)
    if dist == "uniform":
        return 2.0 * _unit(splitmix64(seed, idx)) - 1.0
    if dist == "normal":
        u1 = 1.0 - _unit(splitmix64(seed, 2 * idx))          # (0, 1]
        u2 = _unit(splitmix64(seed, 2 * idx + np.uint64(1)))
        return np.sqrt(-2.0 * np.log(u1)) * np.cos(2.0 * math.pi * u2)
    if dist == "loguniform":
        u = _unit(splitmix64(seed, 2 * idx))
        s = splitmix64(seed, 2 * idx + np.uint64(1)) >> np.uint64(63)
        mag = np.power(10.0, -4.0 + 8.0 * u)
        return np.where(s == 1, -mag, mag)
    if dist == "integer":
        # small integers in [-8, 8]: sums of up to 32 of them are exact in
        # every dtype, which makes an exact closed-form expected value
        return (splitmix64(seed, idx) % np.uint64(17)).astype(np.float64) - 8.0
    raise ValueError("unknown distribution %r" % dist)


def rank_tensor(dist: str, seed: int, n: int, dtype: str) -> torch.Tensor:
    """n values of the stream cast to ``dtype`` (a CPU torch tensor)."""
    out = torch.empty(n, dtype=TORCH_DTYPE[dtype])
    for lo in range(0, n, _CHUNK):
        hi = min(n, lo + _CHUNK)
        x = values_at(dist, seed, np.arange(lo, hi, dtype=np.uint64))
        out[lo:hi] = torch.from_numpy(x).to(TORCH_DTYPE[dtype])
    return out


def make_inputs(config: int, R: int, n: int, dtype: str, dist: str,
                threads: int = 0) -> list[torch.Tensor]:
    """The R ranks' input buffers of a workload, as CPU torch tensors."""
    def one(r):
        return rank_tensor(dist, seed_for(config, r), n, dtype)
    if threads <= 1 or R == 1 or n < _CHUNK:
        return [one(r) for r in range(R)]
    with ThreadPoolExecutor(max_workers=min(threads, R)) as ex:
        return list(ex.map(one, range(R)))


def bits(t: torch.Tensor) -> np.ndarray:
    """The bit patterns of a CPU tensor as the oracle's numpy storage type."""
    t = t.contiguous()
    if t.dtype == torch.float32:
        return t.numpy()
    return t.view(torch.int16).numpy().view(np.uint16)


def from_bits(a: np.ndarray, dtype: str) -> torch.Tensor:
    """Inverse of :func:`bits`."""
    if dtype == "fp32":
        return torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32))
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.uint16).view(np.int16)).view(
        TORCH_DTYPE[dtype])


# Bit patterns at the edges of each format, for the special-value cases.  The
# first TINY_COUNT entries of a pool are signed zeros, subnormals and the
# smallest normals (their binary32 sums are subnormal or cancel into the
# subnormal range); the rest are ones and values near the largest finite one
# (their sums overflow to infinity).
SPECIAL_BITS = {
    "bf16": [0x0000, 0x8000, 0x0001, 0x8001, 0x0002, 0x8002, 0x007F, 0x807F, 0x0040, 0x8040,
             0x0080, 0x8080, 0x0081, 0x8081,
             0x3F80, 0xBF80, 0x7F7F, 0xFF7F, 0x7F00, 0xFF00, 0x4000, 0x3C00],
    "fp16": [0x0000, 0x8000, 0x0001, 0x8001, 0x0002, 0x8002, 0x03FF, 0x83FF, 0x0200, 0x8200,
             0x0400, 0x8400, 0x0401, 0x8401,
             0x3C00, 0xBC00, 0x7BFF, 0xFBFF, 0x7800, 0xF800, 0x4000, 0x1000],
    "fp32": [0x00000000, 0x80000000, 0x00000001, 0x80000001, 0x00000002, 0x80000002,
             0x007FFFFF, 0x807FFFFF, 0x00400000, 0x80400000, 0x00800000, 0x80800000,
             0x00800001, 0x80800001,
             0x3F800000, 0xBF800000, 0x7F7FFFFF, 0xFF7FFFFF, 0x7F000000, 0xFF000000,
             0x40000000, 0x33800000],
}
TINY_COUNT = 14

# binary32 gate weights for the special combine cases: signs, zeros, a
# subnormal, the smallest normal, small scales and the largest value below 1.
# All at most 1 in magnitude, so no product of finite values is infinite and
# no sum of opposite infinities (a NaN) can arise.
SPECIAL_WEIGHT_BITS = [0x3F800000, 0xBF800000, 0x3F000000, 0x00000000, 0x80000000, 0x00800000,
                       0x00000001, 0x3E800000, 0x3F7FFFFF, 0x0D800000]


def special_inputs(seed: int, R: int, n: int, dtype: str) -> list[torch.Tensor]:
    """R buffers of n elements picked from SPECIAL_BITS[dtype] by SplitMix64
    draws (stream seed + rank): even-indexed elements pick only among the
    tiny entries, odd ones among the whole pool."""
    pool = np.array(SPECIAL_BITS[dtype], dtype=np.uint32 if dtype == "fp32" else np.uint16)
    idx = np.arange(n, dtype=np.uint64)
    size = np.where(idx % np.uint64(2) == 0, np.uint64(TINY_COUNT), np.uint64(pool.size))
    return [from_bits(pool[(splitmix64(seed + r, idx) % size).astype(np.int64)].view(
        np.float32 if dtype == "fp32" else np.uint16), dtype) for r in range(R)]


def special_weights(seed: int, T: int, K: int) -> np.ndarray:
    """T x K binary32 gate weights picked from SPECIAL_WEIGHT_BITS."""
    pool = np.array(SPECIAL_WEIGHT_BITS, dtype=np.uint32)
    d = splitmix64(seed, np.arange(T * K, dtype=np.uint64)) % np.uint64(pool.size)
    return pool[d.astype(np.int64)].view(np.float32)


@dataclass(frozen=True)
class Workload:
    """One workload: R virtual ranks of n elements each."""
    config: int
    name: str
    R: int
    n: int
    dtype: str
    dist: str

    @property
    def bytes_per_rank(self) -> int:
        return self.n * ELEM_SIZE[self.dtype]

    def inputs(self, threads: int = 0) -> list[torch.Tensor]:
        return make_inputs(self.config, self.R, self.n, self.dtype, self.dist, threads)


def gate_weights(seed: int, T: int, K: int) -> np.ndarray:
    """Per-token gate weights: K draws in (0, 1] per token, divided by their
    token's sum in binary64 and cast to binary32 (row-major T x K)."""
    u = 1.0 - _unit(splitmix64(seed, np.arange(T * K, dtype=np.uint64))).reshape(T, K)
    return (u / u.sum(axis=1, keepdims=True)).astype(np.float32).reshape(-1)


@dataclass(frozen=True)
class CombineWorkload:
    """Weighted per-token combine: K sources of T tokens x H elements."""
    config: int
    name: str
    K: int
    T: int
    H: int
    dtype: str
    dist: str

    @property
    def R(self) -> int:          # sources, as "ranks"
        return self.K

    @property
    def n(self) -> int:          # elements per source
        return self.T * self.H

    def inputs(self, threads: int = 0) -> list[torch.Tensor]:
        return make_inputs(self.config, self.K, self.T * self.H, self.dtype, self.dist, threads)

    def weights(self) -> np.ndarray:
        return gate_weights(seed_for(self.config, 1000), self.T, self.K)


# The combine workloads: K = 8 sources (top-8 experts), hidden 8192, decode
# batches of 1..128 tokens and one prefill-sized batch of 4096 tokens.
COMBINE = [CombineWorkload(5, "k8_combine_t%d_h8192_bf16_normal" % t, 8, t, 8192, "bf16", "normal")
           for t in (1, 16, 128, 4096)]

# The five workloads.
SMALL = Workload(0, "r8_n512_bf16_uniform", 8, 512, "bf16", "uniform")
LL_SWEEP = [Workload(1, "r8_ll_sweep_n%d_bf16_uniform" % (1 << i), 8, 1 << i, "bf16", "uniform")
            for i in range(9, 19)]
DECODE = [Workload(2, "r8_decode_b%d_h8192_bf16_normal" % b, 8, 8192 * b, "bf16", "normal")
          for b in (1, 8, 32, 128, 256)]
PREFILL = Workload(3, "r16_prefill_8192x8192_bf16_normal", 16, 8192 * 8192, "bf16", "normal")
EDGE_N = 4097 * 4096 + 3
EDGE = [Workload(4, "r%d_edge_n%d_%s_loguniform" % (R, EDGE_N, dt), R, EDGE_N, dt, "loguniform")
        for R in (4, 32) for dt in ("bf16", "fp16", "fp32")]
