"""Helpers shared by the tests (no all-reduce arithmetic here)."""
from __future__ import annotations

import json
import os

import numpy as np
import torch

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")

DT_CODE = {"bf16": 0, "fp16": 1, "fp32": 2}
STORAGE = {"bf16": np.uint16, "fp16": np.uint16, "fp32": np.float32}
UINT = {"bf16": np.uint16, "fp16": np.uint16, "fp32": np.uint32}


def golden(name: str) -> dict:
    with open(os.path.join(GOLDEN, name)) as f:
        return json.load(f)


def hex_array(items, dtype: str) -> np.ndarray:
    """Hex bit-pattern strings -> the oracle's storage array."""
    raw = np.array([int(h, 16) for h in items], dtype=UINT[dtype])
    return raw.view(STORAGE[dtype])


def as_uint(a: np.ndarray, dtype: str) -> np.ndarray:
    return np.ascontiguousarray(a).view(UINT[dtype])


def decode64(bits: np.ndarray, dtype: str) -> np.ndarray:
    """Exact binary64 values of dtype bit patterns, by numpy/torch casts."""
    if dtype == "fp32":
        return np.ascontiguousarray(bits).view(np.float32).astype(np.float64)
    if dtype == "fp16":
        return np.ascontiguousarray(bits).view(np.uint16).view(np.float16).astype(np.float64)
    u = np.ascontiguousarray(bits).view(np.uint16).astype(np.uint32) << np.uint32(16)
    return u.view(np.float32).astype(np.float64)


def spacing(x64: np.ndarray, dtype: str) -> np.ndarray:
    """Distance between consecutive dtype values around |x| (ulp), binary64."""
    mant_bits = {"bf16": 7, "fp16": 10, "fp32": 23}[dtype]
    min_exp = {"bf16": -126, "fp16": -14, "fp32": -126}[dtype]
    ax = np.abs(x64)
    with np.errstate(divide="ignore"):
        e = np.floor(np.log2(np.where(ax > 0, ax, 1.0)))
    e = np.maximum(e, min_exp)
    return np.ldexp(1.0, (e - mant_bits).astype(np.int64))


def to_torch_bits(t: torch.Tensor) -> np.ndarray:
    t = t.detach().cpu().contiguous()
    if t.dtype == torch.float32:
        return t.numpy().view(np.uint32)
    return t.view(torch.int16).numpy().view(np.uint16)


def same_bits(a: np.ndarray, b: np.ndarray, dtype: str) -> bool:
    return np.array_equal(as_uint(a, dtype), as_uint(b, dtype))


def first_mismatch(a: np.ndarray, b: np.ndarray, dtype: str):
    ua, ub = as_uint(a, dtype), as_uint(b, dtype)
    bad = np.nonzero(ua != ub)[0]
    if bad.size == 0:
        return None
    i = int(bad[0])
    return i, hex(int(ua[i])), hex(int(ub[i])), int(bad.size)
