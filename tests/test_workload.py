"""Pins for the seeded input generator, and the separation between the oracle
and the CUDA path.

The generator is SplitMix64 used as a counter-based stream.  Its outputs are
pinned to the first outputs of the reference C generator (Vigna's public
``splitmix64.c``) seeded with 0, and its counter form is checked against the
stateful form (add the golden gamma, then mix) stepped one draw at a time.
The value recipes are checked against their stated supports."""
import ast
import os

import numpy as np
import pytest

from all_reduce_reduction_gb300 import workload as wl

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

# first outputs of splitmix64.c with its state set to 0
SPLITMIX64_SEED0 = [0xE220A8397B1DCDAF, 0x6E789E6AA1B965F4, 0x06C45D188009454F,
                    0xF88BB8A8724C81EC]
M64 = (1 << 64) - 1


def _stateful(seed, count):
    """The generator as a state machine on Python integers."""
    x = seed & M64
    out = []
    for _ in range(count):
        x = (x + 0x9E3779B97F4A7C15) & M64
        z = x
        z = ((z ^ (z >> 30)) * 0xBF58476D1CE4E5B9) & M64
        z = ((z ^ (z >> 27)) * 0x94D049BB133111EB) & M64
        out.append(z ^ (z >> 31))
    return out


def test_splitmix64_matches_the_published_stream():
    got = wl.splitmix64(0, np.arange(4, dtype=np.uint64))
    assert [int(v) for v in got] == SPLITMIX64_SEED0
    assert _stateful(0, 4) == SPLITMIX64_SEED0


@pytest.mark.parametrize("seed", [1, 0xA11ED000, 0xA11ED000 + 97 * 3 + 31, M64])
def test_counter_form_equals_stepping(seed):
    got = wl.splitmix64(seed, np.arange(64, dtype=np.uint64))
    assert [int(v) for v in got] == _stateful(seed, 64)
    # any draw on its own, out of order
    idx = np.array([63, 0, 17, 5], dtype=np.uint64)
    assert [int(v) for v in wl.splitmix64(seed, idx)] == [_stateful(seed, 64)[i] for i in idx]


def test_unit_is_exact_and_below_one():
    d = np.array([0, 1 << 11, M64], dtype=np.uint64)
    u = wl._unit(d)
    assert u[0] == 0.0 and u[1] == 2.0 ** -53 and u[2] == 1.0 - 2.0 ** -53


@pytest.mark.parametrize("dtype", ["bf16", "fp16", "fp32"])
@pytest.mark.parametrize("dist", ["uniform", "normal", "loguniform", "integer"])
def test_prefix_and_rank_streams(dtype, dist):
    long = wl.make_inputs(7, 3, 5000, dtype, dist)
    short = wl.make_inputs(7, 3, 1234, dtype, dist)
    for a, b in zip(long, short):
        assert np.array_equal(wl.bits(a[:1234]), wl.bits(b))
    # every rank draws its own stream
    assert not np.array_equal(wl.bits(long[0]), wl.bits(long[1]))
    # the threaded draw is the same draw
    threaded = wl.make_inputs(7, 3, wl._CHUNK + 5, dtype, dist, threads=3)
    serial = wl.make_inputs(7, 3, wl._CHUNK + 5, dtype, dist)
    for a, b in zip(threaded, serial):
        assert np.array_equal(wl.bits(a), wl.bits(b))


def test_value_supports():
    idx = np.arange(200000, dtype=np.uint64)
    u = wl.values_at("uniform", 11, idx)
    assert u.min() >= -1.0 and u.max() < 1.0 and abs(u.mean()) < 0.01
    g = wl.values_at("normal", 11, idx)
    assert np.isfinite(g).all() and abs(g.mean()) < 0.01 and abs(g.std() - 1.0) < 0.01
    lg = wl.values_at("loguniform", 11, idx)
    m = np.abs(lg)
    assert m.min() >= 1e-4 and m.max() < 1e4
    assert abs(np.log10(m).mean()) < 0.05          # log10|x| uniform on [-4, 4)
    assert 0.49 < (lg < 0).mean() < 0.51
    k = wl.values_at("integer", 11, idx)
    assert np.array_equal(k, np.round(k)) and k.min() == -8.0 and k.max() == 8.0
    with pytest.raises(ValueError):
        wl.values_at("cauchy", 11, idx)


@pytest.mark.parametrize("dtype", ["bf16", "fp16", "fp32"])
def test_special_inputs_come_from_the_pool(dtype):
    bufs = wl.special_inputs(3, 5, 999, dtype)
    pool = set(wl.SPECIAL_BITS[dtype])
    tiny = set(wl.SPECIAL_BITS[dtype][:wl.TINY_COUNT])
    for t in bufs:
        b = wl.bits(t).view(np.uint32 if dtype == "fp32" else np.uint16).astype(np.int64)
        assert set(b.tolist()) <= pool
        assert set(b[0::2].tolist()) <= tiny
        # the odd elements reach past the tiny entries
        assert not set(b[1::2].tolist()) <= tiny


def test_special_and_gate_weights():
    w = wl.special_weights(5, 300, 8)
    assert w.dtype == np.float32 and w.shape == (2400,)
    assert np.isfinite(w).all() and np.abs(w).max() <= 1.0
    g = wl.gate_weights(5, 300, 8).reshape(300, 8).astype(np.float64)
    assert (g > 0).all()
    # binary64 row sums of 1, each term then rounded once to binary32
    assert np.abs(g.sum(axis=1) - 1.0).max() <= 8 * 2.0 ** -24


def _python_imports(path):
    tree = ast.parse(open(path).read())
    names = set()
    for node in ast.walk(tree):
        if isinstance(node, ast.Import):
            names.update(a.name.split(".")[0] for a in node.names)
        elif isinstance(node, ast.ImportFrom) and node.module and node.level == 0:
            names.add(node.module.split(".")[0])
    return names


def _files(folder, exts):
    for dp, _, fs in os.walk(os.path.join(ROOT, folder)):
        if "__pycache__" in dp or "_build" in dp:
            continue
        for f in fs:
            if f.endswith(exts):
                yield os.path.join(dp, f)


def test_oracle_and_cuda_path_share_no_code():
    # the product package never imports the oracle, and the oracle never
    # imports the package (its inputs arrive as arrays)
    for p in _files("all_reduce_reduction_gb300", (".py",)):
        assert "oracle" not in _python_imports(p), p
    for p in _files("oracle", (".py",)):
        assert "all_reduce_reduction_gb300" not in _python_imports(p), p
    # the C sides include nothing from each other
    for p in _files("all_reduce_reduction_gb300", (".cu", ".cuh", ".h", ".cpp", ".c")):
        for line in open(p):
            if line.lstrip().startswith("#include"):
                assert "oracle" not in line, (p, line)
    for p in _files("oracle", (".c", ".h")):
        for line in open(p):
            if line.lstrip().startswith("#include"):
                assert "<" in line, (p, line)      # system headers only

