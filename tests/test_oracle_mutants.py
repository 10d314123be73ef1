"""The oracle's pins catch plausible mistakes.

Each case plants one mistake in a private copy of the oracle's C source,
compiles that copy on the CPU, and checks that the pin suite below rejects
it.  The oracle itself is never modified.
"""
import subprocess

import numpy as np
import pytest
import torch

import oracle
from all_reduce_reduction_gb300 import workload as wl
from _util import DT_CODE, as_uint, decode64, golden, hex_array, spacing

MUTANTS = {
    "acc_starts_at_positive_zero": (
        "float acc = load_widened(dtype, in[0], i);\n    int k;\n    for (k = 1; k < R; ++k) {",
        "float acc = 0.0f;\n    int k;\n    for (k = 0; k < R; ++k) {"),
    "last_rank_dropped": ("for (k = 1; k < R; ++k) {", "for (k = 1; k < R - 1; ++k) {"),
    "ranks_folded_in_reverse": [
        ("float acc = load_widened(dtype, in[0], i);", "float acc = load_widened(dtype, in[R - 1], i);"),
        ("float x = load_widened(dtype, in[k], i);", "float x = load_widened(dtype, in[R - 1 - k], i);")],
    "wrong_sign": ("acc = acc + x;", "acc = acc - x;"),
    "element_index_shifted": ("float x = load_widened(dtype, in[k], i);",
                              "float x = load_widened(dtype, in[k], i ? i - 1 : i);"),
    "rounded_every_add": ("acc = acc + x;",
                          "acc = acc + x;\n        if (dtype == OR_BF16) acc = oracle_bf16_to_f32(oracle_f32_to_bf16(acc));"),
    "ties_to_odd": ("(D == 0x8000u && (K & 1u) != 0u)", "(D == 0x8000u && (K & 1u) == 0u)"),
    "bf16_truncates": ("        K += 1u;\n    return (uint16_t)((sign >> 16) | K);",
                       "        K += 0u;\n    return (uint16_t)((sign >> 16) | K);"),
    "fp16_flushes_subnormals": ("    if (q < 1024u)                     /* only reachable with Q == -24 */\n        return (uint16_t)(sign | q);",
                                "    if (q < 1024u)\n        return (uint16_t)sign;"),
    "fp16_ties_away": ("if (rest > half || (rest == half && (q & 1u) != 0u))", "if (rest >= half)"),
    "fp16_decode_bias_off": ("mag = ldexpf((float)(1024u + m), (int)e - 25);",
                             "mag = ldexpf((float)(1024u + m), (int)e - 24);"),
    "packet_bytes_big_endian": ("payload |= byte << (8 * j);", "payload |= byte << (8 * (3 - j));"),
    "combine_fuses_multiply_add": ("                float p = w[t * (size_t)K + (size_t)k] * load_widened(dtype, y[k], i);\n                acc = acc + p;",
                                   "                acc = fmaf(w[t * (size_t)K + (size_t)k], load_widened(dtype, y[k], i), acc);"),
    "combine_weights_transposed": ("float p = w[t * (size_t)K + (size_t)k]", "float p = w[(size_t)k * T + t]"),
    "flag_in_low_half": ("pkts[p] = ((uint64_t)flag << 32) | (uint64_t)payload;",
                         "pkts[p] = ((uint64_t)payload << 32) | (uint64_t)flag;"),
    "plan_chunks_not_whole_vectors": ("C = (C + per_vec - 1) / per_vec * per_vec;", "C = C + 0 * per_vec;"),
    "plan_last_chunk_dropped": ("for (c = cbeg[k]; c < cend[k]; ++c) {",
                                "for (c = cbeg[k]; c < cend[k] - 1; ++c) {"),
    "plan_in_and_out_swapped": ("d = dst[k] < R ? (void *)in[dst[k]] : out[dst[k] - R];",
                                "d = dst[k] < R ? out[dst[k]] : (void *)in[dst[k] - R];"),
    "plan_steps_reversed": ("for (k = 0; k < nsteps; ++k) {", "for (k = nsteps - 1; k >= 0; --k) {"),
    "shards_not_whole_vectors": ("    S = (S + per_vec - 1) / per_vec * per_vec;\n    a = (size_t)j * S;",
                                 "    S = S + 0 * per_vec;\n    a = (size_t)j * S;"),
    "shards_floor_division": ("size_t S = (N + (size_t)R - 1) / (size_t)R;", "size_t S = N / (size_t)R;"),
    "combine_starts_at_positive_zero": (
        "float acc = w[t * (size_t)K] * load_widened(dtype, y[0], i);\n            for (k = 1; k < K; ++k) {",
        "float acc = 0.0f;\n            for (k = 0; k < K; ++k) {"),
    "bf16_overflow_saturates": ("        K += 1u;\n    return (uint16_t)((sign >> 16) | K);",
                                "        K += 1u;\n    if (K > 0x7F7Fu)\n        K = 0x7F7Fu;\n"
                                "    return (uint16_t)((sign >> 16) | K);"),
    "fp16_overflow_saturates": ("    if (field >= 31)\n        return (uint16_t)(sign | 0x7C00u);",
                                "    if (field >= 31)\n        return (uint16_t)(sign | 0x7BFFu);"),
    "fp16_subnormal_widen_scale": ("mag = ldexpf((float)m, -24);", "mag = ldexpf((float)m, -25);"),
    "packet_tail_padded_with_ones": ("uint32_t byte = at < bytes ? (uint32_t)b[at] : 0u;",
                                     "uint32_t byte = at < bytes ? (uint32_t)b[at] : 0xFFu;"),
    "packet_count_rounds_down": ("    return (bytes + 3) / 4;", "    return bytes / 4;"),
    "unpack_accepts_any_flag": ("        if (f != flag) {\n            ++bad;\n            continue;\n        }",
                                "        if (f != flag)\n            ++bad;"),
}


def _pins_pass(lib) -> bool:
    """A compact run of the oracle's pins against a given build; False as
    soon as one fails."""
    # hand-derived fold cases
    for case in golden("fold_cases.json")["cases"]:
        dt = case["dtype"]
        ins = [hex_array([h], dt) for h in case["inputs"]]
        out = oracle.allreduce(ins, DT_CODE[dt], lib=lib)[0]
        if int(as_uint(out, dt)[0]) != int(case["expected"], 16):
            return False
    # exact integer sums and the binary64 bound
    for dt in ("bf16", "fp16", "fp32"):
        ts = wl.make_inputs(91, 7, 513, dt, "integer")
        exact = sum(t.to(torch.int64) for t in ts).to(torch.float64).to(wl.TORCH_DTYPE[dt])
        out = oracle.allreduce([wl.bits(t) for t in ts], DT_CODE[dt], lib=lib)[0]
        if not np.array_equal(as_uint(out, dt), as_uint(wl.bits(exact), dt)):
            return False
        ins = [wl.bits(t) for t in wl.make_inputs(90, 16, 1025, dt, "loguniform")]
        x = np.stack([decode64(a, dt) for a in ins])
        s = x.sum(axis=0)
        y = decode64(oracle.allreduce(ins, DT_CODE[dt], lib=lib)[0], dt)
        tol = spacing(s, dt) + 16 * 2.0 ** -24 * np.abs(x).sum(axis=0)
        fin = np.isfinite(y)
        if np.any(np.abs(y[fin] - s[fin]) > tol[fin]):
            return False
    # conversions against torch on a sample (subnormals and ties included)
    rng = np.random.default_rng(7)
    f = rng.integers(0, 1 << 32, size=1 << 18, dtype=np.uint64).astype(np.uint32)
    f = np.concatenate([f, np.arange(0, 1 << 16, dtype=np.uint32) << np.uint32(8)]).view(np.float32)
    f = f[np.isfinite(f)]
    for dt, td in ((0, torch.bfloat16), (1, torch.float16)):
        ours = oracle.round_f32(f, dt, lib=lib)
        ref = torch.from_numpy(f).to(td).view(torch.int16).numpy().view(np.uint16)
        if not np.array_equal(ours, ref):
            return False
        pats = np.arange(1 << 16, dtype=np.uint32).astype(np.uint16)
        w = oracle.widen(pats, dt, lib=lib)
        ref = torch.from_numpy(pats.view(np.int16)).view(td).float().numpy()
        ok = ~np.isnan(ref)
        if not np.array_equal(w[ok].view(np.uint32), ref[ok].view(np.uint32)):
            return False
    # weighted combine: hand-derived cases and power-of-two weights
    for case in golden("combine_cases.json")["cases"]:
        dt = case["dtype"]
        ys = [hex_array([h], dt) for h in case["y"]]
        w = np.array([int(x, 16) for x in case["w"]], dtype=np.uint32).view(np.float32)
        if int(as_uint(oracle.combine(ys, w, 1, 1, DT_CODE[dt], lib=lib), dt)[0]) != int(case["expected"], 16):
            return False
    ys = [wl.bits(t) for t in wl.make_inputs(88, 3, 4 * 8, "fp32", "uniform")]
    e = np.array([[0, 1, 2], [3, -1, 0], [1, 1, -2], [2, 0, 1]])
    scaled = [(ys[k].reshape(4, 8).astype(np.float64) * np.ldexp(1.0, e[:, k])[:, None])
              .astype(np.float32).reshape(-1) for k in range(3)]
    want = oracle.allreduce(scaled, DT_CODE["fp32"], lib=lib)[0]
    got = oracle.combine(ys, np.ldexp(1.0, e).astype(np.float32).reshape(-1), 4, 8, DT_CODE["fp32"], lib=lib)
    if not np.array_equal(got.view(np.uint32), want.view(np.uint32)):
        return False
    # plans: a built-in two-shot plan is the all-reduce, and random programs
    # equal a pure-Python restatement of a plan's meaning
    from plan_helpers import builtin_steps
    from test_oracle_plan import _python_plan, random_program
    ins = [wl.bits(t) for t in wl.make_inputs(89, 5, 203, "bf16", "normal")]
    outs = [np.zeros(203, np.uint16) for _ in range(5)]
    got = oracle.plan_run(builtin_steps(5, "two_shot", 2), [a.copy() for a in ins], outs,
                          DT_CODE["bf16"], 10, lib=lib)
    want = oracle.allreduce(ins, DT_CODE["bf16"], lib=lib)
    if any(not np.array_equal(got[r], want[r]) for r in range(5)):
        return False
    for seed in range(3):
        steps, ins, outs, nch = random_program("bf16", seed)
        w_in, w_out = _python_plan(steps, ins, outs, "bf16", nch)
        g_in, g_out = [a.copy() for a in ins], [a.copy() for a in outs]
        oracle.plan_run(steps, g_in, g_out, DT_CODE["bf16"], nch, lib=lib)
        if any(not np.array_equal(a, b) for a, b in zip(g_in + g_out, w_in + w_out)):
            return False
    # shards: a partition of [0, N) into R ranges, every boundary on a whole
    # 16-byte vector (or at N), at most one vector of difference in length
    # between consecutive full shards; the reduce-scatter writes only shard j
    # (33 = 4 * 8 + 1: floor(n / R) is already a whole vector, so a floor in
    # place of the ceiling would leave the last element in no shard)
    for dt, R, n in (("bf16", 4, 4097 * 3 + 3), ("fp32", 5, 9), ("fp16", 16, 1001),
                     ("bf16", 4, 33)):
        per_vec = 16 // wl.ELEM_SIZE[dt]
        bounds = [oracle.shard_bounds(R, n, DT_CODE[dt], j, lib=lib) for j in range(R)]
        if bounds[0][0] != 0 or bounds[-1][1] != n:
            return False
        if any(bounds[j][1] != bounds[j + 1][0] for j in range(R - 1)):
            return False
        if any(lo % per_vec and lo != n for lo, _ in bounds):
            return False
        if bounds[0][1] - bounds[0][0] < -(-n // R):     # the first shard holds ceil(n/R) or more
            return False
        ins = [wl.bits(t) for t in wl.make_inputs(87, R, n, dt, "normal")]
        full = oracle.allreduce(ins, DT_CODE[dt], lib=lib)[0]
        outs = [np.zeros(n, ins[0].dtype) for _ in range(R)]
        oracle.reduce_scatter(ins, DT_CODE[dt], outs, lib=lib)
        for j, (lo, hi) in enumerate(bounds):
            if not np.array_equal(as_uint(outs[j][lo:hi], dt), as_uint(full[lo:hi], dt)):
                return False
            rest = np.concatenate([as_uint(outs[j][:lo], dt), as_uint(outs[j][hi:], dt)])
            if rest.any():
                return False
    # packets, and an unpack that must leave the destination alone where the
    # flag does not match
    for case in golden("ll_packets.json")["cases"]:
        dt = case["dtype"]
        x = hex_array(case["elements"], dt)
        pk = oracle.ll_pack(x, DT_CODE[dt], int(case["flag"], 16), lib=lib)
        if [int(p) for p in pk] != [int(h, 16) for h in case["packets"]]:
            return False
        keep = np.full(x.size, 0x5A5A, np.uint32 if dt == "fp32" else np.uint16)
        keep = keep.view(np.float32) if dt == "fp32" else keep
        dst, bad = oracle.ll_unpack(pk, DT_CODE[dt], x.size, int(case["flag"], 16) ^ 1,
                                    dst=keep.copy(), lib=lib)
        if bad != len(pk) or not np.array_equal(as_uint(dst, dt), as_uint(keep, dt)):
            return False
    return True


def test_pins_accept_the_oracle(oracle_lib):
    assert _pins_pass(oracle_lib)


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_pins_reject_mutant(tmp_path, name):
    edits = MUTANTS[name]
    if isinstance(edits, tuple):
        edits = [edits]
    src = open(oracle.SRC).read()
    for old, new in edits:
        assert src.count(old) == 1, "mutation anchor not found: " + name
        src = src.replace(old, new)
    path = tmp_path / "mutant.c"
    path.write_text(src)
    so = str(tmp_path / ("lib_%s.so" % name))
    subprocess.check_call(["gcc", *oracle.CFLAGS, "-w", "-o", so, str(path), "-lm"])
    assert not _pins_pass(oracle.load(so)), "pins missed the planted mistake " + name
