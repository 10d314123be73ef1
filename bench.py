#!/usr/bin/env python3
"""Benchmark of the virtual-rank sum all-reduce on GB300.

Default workload: 8 virtual ranks, bf16, one-shot LL, message sizes
N = 2^9 .. 2^18 elements per rank (1 KiB .. 512 KiB), uniform [-1, 1) inputs;
10 all-reduce calls captured in one CUDA graph per size, 2 warm-up replays
(the message-size sweep and graph timing of "SGLang 中的 MSCCL++ All-Reduce
基准测试与推理集成指南", section 3.3).  One step = one replay of every size's
graph.  L2 is flushed (a 256 MiB write) before every replay, outside the
timed events.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload sweep|decode|prefill|edge]
                    [--impl ours|reference]

Prints one JSON line.  `value` is the whole job's throughput in GB/s on the
minimal-bytes basis (every input byte read once, every output byte written
once: 2 * R * N * elem_size per call), summed over all ranks; `sweep` gives
µs/call per message size.  `--impl reference` times the CPU oracle on the
host cores instead (the only other place this script runs it).  N > 1 runs N
independent replicas, one per GPU (the path has no cross-GPU exchange).
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import platform
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = ("all-reduce µs/call and GB/s vs msg size (R=8 bf16, 1 GB300), "
          "% of HBM roofline")
FALLBACK_HBM_GBS = 6800.0
NOMINAL_HBM_GBS = 7900.0        # GB300 HBM3e, nominal (context beside the measured peak)
TRANSPORTS = {"auto": 0, "global": 1, "cluster": 2}   # enum ar_ll_transport
STAGINGS = {"auto": 0, "tma": 1, "direct": 2}          # enum ar_hb_staging
L2_FLUSH_BYTES = 256 << 20


# ---------------------------------------------------------------------------
# workloads
# ---------------------------------------------------------------------------
def workload_cases(name: str, args=None):
    """(workload description, list of cases).  A case is one all-reduce
    configuration timed as a graph of `calls` calls."""
    from all_reduce_reduction_gb300 import workload as wl
    if name == "custom":
        dist_name = "uniform" if args.n <= (1 << 18) else "normal"
        w = wl.Workload(9, "custom_r%d_n%d_%s" % (args.R, args.n, args.dtype), args.R, args.n,
                        args.dtype, dist_name)
        big = 2 * w.R * w.n * wl.ELEM_SIZE[w.dtype] > (256 << 20)
        cases = [dict(w=w, algo=args.algo, proto=args.proto, calls=args.calls, flush=not big,
                      plan=args.plan, plan_chunks=args.plan_chunks, plan_ctas=args.plan_ctas)]
        desc = "custom: R=%d, N=%d %s per rank, %s, %d calls per CUDA graph" % (
            args.R, args.n, args.dtype,
            ("%s plan (%d chunks/rank, %d CTAs/rank)" % (args.plan, args.plan_chunks, args.plan_ctas))
            if args.plan else "%s %s" % (args.algo, args.proto), args.calls)
        if args.staging != "auto":
            desc += " (two-shot HB staging: %s)" % args.staging
    elif name == "sweep":
        cases = [dict(w=w, algo="one_shot", proto="ll", calls=10, flush=True) for w in wl.LL_SWEEP]
        desc = ("r8_bf16_ll_sweep: R=8 virtual ranks, bf16, N=2^9..2^18 elements per rank "
                "(1 KiB..512 KiB), uniform[-1,1), one-shot LL, 10 calls per CUDA graph")
    elif name == "decode":
        cases = [dict(w=w, algo="auto", proto="auto", calls=10, flush=True) for w in wl.DECODE]
        desc = ("r8_bf16_decode: R=8, bf16 [B, 8192] for B in 1,8,32,128,256, N(0,1), "
                "AUTO (tuned) schedule and protocol, 10 calls per CUDA graph")
    elif name == "combine":
        cases = [dict(w=w, combine=True, algo="combine", proto="hb", calls=10,
                      flush=True) for w in wl.COMBINE]
        desc = ("k8_bf16_combine: weighted per-token combine of K=8 sources, T in 1,16,128,4096 "
                "tokens x H=8192 bf16, N(0,1) values, normalised gate weights; 10 calls per graph")
    elif name == "prefill":
        cases = [dict(w=wl.PREFILL, algo="two_shot", proto="hb", calls=1, flush=False)]
        desc = ("r16_bf16_prefill: R=16, bf16 [8192, 8192] per rank (128 MiB), N(0,1), "
                "two-shot HB (staging: %s)" % (args.staging if args else "auto"))
    elif name == "edge":
        w = [x for x in wl.EDGE if x.R == 32 and x.dtype == "fp32"][0]
        cases = [dict(w=w, algo="two_shot", proto="hb", calls=1, flush=False)]
        desc = ("r32_fp32_edge: R=32, fp32, N=4097*4096+3 per rank, log-uniform |x| in "
                "[1e-4,1e4), two-shot HB (staging: %s)" % (args.staging if args else "auto"))
    else:
        raise SystemExit("unknown workload " + name)
    return desc, cases


def case_bytes(c) -> int:
    """Minimal bytes of one call: every input byte read once, every output
    byte written once (combine: K sources + the weights + one output)."""
    w = c["w"]
    from all_reduce_reduction_gb300 import workload as wl
    if c.get("combine"):
        return (w.K + 1) * w.T * w.H * wl.ELEM_SIZE[w.dtype] + 4 * w.T * w.K
    return 2 * w.R * w.n * wl.ELEM_SIZE[w.dtype]


# ---------------------------------------------------------------------------
# distributed plumbing (host side only: a barrier and a max over ranks)
# ---------------------------------------------------------------------------
class Dist:
    def __init__(self):
        self.world = int(os.environ.get("WORLD_SIZE", "1"))
        self.rank = int(os.environ.get("RANK", "0"))
        self.local_rank = int(os.environ.get("LOCAL_RANK", "0"))
        self.pg = None
        if self.world > 1:
            import torch.distributed as dist
            dist.init_process_group("gloo")
            self.pg = dist

    def barrier(self):
        if self.pg:
            self.pg.barrier()

    def max(self, x: float) -> float:
        if not self.pg:
            return x
        import torch
        t = torch.tensor([x], dtype=torch.float64)
        self.pg.all_reduce(t, op=self.pg.ReduceOp.MAX)
        return float(t.item())

    def sum(self, x: float) -> float:
        if not self.pg:
            return x
        import torch
        t = torch.tensor([x], dtype=torch.float64)
        self.pg.all_reduce(t, op=self.pg.ReduceOp.SUM)
        return float(t.item())

    def close(self):
        if self.pg:
            self.pg.destroy_process_group()


# ---------------------------------------------------------------------------
# clocks during the timed region
# ---------------------------------------------------------------------------
REASONS = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]


class ClockSampler:
    def __init__(self, bus_id: str | None):
        self.bus_id = bus_id
        self.proc = None
        self.path = None

    def start(self):
        q = ("pci.bus_id,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             + ",".join("clocks_event_reasons." + r for r in REASONS) + ",timestamp")
        try:
            import tempfile
            fd, self.path = tempfile.mkstemp(prefix="clocks_", suffix=".csv")
            os.close(fd)
            self.out = open(self.path, "w")
            self.proc = subprocess.Popen(
                ["nvidia-smi", "--query-gpu=" + q, "--format=csv,noheader,nounits", "-lms", "50"],
                stdout=self.out, stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None

    def stop(self) -> dict | None:
        if not self.proc:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        self.out.close()
        with open(self.path) as f:
            lines = f.readlines()
        os.unlink(self.path)
        return parse_clock_rows(lines, self.bus_id)


def parse_smi_time(text: str) -> float | None:
    """Seconds since the epoch of an nvidia-smi timestamp such as
    "2026/12/03 05:29:26.123" (the host's local time, as time.time() counts)."""
    import datetime
    for fmt in ("%Y/%m/%d %H:%M:%S.%f", "%Y/%m/%d %H:%M:%S"):
        try:
            return datetime.datetime.strptime(text.strip(), fmt).timestamp()
        except ValueError:
            pass
    return None


def parse_clock_rows(lines, bus_id: str | None) -> dict | None:
    """Summarise nvidia-smi CSV rows (pci.bus_id, clocks.sm, clocks.max.sm,
    power.draw, reasons.active, then one Active/Not Active column per REASONS
    entry, then an optional timestamp) of the GPU whose bus id ends with
    `bus_id`.  `series` lists (seconds since the epoch, SM MHz) of the rows
    that carry both."""
    rows = []
    for line in lines:
        f = [x.strip() for x in line.split(",")]
        if len(f) < 5 + len(REASONS):
            continue
        if bus_id and not f[0].lower().endswith(bus_id.lower()):
            continue
        rows.append(f)
    if not rows:
        return None
    sm = [float(r[1]) for r in rows if r[1].replace(".", "").isdigit()]
    mx = [float(r[2]) for r in rows if r[2].replace(".", "").isdigit()]
    seen = sorted({REASONS[i] for r in rows for i in range(len(REASONS))
                   if r[5 + i].lower().startswith("active")})
    series = []
    for r in rows:
        if len(r) > 5 + len(REASONS) and r[1].replace(".", "").isdigit():
            t = parse_smi_time(r[5 + len(REASONS)])
            if t is not None:
                series.append((t, float(r[1])))
    return {"sm_mhz": statistics.median(sm) if sm else None,
            "sm_max_mhz": max(mx) if mx else None,
            "reasons": seen, "samples": len(rows), "series": series}


def clocks_for_windows(series, windows, reach: float = 0.06) -> dict:
    """The SM clock seen by a set of replays: for every replay window
    (start, end) in seconds since the epoch, the clock sample nearest to the
    window's middle, if one lies within `reach` seconds; returns the median
    of those samples and how many replays had one."""
    if not series:
        return {"sm_mhz_median": None, "replays_with_sample": 0}
    ts = sorted(series)
    got = []
    for lo, hi in windows:
        mid = 0.5 * (lo + hi)
        t, mhz = min(ts, key=lambda x: abs(x[0] - mid))
        if abs(t - mid) <= reach + 0.5 * (hi - lo):
            got.append(mhz)
    return {"sm_mhz_median": statistics.median(got) if got else None,
            "replays_with_sample": len(got)}


def replay_stats(times_ms, calls: int) -> dict:
    """µs per call of individual graph replays (each `calls` calls): median,
    90th percentile (nearest rank), minimum and maximum."""
    us = sorted(t * 1e3 / calls for t in times_ms)
    if not us:
        return {}
    p90 = us[min(len(us) - 1, max(0, -(-9 * len(us) // 10) - 1))]
    return {"us_p50": round(statistics.median(us), 3), "us_p90": round(p90, 3),
            "us_min": round(us[0], 3), "us_max": round(us[-1], 3), "replays": len(us)}


def clocks_rejected(c: dict | None) -> bool:
    if not c:
        return False
    if set(c["reasons"]) & {"hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown"}:
        return True
    if c["sm_mhz"] and c["sm_max_mhz"] and not c["reasons"] and c["sm_mhz"] < 0.6 * c["sm_max_mhz"]:
        return True
    return False


# ---------------------------------------------------------------------------
# peaks and committed ncu traffic
# ---------------------------------------------------------------------------
def ll_wire_bytes(r):
    """Bytes the one-shot LL call moves through L2 with its packets counted
    (8-byte packets carry 4 payload bytes): every input read, every packet
    stored and loaded once, every output written.  None for other paths,
    whose bytes are the minimal ones."""
    import all_reduce_reduction_gb300 as ar
    from all_reduce_reduction_gb300 import workload as wl
    if r.c.get("plan") or r.c.get("combine"):
        return None
    if (r.choice or "%s_%s" % (r.c["algo"], r.c["proto"])) != "one_shot_ll":
        return None
    if r.c.get("transport", ar.AR_LL_AUTO) == ar.AR_LL_CLUSTER:
        return None                     # its packets travel through shared memory
    nb = r.w.n * wl.ELEM_SIZE[r.w.dtype]
    packets = 8 * -(-nb // 4)
    return r.w.R * (2 * nb + 2 * packets)


def staged_path(r, path: str) -> str:
    """The kernel family of a case's path: two-shot HB is named with the
    staging its calls use (its buffers are all 16-byte aligned here)."""
    import all_reduce_reduction_gb300 as ar
    from all_reduce_reduction_gb300 import workload as wl
    if path != "two_shot_hb":
        return path
    st = ar.ar_get_hb_staging(r.h.h, r.w.n * wl.ELEM_SIZE[r.w.dtype])
    return "two_shot_hb_tma" if st == ar.AR_HB_STAGING_TMA else "two_shot_hb_direct"


def hbm_peak():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            return float(json.load(f)["hbm_gbs"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


# device sources of each kernel family (the key's leading words): whole
# files, or, where a file holds several kernels, (file, functions): the
# file's helpers before its first kernel plus those functions alone
KERNEL_SOURCES = {
    "one_shot_ll_global": [("ar_ll.cu", ["k_ll_staged", "launch_ll_staged"])],
    "two_shot_ll": [("ar_ll.cu", ["k_ll2_staged", "launch_ll_staged"])],
    "one_shot_ll_cluster": ["ar_ll_cluster.cu"],
    "one_shot_hb": [("ar_hb.cu", ["k_one_shot_hb", "one_shot_smem", "one_shot_unrolled", "one_shot_dt",
                                  "one_shot_prepare_dt", "one_shot_prepare", "launch_one_shot_hb"])],
    # the two-shot launcher picks each staging's form (tile, stages, grid;
    # CTA width) by message size: it counts too
    "two_shot_hb_tma": ["ar_tma.cu", ("ar_api.cu", ["two_shot_hb"])],
    "two_shot_hb_direct": [("ar_hb.cu", ["reduce_body", "k_reduce", "k_reduce_o4", "k_reduce_wide",
                                         "reduce_dt", "launch_reduce"]),
                           ("ar_api.cu", ["two_shot_hb"])],
    "combine": ["ar_combine.cu"],
    # a plan's traffic follows its compiled tasks: the compiler counts too
    "plan_": [("ar_plan.cu", ["k_plan", "compile_plan", "builtin_plan", "ar_plan_execute"])],
}


def strip_comments(src: str) -> str:
    """C/C++ source without its comments and with whitespace runs collapsed
    (string and character literals kept as they are)."""
    out, i, n = [], 0, len(src)
    while i < n:
        c = src[i]
        if c in "\"'":
            j = i + 1
            while j < n and src[j] != c:
                j += 2 if src[j] == "\\" else 1
            out.append(src[i:j + 1])
            i = j + 1
        elif src.startswith("//", i):
            j = src.find("\n", i)
            i = n if j < 0 else j
        elif src.startswith("/*", i):
            j = src.find("*/", i + 2)
            out.append(" ")
            i = n if j < 0 else j + 2
        else:
            out.append(c)
            i += 1
    return " ".join("".join(out).split())


def function_source(src: str, name: str) -> str:
    """The definition of function `name` in comment-stripped source: from its
    name to the brace that closes its body (the first occurrence whose
    parameter list is followed by a body, not a call or a declaration)."""
    i = 0
    while True:
        i = src.find(name + "(", i)
        if i < 0:
            raise KeyError(name)
        if i > 0 and (src[i - 1].isalnum() or src[i - 1] == "_"):
            i += 1
            continue
        depth, j = 0, i + len(name)
        while j < len(src):                 # the parameter list's closing parenthesis
            if src[j] == "(":
                depth += 1
            elif src[j] == ")":
                depth -= 1
                if depth == 0:
                    break
            j += 1
        k = j + 1
        while k < len(src) and src[k].isspace():
            k += 1
        if k >= len(src) or src[k] != "{":
            i += 1
            continue
        depth = 0
        while k < len(src):                 # the body's closing brace
            if src[k] == "{":
                depth += 1
            elif src[k] == "}":
                depth -= 1
                if depth == 0:
                    return src[i:k + 1]
            k += 1
        raise KeyError(name)


def kernel_source_digest(kernel_key: str) -> str:
    """Digest of the device code a kernel key names: its .cu file (or, for a
    file holding several kernels, the file's helpers and the named functions)
    plus the shared device header, comments and layout aside.  Any change to
    that code invalidates recorded counters."""
    files = None
    for prefix, fs in KERNEL_SOURCES.items():
        if kernel_key.startswith(prefix):
            files = fs
    if files is None:
        return "unknown"
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "all_reduce_reduction_gb300", "csrc")
    for entry in files + ["ar_device.cuh"]:
        fn, funcs = entry if isinstance(entry, tuple) else (entry, None)
        text = strip_comments(open(os.path.join(csrc, fn)).read())
        if funcs is None:
            h.update(text.encode())
            continue
        first = text.find("__global__")     # a kernel file's helpers precede its kernels
        h.update(text[:first if first >= 0 else 0].encode())
        for f in funcs:
            h.update(function_source(text, f).encode())
    return h.hexdigest()[:16]


def committed_traffic(kernel_key: str):
    """DRAM bytes per launch recorded by an ncu capture in profiles/, if the
    kernel's device code has not changed since (same digest); else None."""
    path = os.path.join(ROOT, "profiles", "traffic.txt")
    if not os.path.exists(path):
        return None
    digest = kernel_source_digest(kernel_key)
    for line in open(path):
        f = line.split()
        if len(f) >= 3 and f[0] == kernel_key and f[2] == digest:
            return float(f[1])
    return None


# ---------------------------------------------------------------------------
# our arm
# ---------------------------------------------------------------------------
def rank_stride(n: int, elem_size: int) -> int:
    """Elements between the starts of consecutive ranks' buffers in a block:
    n rounded up to a whole 256 bytes."""
    per = 256 // elem_size
    return -(-n // per) * per


class CaseRunner:
    """Handle, device inputs/outputs and a captured graph for one case."""

    def __init__(self, c, stream, host_buffers: bool = True):
        import torch
        import all_reduce_reduction_gb300 as ar
        from all_reduce_reduction_gb300 import workload as wl
        self.c, self.w, self.s = c, c["w"], stream
        w = self.w
        self.cpu_inputs = w.inputs(threads=16)
        # the R rank buffers of each direction are views of one allocation, so
        # the end-to-end leg moves them with one copy each way; every rank
        # starts on a 256-byte boundary, as separately allocated buffers would
        # (an odd N would otherwise leave ranks 1.. off 16-byte alignment and
        # send them down the element-wise paths)
        n = self.cpu_inputs[0].numel()
        self.stride = rank_stride(n, self.cpu_inputs[0].element_size())
        nin = len(self.cpu_inputs)
        in_block = torch.zeros(nin * self.stride, dtype=self.cpu_inputs[0].dtype, device="cuda")
        self.ins = [in_block[r * self.stride:r * self.stride + n] for r in range(nin)]
        for d, t in zip(self.ins, self.cpu_inputs):
            d.copy_(t)
        self.in_block = in_block
        nout = 1 if c.get("combine") else nin
        self.out_block = torch.zeros(nout * self.stride, dtype=in_block.dtype, device="cuda")
        self.outs = [self.out_block[r * self.stride:r * self.stride + n] for r in range(nout)]
        assert all(t.data_ptr() % 256 == 0 for t in self.ins + self.outs)
        if c.get("combine"):
            self.weights = torch.from_numpy(w.weights()).cuda()
            self.h = ar.Handle(w.K, w.T * w.H, w.dtype)
        else:
            self.h = ar.Handle(w.R, w.n, w.dtype)
        ar.ar_set_ll_transport(self.h.h, c.get("transport", ar.AR_LL_AUTO))
        ar.ar_set_hb_staging(self.h.h, c.get("staging", ar.AR_HB_STAGING_AUTO))
        ar.ar_set_grid_divisor(self.h.h, c.get("grid_divisor", 0))
        ar.ar_set_pdl(self.h.h, c.get("pdl", 1))
        self.algo, self.proto = ar.ALGOS.get(c["algo"], 0), ar.PROTOS[c["proto"]]
        self.choice = "combine" if c.get("combine") else None
        if c["algo"] == "auto" or c["proto"] == "auto":
            ar.ar_tune(self.h.h, stream)
            a, p, _ = ar.ar_get_tuning(self.h.h, w.n * wl.ELEM_SIZE[w.dtype])
            self.choice = "%s_%s" % ({0: "one_shot", 1: "two_shot"}[a], {0: "ll", 1: "hb"}[p])
        self.bytes = case_bytes(c)
        self.plan = None
        if c.get("plan"):
            # the same all-reduce as a compiled plan run by the interpreter kernel
            self.plan = ar.ar_plan_builtin(self.h.h, c["plan"], c.get("plan_chunks", 0),
                                           c.get("plan_ctas", 0))

        def call():
            if c.get("combine"):
                ar.ar_combine(self.h.h, self.ins, self.weights, self.outs[0], w.T, w.H,
                              stream=stream)
            elif self.plan:
                ar.ar_plan_execute(self.plan, self.ins, self.outs, stream=stream)
            else:
                ar.ar_allreduce(self.h.h, self.ins, self.outs, self.algo, self.proto,
                                stream=stream)

        self.call = call
        with torch.cuda.stream(stream):
            call()
        stream.synchronize()
        self.graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(self.graph, stream=stream):
            for _ in range(c["calls"]):
                call()
        for _ in range(2):
            self.graph.replay()
        torch.cuda.synchronize()
        if ar.ar_status(self.h.h) != ar.AR_OK:
            raise RuntimeError("device status after warm-up: " + ar.ar_strerror(ar.ar_status(self.h.h)))
        self.pinned_in = self.pinned_out = None
        if not host_buffers:
            self.cpu_inputs = None
            return
        self.pinned_in = torch.zeros(in_block.shape, dtype=in_block.dtype).pin_memory()
        for r, t in enumerate(self.cpu_inputs):
            self.pinned_in[r * self.stride:r * self.stride + n].copy_(t)
        self.pinned_out = torch.empty(self.out_block.shape, dtype=self.out_block.dtype).pin_memory()
        self.host_bytes = (nin * n * self.pinned_in.element_size(),
                           nout * n * self.pinned_out.element_size())
        self.host_call = None
        if not c.get("combine") and not self.plan:
            # the same all-reduce on the page-locked host buffers themselves
            hins = [self.pinned_in[r * self.stride:r * self.stride + n] for r in range(nin)]
            houts = [self.pinned_out[r * self.stride:r * self.stride + n] for r in range(nout)]

            def host_call():
                ar.ar_allreduce_host(self.h.h, hins, houts, n, self.algo, self.proto,
                                     stream=stream)

            self.host_call = host_call

    def close(self):
        import all_reduce_reduction_gb300 as ar
        if self.plan:
            ar.ar_plan_destroy(self.plan)
        self.h.close()


def run_ours(args, dist: Dist):
    import torch
    import all_reduce_reduction_gb300 as ar
    from all_reduce_reduction_gb300 import workload as wl

    torch.cuda.set_device(dist.local_rank)
    desc, cases = workload_cases(args.workload, args)
    if args.only:
        cases = [c for c in cases if c["w"].n == args.only]
        if not cases:
            raise SystemExit("--only %d matches no case of the workload" % args.only)
        desc += " (only the case of %d elements per rank)" % args.only
    if args.grid_divisor:
        desc += " (CTA-cap divisor %d)" % args.grid_divisor
    for c in cases:
        c["transport"] = TRANSPORTS[args.ll_transport]
        c["staging"] = STAGINGS[args.staging]
        c["grid_divisor"] = args.grid_divisor
        c["pdl"] = 0 if args.no_pdl else 1
    stream = torch.cuda.Stream()
    runners = [CaseRunner(c, stream) for c in cases]
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device="cuda")

    def one_step(events):
        for i, r in enumerate(runners):
            with torch.cuda.stream(stream):
                if r.c["flush"]:
                    flush.fill_(i & 0xFF)
                e0 = torch.cuda.Event(enable_timing=True)
                e1 = torch.cuda.Event(enable_timing=True)
                e0.record(stream)
                r.graph.replay()
                e1.record(stream)
            events.append((i, e0, e1))

    def timed(K):
        """Sum of event time per case, each replay's time per case, and each
        replay's (start, end) in host seconds since the epoch (the GPU's
        event clock anchored at an event recorded on an idle stream)."""
        events = []
        dist.barrier()
        torch.cuda.synchronize()
        anchor = torch.cuda.Event(enable_timing=True)
        with torch.cuda.stream(stream):
            anchor.record(stream)
        t_anchor = time.time()
        for _ in range(K):
            one_step(events)
        torch.cuda.synchronize()
        dist.barrier()
        per_case = [0.0] * len(runners)
        replays = [[] for _ in runners]
        windows = [[] for _ in runners]
        for i, e0, e1 in events:
            ms = e0.elapsed_time(e1)
            per_case[i] += ms
            replays[i].append(ms)
            t0 = t_anchor + anchor.elapsed_time(e0) * 1e-3
            windows[i].append((t0, t0 + ms * 1e-3))
        return per_case, replays, windows

    for _ in range(args.warmup):
        one_step([])
    torch.cuda.synchronize()

    props = torch.cuda.get_device_properties(dist.local_rank)
    bus = None
    if hasattr(props, "pci_bus_id"):
        bus = "%02X:%02X.0" % (props.pci_bus_id, props.pci_device_id)
    sampler = ClockSampler(bus)
    sampler.start()
    time.sleep(0.2)                     # the sampler's first rows precede the timed region
    per_case, replays, windows = timed(args.steps)
    time.sleep(0.1)
    clocks = sampler.stop()
    remeasured = False
    if clocks_rejected(clocks):
        sampler = ClockSampler(bus)
        sampler.start()
        time.sleep(0.2)
        per_case, replays, windows = timed(args.steps)
        time.sleep(0.1)
        clocks = sampler.stop()
        remeasured = True
    series = clocks.pop("series", []) if clocks else []

    total_ms = sum(per_case)
    for r in runners:
        st = ar.ar_status(r.h.h, stream)
        if st != ar.AR_OK:
            raise RuntimeError("device status after the timed region: " + ar.ar_strerror(st))
    calls = [r.c["calls"] for r in runners]
    bytes_step = sum(r.bytes * k for r, k in zip(runners, calls))
    ms_step = dist.max(total_ms / args.steps)
    value = dist.sum(bytes_step) / (ms_step * 1e-3) / 1e9

    # dominant kernel: the case with the largest share of the step
    dom = max(range(len(runners)), key=lambda i: per_case[i])
    dr = runners[dom]
    launch_s = per_case[dom] * 1e-3 / (args.steps * dr.c["calls"])
    peak, peak_kind = hbm_peak()
    achieved = dr.bytes / launch_s / 1e9
    path = dr.choice or ("plan_" + dr.c["plan"] if dr.c.get("plan") else
                         "%s_%s" % (dr.c["algo"], dr.c["proto"]))
    kkey = "%s_r%d_n%d_%s" % (staged_path(dr, path), dr.w.R, dr.w.n, dr.w.dtype)
    if path == "one_shot_ll":
        info = ar.ar_get_info(dr.h.h)
        tr = dr.c.get("transport", ar.AR_LL_AUTO)
        cluster = bool(info["ll_cluster_ok"]) and tr == ar.AR_LL_CLUSTER
        kkey = kkey.replace("_ll_", "_ll_cluster_" if cluster else "_ll_global_")
    roofline = {"bound": "hbm", "achieved": round(achieved, 1), "peak": peak, "unit": "GB/s",
                "frac": round(achieved / peak, 4), "traffic": committed_traffic(kkey),
                "kernel": kkey, "peak_source": peak_kind + " (MEASURED_PEAKS.json hbm_gbs)"
                if peak_kind == "measured" else "fallback 6800 GB/s",
                "nominal_peak": NOMINAL_HBM_GBS,
                "frac_of_nominal": round(achieved / NOMINAL_HBM_GBS, 4)}

    sweep = {}
    for i, r in enumerate(runners):
        us = per_case[i] * 1e3 / (args.steps * r.c["calls"])
        nb = r.w.n * wl.ELEM_SIZE[r.w.dtype]
        sweep[str(r.w.n)] = {
            "bytes_per_rank": nb, "us_per_call": round(us, 3),
            "algbw_GBps": round(nb / us / 1e3, 2),
            "busbw_GBps": round(nb / us / 1e3 * 2 * (r.w.R - 1) / r.w.R, 2),
            "min_bytes_GBps": round(r.bytes / us / 1e3, 1),
            "frac_of_hbm_peak": round(r.bytes / us / 1e3 / peak, 4),
            "l2_resident": 2 * r.bytes <= 100 << 20,
        }
        sweep[str(r.w.n)].update(replay_stats(replays[i], r.c["calls"]))
        sweep[str(r.w.n)]["clock"] = clocks_for_windows(series, windows[i])
        wire = ll_wire_bytes(r)
        if wire is not None:
            sweep[str(r.w.n)]["wire_bytes_per_call"] = wire
            sweep[str(r.w.n)]["wire_GBps"] = round(wire / us / 1e3, 1)
        if r.choice:
            sweep[str(r.w.n)]["auto_choice"] = r.choice

    # end to end, one host round trip per all-reduce: every step, each case's
    # R inputs come from page-locked host memory and all its outputs go back
    # to page-locked host memory, one all-reduce per case.  Two forms, each
    # captured once per case as a one-call CUDA graph and replayed, with CUDA
    # events on the stream around each replay:
    #   host:   the library's host-buffer call (ar_allreduce_host): its
    #           kernels read the inputs from and write the outputs to host
    #           memory through the CPU-GPU link;
    #   copies: the inputs copied in, the device-buffer call, the outputs
    #           copied back (two copy nodes around the call).
    # The host form is the headline where every case has it (plans and the
    # combine have no host-buffer call).  The host form enqueued eagerly is
    # reported beside them.
    e2e_steps = max(3, min(args.steps, 50))
    host_form = all(r.host_call is not None for r in runners)
    host_refused = None
    for r in runners:                   # warm the eager paths of every case first
        with torch.cuda.stream(stream):
            r.in_block.copy_(r.pinned_in, non_blocking=True)
            r.call()
            r.pinned_out.copy_(r.out_block, non_blocking=True)
            if host_form:
                try:
                    r.host_call()
                except ar.ArError as e:     # e.g. host memory not mapped at its address
                    host_form, host_refused = False, str(e)
    torch.cuda.synchronize()
    for r in runners:
        r.e2e_graphs = {}
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            r.in_block.copy_(r.pinned_in, non_blocking=True)
            r.call()
            r.pinned_out.copy_(r.out_block, non_blocking=True)
        r.e2e_graphs["copies"] = g
        if host_form:
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=stream):
                r.host_call()
            r.e2e_graphs["host"] = g
    for form in list(runners[0].e2e_graphs):    # each form really moves the data
        for r in runners:
            r.pinned_out.zero_()
            r.e2e_graphs[form].replay()
        torch.cuda.synchronize()
        for r in runners:
            if not torch.equal(r.pinned_out, r.out_block.cpu()):
                raise SystemExit("e2e (%s): host outputs differ from the device outputs" % form)
    if ar.ar_status(runners[0].h.h) != ar.AR_OK:
        raise SystemExit("e2e: device status " + ar.ar_strerror(ar.ar_status(runners[0].h.h)))
    e2e_bytes = sum(r.bytes for r in runners)          # one call per case per step

    def round_trips(form: str, graph: bool = True) -> float:
        ms = 0.0
        dist.barrier()
        torch.cuda.synchronize()
        for _ in range(e2e_steps):
            for r in runners:
                with torch.cuda.stream(stream):
                    e0 = torch.cuda.Event(enable_timing=True)
                    e1 = torch.cuda.Event(enable_timing=True)
                    e0.record(stream)
                    if graph:
                        r.e2e_graphs[form].replay()
                    else:
                        r.host_call()
                    e1.record(stream)
                e1.synchronize()
                ms += e0.elapsed_time(e1)
        return dist.max(ms / e2e_steps)

    def rate(ms: float) -> float:
        return dist.sum(e2e_bytes) / (ms * 1e-3) / 1e9

    copies_ms = round_trips("copies")
    if host_form:
        e2e_ms = round_trips("host")
        eager_ms = round_trips("host", graph=False)
        h2d = sum(r.host_bytes[0] for r in runners)
        d2h = sum(r.host_bytes[1] for r in runners)
    else:
        e2e_ms, eager_ms = copies_ms, None
        h2d = sum(r.pinned_in.numel() * r.pinned_in.element_size() for r in runners)
        d2h = sum(r.pinned_out.numel() * r.pinned_out.element_size() for r in runners)
    for r in runners:
        r.e2e_graphs = None
    e2e = {"value": round(rate(e2e_ms), 2), "unit": "GB/s", "h2d_bytes_per_step": h2d,
           "d2h_bytes_per_step": d2h, "ms_per_step": round(e2e_ms, 5),
           "calls_per_step": len(runners), "method": "host" if host_form else "copies",
           "host_call_refused": host_refused,
           "note": ("one all-reduce per case per step through the library's host-buffer call "
                    "(ar_allreduce_host): the kernels read the case's R inputs from page-locked "
                    "host memory and write its outputs to page-locked host memory; one-call "
                    "CUDA graph per case, CUDA events on the stream around each replay; "
                    "minimal bytes of the step's calls / that time"
                    if host_form else
                    "one all-reduce per case per step, each with its own host round trip: "
                    "the inputs copied in from page-locked host memory, the call, the outputs "
                    "copied back, captured as a one-call CUDA graph per case; CUDA events "
                    "around each replay; minimal bytes of the step's calls / that time"),
           "copies": {"value": round(rate(copies_ms), 2), "unit": "GB/s",
                      "ms_per_step": round(copies_ms, 5),
                      "note": "the same round trips with copies: inputs copied in, the "
                              "device-buffer call, outputs copied back (one graph per case)"}}
    if eager_ms is not None:
        e2e["eager"] = {"value": round(rate(eager_ms), 2), "unit": "GB/s",
                        "ms_per_step": round(eager_ms, 5),
                        "note": "the host-buffer call enqueued eagerly, the host's enqueue "
                                "gaps inside the timed events"}

    hbm = None
    if args.workload == "sweep" and not args.no_hbm:
        for r in runners:               # release the sweep's pinned host buffers first
            r.pinned_in = r.pinned_out = None
        hbm = measure_hbm_workloads(stream, bus, peak, dist)

    variants = None
    if args.workload in ("sweep", "decode") and not args.no_variants:
        variants = measure_variants(runners, stream, flush, max(20, args.steps // 10))

    eager = measure_eager(runners, stream, flush)

    cpu = None
    if dist.world == 1 and not args.no_cpu_baseline:
        cpu = cpu_baseline(runners, seconds=args.cpu_seconds)

    launches = args.steps * sum(calls)
    line = {
        "metric": METRIC, "value": round(value, 2), "unit": "GB/s",
        "n_gpus": dist.world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(ms_step, 5), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": runners[0].w.dtype, "data": "synthetic",
        "config": {"workload": desc, "R": runners[0].w.R,
                   "sizes_elems_per_rank": [r.w.n for r in runners],
                   "algo": None if cases[0].get("plan") else cases[0]["algo"],
                   "proto": None if cases[0].get("plan") else cases[0]["proto"],
                   "plan": cases[0].get("plan"),
                   "ll_transport": (args.ll_transport if cases[0]["proto"] == "ll"
                                    and not cases[0].get("plan") else None),
                   "calls_per_graph": cases[0]["calls"],
                   "programmatic_dependent_launch": not args.no_pdl,
                   "l2": ("flushed (256 MiB write) before every graph replay, outside the timed events"
                          if cases[0]["flush"] else "inputs larger than L2 (no flush)"),
                   "bytes_basis": "minimal: 2*R*N*elem_size per call",
                   "parallelism": "replicas" if dist.world > 1 else "single GPU"},
        "roofline": roofline,
        "cpu_baseline": cpu,
        "e2e": e2e,
        "gpu_launches": launches,
        "clocks": clocks, "clocks_remeasured": remeasured,
        "sweep": sweep,
    }
    if hbm is not None:
        line["hbm_workloads"] = hbm
    if variants is not None:
        line["variants_us_per_call"] = variants
    if eager is not None:
        line["eager_us_per_call"] = eager
        if dist.rank == 0:
            print_table(runners, sweep, eager)
    for r in runners:
        r.close()
    return line


# the bandwidth-bound workloads timed after the default sweep: the prefill
# all-reduce (R=16, 128 MiB per rank, bf16, two-shot HB) and the R=32 binary32
# edge case (two-shot HB), each with both two-shot HB stagings
HBM_WORKLOADS = ("prefill", "edge")


def measure_hbm_workloads(stream, bus, peak, dist, replays=20, warmup=3) -> dict:
    """µs/call and minimal-bytes GB/s of the HBM_WORKLOADS, one at a time,
    each with TMA staging and with direct staging (keys `<workload>_tma`,
    `<workload>_direct`; `auto_staging` marks the one AUTO picks): the case's
    single-call graph replayed `warmup` times, then `replays` times with a
    CUDA event pair around each replay, under its own clock sampler.  Inputs
    and outputs (4.3 GB per call) are far larger than L2, so no flush is
    needed.  Each workload's buffers are freed before the next."""
    import torch
    import all_reduce_reduction_gb300 as ar
    out = {}
    for name in HBM_WORKLOADS:
        desc, cases = workload_cases(name)
        c = dict(cases[0])
        r = CaseRunner(c, stream, host_buffers=False)
        auto = staged_path(r, "two_shot_hb")
        for st_name, st in (("tma", ar.AR_HB_STAGING_TMA), ("direct", ar.AR_HB_STAGING_DIRECT)):
            ar.ar_set_hb_staging(r.h.h, st)
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=stream):
                for _ in range(c["calls"]):
                    r.call()
            for _ in range(warmup):
                g.replay()
            torch.cuda.synchronize()
            sampler = ClockSampler(bus)
            sampler.start()
            time.sleep(0.2)
            evs = []
            dist.barrier()
            torch.cuda.synchronize()
            for _ in range(replays):
                with torch.cuda.stream(stream):
                    e0 = torch.cuda.Event(enable_timing=True)
                    e1 = torch.cuda.Event(enable_timing=True)
                    e0.record(stream)
                    g.replay()
                    e1.record(stream)
                evs.append((e0, e1))
            torch.cuda.synchronize()
            dist.barrier()
            time.sleep(0.1)
            clocks = sampler.stop()
            if clocks:
                clocks.pop("series", None)
            stc = ar.ar_status(r.h.h, stream)
            if stc != ar.AR_OK:
                raise RuntimeError("device status after the %s workload: %s"
                                   % (name, ar.ar_strerror(stc)))
            times = [e0.elapsed_time(e1) for e0, e1 in evs]
            calls = c["calls"]
            us = dist.max(sum(times) * 1e3 / (replays * calls))
            gbs = r.bytes / us / 1e3
            key = "two_shot_hb_%s_r%d_n%d_%s" % (st_name, r.w.R, r.w.n, r.w.dtype)
            out["%s_%s" % (name, st_name)] = {
                "workload": desc.replace("staging: auto", "staging: " + st_name),
                "R": r.w.R, "n": r.w.n, "dtype": r.w.dtype,
                "algo": "two_shot", "proto": "hb", "staging": st_name,
                "auto_staging": auto == "two_shot_hb_" + st_name,
                "warmup_calls": warmup * calls, "timed_calls": replays * calls,
                "us_per_call": round(us, 3), **replay_stats(times, calls),
                "min_bytes_per_call": r.bytes, "min_bytes_GBps": round(gbs, 1),
                "peak": peak, "frac_of_hbm_peak": round(gbs / peak, 4),
                "frac_of_nominal": round(gbs / NOMINAL_HBM_GBS, 4),
                "traffic": committed_traffic(key), "kernel": key,
                "l2": "inputs and outputs far larger than L2 (no flush)",
                "clocks": clocks, "clocks_rejected": clocks_rejected(clocks),
            }
            del g
        r.close()
        del r
        torch.cuda.empty_cache()
    return out


def measure_eager(runners, stream, flush, warmup=2, calls=10):
    """µs/call of the same calls launched one by one, without a graph: every
    case warmed first (`warmup` calls each, so no case pays for the idle
    time before this pass), then per case the mean of `calls` calls after
    an L2 flush (informative; not part of `value`)."""
    import torch
    out = {}
    with torch.cuda.stream(stream):
        for r in runners:
            for _ in range(warmup):
                r.call()
    torch.cuda.synchronize()
    for r in runners:
        with torch.cuda.stream(stream):
            flush.fill_(3)
            e0 = torch.cuda.Event(enable_timing=True)
            e1 = torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            for _ in range(calls):
                r.call()
            e1.record(stream)
        e1.synchronize()
        out[str(r.w.n)] = round(e0.elapsed_time(e1) * 1e3 / calls, 3)
    return out


def print_table(runners, sweep, eager):
    """GitHub-style markdown table of the sweep, on stderr (stdout carries
    the one JSON line)."""
    from all_reduce_reduction_gb300 import workload as wl
    rows = ["| msg_size | eager µs/call | graph µs/call | algbw GB/s | busbw GB/s | min-bytes GB/s |",
            "|---|---|---|---|---|---|"]
    for r in runners:
        k = str(r.w.n)
        sw = sweep[k]
        size = r.w.n * wl.ELEM_SIZE[r.w.dtype]
        label = "%d KiB" % (size >> 10) if size < (1 << 20) else "%d MiB" % (size >> 20)
        rows.append("| %s | %.2f | %.2f | %.1f | %.1f | %.1f |" % (
            label, eager[k], sw["us_per_call"], sw["algbw_GBps"], sw["busbw_GBps"],
            sw["min_bytes_GBps"]))
    sys.stderr.write("\n".join(rows) + "\n")


def measure_variants(runners, stream, flush, K):
    """µs/call of the other schedule/protocol pairs at the sweep's sizes
    (informative; not part of `value`)."""
    import torch
    import all_reduce_reduction_gb300 as ar
    out = {}
    for algo, proto, tr, st in (("one_shot", "hb", ar.AR_LL_AUTO, 0), ("two_shot", "hb", ar.AR_LL_AUTO, 0),
                                ("two_shot", "hb", ar.AR_LL_AUTO, ar.AR_HB_STAGING_TMA),
                                ("two_shot", "hb", ar.AR_LL_AUTO, ar.AR_HB_STAGING_DIRECT),
                                ("two_shot", "ll", ar.AR_LL_AUTO, 0),
                                ("one_shot", "ll", ar.AR_LL_GLOBAL, 0),
                                ("one_shot", "ll", ar.AR_LL_CLUSTER, 0),
                                ("auto", "auto", ar.AR_LL_AUTO, 0)):
        row = {}
        for r in runners:
            if algo == "auto" and r.choice is None:
                ar.ar_tune(r.h.h, stream)
            ar.ar_set_ll_transport(r.h.h, tr)
            ar.ar_set_hb_staging(r.h.h, st)
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=stream):
                for _ in range(r.c["calls"]):
                    ar.ar_allreduce(r.h.h, r.ins, r.outs, ar.ALGOS[algo], ar.PROTOS[proto],
                                    stream=stream)
            for _ in range(2):
                g.replay()
            tot = 0.0
            for _ in range(K):
                with torch.cuda.stream(stream):
                    flush.fill_(1)
                    e0 = torch.cuda.Event(enable_timing=True)
                    e1 = torch.cuda.Event(enable_timing=True)
                    e0.record(stream)
                    g.replay()
                    e1.record(stream)
                e1.synchronize()
                tot += e0.elapsed_time(e1)
            row[str(r.w.n)] = round(tot * 1e3 / (K * r.c["calls"]), 3)
            ar.ar_set_ll_transport(r.h.h, r.c.get("transport", ar.AR_LL_AUTO))
            ar.ar_set_hb_staging(r.h.h, r.c.get("staging", ar.AR_HB_STAGING_AUTO))
        key = "%s_%s" % (algo, proto) if algo != "auto" else "auto_tuned"
        if proto == "ll" and algo == "one_shot":
            key += "_" + {ar.AR_LL_GLOBAL: "global", ar.AR_LL_CLUSTER: "cluster"}[tr]
        if st:
            key += "_" + {ar.AR_HB_STAGING_TMA: "tma", ar.AR_HB_STAGING_DIRECT: "direct"}[st]
        out[key] = row
    torch.cuda.synchronize()
    return out


def host_threads() -> int:
    """Host cores this process may run on."""
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count() or 1


def cpu_model() -> str:
    """The host CPU's name: /proc/cpuinfo's model name where it has one (x86),
    else lscpu's (Arm cores list only part numbers in /proc/cpuinfo)."""
    try:
        with open("/proc/cpuinfo") as f:
            for line in f:
                if line.lower().startswith("model name"):
                    return line.split(":", 1)[1].strip()
    except OSError:
        pass
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for line in out.splitlines():
            if line.startswith("Model name:"):
                return line.split(":", 1)[1].strip()
    except (OSError, subprocess.SubprocessError):
        pass
    return platform.machine() or "unknown"


def split_range(n: int, parts: int, align: int):
    """At most `parts` [lo, hi) ranges covering 0..n, each a multiple of
    `align` long except the last."""
    step = max(1, -(-n // max(1, parts)))
    step = -(-step // align) * align
    return [(lo, min(n, lo + step)) for lo in range(0, n, step)]


def oracle_case(lib, case, pool=None, threads=1) -> int:
    """One oracle call over one case's sample; returns its minimal bytes.
    `case` = (workload, combine?, input bit arrays, gate weights or None).
    With a pool the call is split by element range (by token range for the
    combine) over `threads` host threads: the oracle releases the GIL, so
    the unchanged oracle code runs on every core."""
    import oracle
    from all_reduce_reduction_gb300 import workload as wl
    w, combine, ins, wts = case
    dt = wl.DTYPE_CODE[w.dtype]
    if combine:
        T = ins[0].size // w.H
        ranges = split_range(T, threads, 1)

        def part(rg):
            t0, t1 = rg
            oracle.combine([a[t0 * w.H: t1 * w.H] for a in ins], wts[t0 * w.K: t1 * w.K],
                           t1 - t0, w.H, dt, lib=lib)
        nbytes = (len(ins) + 1) * ins[0].nbytes + 4 * T * w.K
    else:
        ranges = split_range(ins[0].size, threads, 64)

        def part(rg):
            oracle.allreduce([a[rg[0]: rg[1]] for a in ins], dt, lib=lib)
        nbytes = 2 * len(ins) * ins[0].nbytes
    if pool is None or len(ranges) == 1:
        for rg in ranges:
            part(rg)
    else:
        list(pool.map(part, ranges))
    return nbytes


def time_oracle(lib, sample, seconds: float, threads: int):
    """Passes over the sample's cases until `seconds` have elapsed; returns
    (GB/s, passes, elapsed seconds)."""
    from concurrent.futures import ThreadPoolExecutor
    pool = ThreadPoolExecutor(threads) if threads > 1 else None
    try:
        done, passes, t0 = 0, 0, time.perf_counter()
        while True:
            for case in sample:
                done += oracle_case(lib, case, pool, threads)
            passes += 1
            if time.perf_counter() - t0 >= seconds:
                break
        dt = time.perf_counter() - t0
    finally:
        if pool is not None:
            pool.shutdown()
    return done / dt / 1e9, passes, dt


def cpu_baseline(runners, seconds: float):
    """The oracle, as it stands, on a bounded sample of the same workload:
    the step's cases one call each, repeated for ~`seconds` on all host
    cores (each call split by element range), then for ~`seconds`/2 on one
    thread."""
    import oracle
    from all_reduce_reduction_gb300 import workload as wl
    lib = oracle.load()
    sample = []
    for r in runners:
        ins = [wl.bits(t) for t in r.cpu_inputs]
        if r.w.n > (1 << 22):           # large messages: a leading slice of every rank
            ins = [a[: 1 << 22].copy() for a in ins]
        combine = bool(r.c.get("combine"))
        wts = r.w.weights() if combine else None
        sample.append((r.w, combine, ins, wts))
    threads = host_threads()
    value, passes, dt = time_oracle(lib, sample, seconds, threads)
    one, passes1, dt1 = time_oracle(lib, sample, seconds / 2, 1)
    sliced = ", first 2^22 elements per rank" if any(r.w.n > (1 << 22) for r in runners) else ""
    return {"value": round(value, 4), "unit": "GB/s", "cores": threads, "kind": "oracle",
            "cpu_model": cpu_model(),
            "sample": "%d passes over the step's %d cases, one call each%s, every call split "
                      "by element range over %d threads (%.1f s)" % (
                          passes, len(sample), sliced, threads, dt),
            "one_thread": {"value": round(one, 4), "cores": 1,
                           "sample": "%d passes, same cases, one thread (%.1f s)" % (passes1, dt1)}}


# ---------------------------------------------------------------------------
# reference arm: the CPU oracle on the host cores
# ---------------------------------------------------------------------------
def run_reference(args, world: int):
    from concurrent.futures import ThreadPoolExecutor
    from all_reduce_reduction_gb300 import workload as wl
    import oracle
    desc, cases = workload_cases(args.workload, args)
    lib = oracle.load()
    sample = []
    for c in cases:
        w = c["w"]
        n = min(w.n, 1 << 20)
        if c.get("combine"):
            n = min(w.T, max(1, (1 << 20) // w.H)) * w.H
        ins = [wl.bits(t) for t in wl.make_inputs(w.config, w.R, n, w.dtype, w.dist)]
        sample.append((w, bool(c.get("combine")), ins, w.weights() if c.get("combine") else None))
    threads = host_threads()
    pool = ThreadPoolExecutor(threads) if threads > 1 else None

    def step():
        return sum(oracle_case(lib, case, pool, threads) for case in sample)

    try:
        for _ in range(args.warmup):
            step()
        t0 = time.perf_counter()
        done = 0
        for _ in range(args.steps):
            done += step()
        dt = time.perf_counter() - t0
    finally:
        if pool is not None:
            pool.shutdown()
    value = done / dt / 1e9
    sample_desc = ("per step: each of the %d cases once (the GPU arm's step runs each %d times)%s; "
                   "every call split by element range over %d threads"
                   % (len(sample), cases[0]["calls"],
                      "; at most 2^20 elements per rank" if any(c["w"].n > (1 << 20) for c in cases)
                      else "", threads))
    return {
        "impl": "reference", "metric": METRIC, "value": round(value, 4), "unit": "GB/s",
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(dt * 1e3 / args.steps, 4), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": cases[0]["w"].dtype, "data": "synthetic",
        "config": {"workload": desc, "R": cases[0]["w"].R,
                   "sizes_elems_per_rank": [c["w"].n for c in cases],
                   "algo": cases[0]["algo"], "proto": cases[0]["proto"]},
        "cpu_baseline": {"value": round(value, 4), "unit": "GB/s", "cores": threads,
                         "kind": "oracle", "cpu_model": cpu_model(), "sample": sample_desc},
        "e2e": {"value": round(value, 4), "unit": "GB/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }


def make_parser() -> argparse.ArgumentParser:
    p = argparse.ArgumentParser()
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=1000)
    p.add_argument("--warmup", type=int, default=10)
    p.add_argument("--workload", default="sweep",
                   choices=["sweep", "decode", "prefill", "edge", "combine", "custom"])
    # --workload custom: one case (used for profiling single kernels)
    p.add_argument("--R", type=int, default=8)
    p.add_argument("--n", type=int, default=1 << 18)
    p.add_argument("--dtype", default="bf16", choices=["bf16", "fp16", "fp32"])
    p.add_argument("--algo", default="one_shot", choices=["one_shot", "two_shot", "auto"])
    p.add_argument("--proto", default="ll", choices=["ll", "hb", "auto"])
    p.add_argument("--calls", type=int, default=10)
    p.add_argument("--plan", default=None, choices=["one_shot", "two_shot"],
                   help="custom workload: run the built-in plan of that algorithm")
    p.add_argument("--plan-chunks", type=int, default=0,
                   help="0: the library's default (ar_plan_builtin)")
    p.add_argument("--plan-ctas", type=int, default=0, help="0: fill the resident capacity")
    p.add_argument("--ll-transport", default="auto", choices=["auto", "global", "cluster"])
    p.add_argument("--staging", default="auto", choices=["auto", "tma", "direct"],
                   help="two-shot HB staging (enum ar_hb_staging)")
    p.add_argument("--grid-divisor", type=int, default=0, choices=[0, 1, 2, 4, 8],
                   help="divisor of every path's CTA cap (ar_set_grid_divisor); 0: tuned or default")
    p.add_argument("--no-pdl", action="store_true",
                   help="launch without programmatic dependent launch")
    p.add_argument("--impl", default="ours", choices=["ours", "reference"])
    p.add_argument("--cpu-seconds", type=float, default=10.0)
    p.add_argument("--only", type=int, default=0,
                   help="run only the workload's case with this many elements per rank")
    p.add_argument("--no-cpu-baseline", action="store_true")
    p.add_argument("--no-variants", action="store_true")
    p.add_argument("--no-hbm", action="store_true",
                   help="default workload: skip the prefill and edge cases timed after the sweep")
    return p


def main():
    args = make_parser().parse_args()
    if args.warmup < 3:
        raise SystemExit("--warmup must be >= 3")

    if args.impl == "reference":
        # rank 0 alone times the oracle; the other ranks exit without work
        if int(os.environ.get("RANK", "0")) == 0:
            print(json.dumps(run_reference(args, int(os.environ.get("WORLD_SIZE", "1")))),
                  flush=True)
        return
    dist = Dist()
    line = run_ours(args, dist)
    if dist.rank == 0:
        print(json.dumps(line), flush=True)
    dist.close()


if __name__ == "__main__":
    main()
