"""Host-side logic of bench.py, on the CPU: the max/sum over ranks with two
gloo processes, the reference arm (alone and under torchrun), and the
parsing of the clock samples."""
import json
import os
import subprocess
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)
import bench  # noqa: E402


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    d = bench.Dist()
    d.barrier()
    q.put((rank, d.max(float(rank + 1) * 1.5), d.sum(10.0 * (rank + 1))))
    d.close()


def test_dist_max_and_sum_two_ranks():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = 29500 + os.getpid() % 2000
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    got = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert got == [(0, 3.0, 30.0), (1, 3.0, 30.0)]


def _lines(out: str):
    return [l for l in out.splitlines() if l.strip().startswith("{")]


def test_reference_arm_line():
    res = subprocess.run([sys.executable, "bench.py", "--impl", "reference", "--steps", "3",
                          "--warmup", "3"], cwd=ROOT, capture_output=True, text=True, timeout=300)
    assert res.returncode == 0, res.stderr
    lines = _lines(res.stdout)
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["unit"] == "GB/s" and d["value"] > 0
    assert d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["value"] == d["value"]
    assert d["e2e"]["h2d_bytes_per_step"] == 0 and d["e2e"]["d2h_bytes_per_step"] == 0
    assert d["higher_is_better"] is True and d["steps"] == 3 and d["warmup"] == 3


def test_reference_arm_under_torchrun_prints_once():
    port = 31000 + os.getpid() % 2000
    res = subprocess.run([sys.executable, "-m", "torch.distributed.run", "--nnodes=1",
                          "--nproc-per-node", "2", "--master-addr", "127.0.0.1",
                          "--master-port", str(port), "bench.py", "--impl", "reference",
                          "--gpus", "2", "--steps", "3", "--warmup", "3"],
                         cwd=ROOT, capture_output=True, text=True, timeout=300)
    assert res.returncode == 0, res.stderr[-2000:]
    lines = _lines(res.stdout)
    assert len(lines) == 1
    assert json.loads(lines[0])["n_gpus"] == 2


def test_warmup_below_three_is_refused():
    res = subprocess.run([sys.executable, "bench.py", "--impl", "reference", "--warmup", "2"],
                         cwd=ROOT, capture_output=True, text=True, timeout=120)
    assert res.returncode != 0


def test_clock_rows():
    hdr = "00000000:1B:00.0, {sm}, 2070, 900.5, 0x0, {a}, Not Active, Not Active, {b}"
    lines = [hdr.format(sm=s, a="Not Active", b="Not Active") for s in (1965, 1980, 1995)]
    lines.append("00000000:2C:00.0, 300, 2070, 100, 0x0, Active, Not Active, Not Active, Not Active")
    c = bench.parse_clock_rows(lines, "1B:00.0")
    assert c == {"sm_mhz": 1980.0, "sm_max_mhz": 2070.0, "reasons": [], "samples": 3,
                 "series": []}
    assert not bench.clocks_rejected(c)
    lines.append(hdr.format(sm=1900, a="Active", b="Active"))
    c = bench.parse_clock_rows(lines, "1B:00.0")
    assert c["reasons"] == ["hw_slowdown", "sw_power_cap"] and bench.clocks_rejected(c)
    low = [hdr.format(sm=900, a="Not Active", b="Not Active")] * 3
    assert bench.clocks_rejected(bench.parse_clock_rows(low, None))
    capped = [hdr.format(sm=1500, a="Not Active", b="Active")] * 3
    assert not bench.clocks_rejected(bench.parse_clock_rows(capped, None))


def test_traffic_lookup_needs_matching_digest():
    d = bench.kernel_source_digest("two_shot_hb_tma_r16_n67108864_bf16")
    assert len(d) == 16
    # the two stagings of the two-shot HB are different kernels
    assert bench.kernel_source_digest("two_shot_hb_direct_r16_n67108864_bf16") not in (d, "unknown")
    assert bench.kernel_source_digest("two_shot_hb_r16_n67108864_bf16") == "unknown"
    assert bench.kernel_source_digest("no_such_kernel") == "unknown"
    assert bench.committed_traffic("no_such_kernel") is None


@pytest.mark.parametrize("n", [0, 1, 63, 64, 65, 1000, 4097 * 4096 + 3])
@pytest.mark.parametrize("parts", [1, 3, 8, 16])
def test_split_range_covers_every_element_once(n, parts):
    rs = bench.split_range(n, parts, 64)
    assert len(rs) <= parts
    assert all(rs[i][1] == rs[i + 1][0] for i in range(len(rs) - 1))      # contiguous
    if n:
        assert rs[0][0] == 0 and rs[-1][1] == n
        assert all((hi - lo) % 64 == 0 for lo, hi in rs[:-1]) and all(hi > lo for lo, hi in rs)
    else:
        assert rs == []


def test_threaded_oracle_timing_runs_every_case():
    import oracle
    from all_reduce_reduction_gb300 import workload as wl
    lib = oracle.load()
    w = wl.SMALL
    ar_case = (w, False, [wl.bits(t) for t in w.inputs()], None)
    cw = wl.COMBINE[1]
    small = wl.CombineWorkload(cw.config, cw.name, cw.K, 3, 64, cw.dtype, cw.dist)
    cb_case = (small, True, [wl.bits(t) for t in small.inputs()], small.weights())
    assert bench.oracle_case(lib, ar_case) == 2 * 8 * 512 * 2
    assert bench.oracle_case(lib, cb_case) == (8 + 1) * 3 * 64 * 2 + 4 * 3 * 8
    gbs, passes, dt = bench.time_oracle(lib, [ar_case, cb_case], 0.05, 3)
    assert gbs > 0 and passes >= 1 and dt >= 0.05


@pytest.mark.parametrize("n", [1, 7, 512, 4097 * 4096 + 3, 8192 * 8192])
@pytest.mark.parametrize("esz", [2, 4])
def test_rank_stride_keeps_every_rank_256_byte_aligned(n, esz):
    st = bench.rank_stride(n, esz)
    assert st >= n and (st * esz) % 256 == 0 and (st - n) * esz < 256


def test_digest_ignores_comments_but_not_code():
    src = 'int a = 1; // note\n/* block */ asm("ld.global.u32 %0, [%1]; // not a comment");\n'
    assert bench.strip_comments(src) == bench.strip_comments(src.replace("note", "other words"))
    assert "// not a comment" in bench.strip_comments(src)
    assert bench.strip_comments(src) != bench.strip_comments(src.replace("a = 1", "a = 2"))


def test_ll_wire_bytes_count_packets():
    import types
    import all_reduce_reduction_gb300 as ar

    def runner(algo, proto, n, dtype="bf16", R=8, **extra):
        w = types.SimpleNamespace(R=R, n=n, dtype=dtype)
        return types.SimpleNamespace(c=dict(algo=algo, proto=proto, **extra), choice=None, w=w)
    # whole packets: inputs + outputs 2RNs, packets stored and loaded 2 x 2RNs
    assert bench.ll_wire_bytes(runner("one_shot", "ll", 1 << 18)) == 6 * 8 * (1 << 19)
    # a partial last packet still travels as 8 bytes
    assert bench.ll_wire_bytes(runner("one_shot", "ll", 513)) == 8 * (2 * 1026 + 2 * 8 * 257)
    assert bench.ll_wire_bytes(runner("one_shot", "ll", 3, "fp32", 2)) == 2 * (2 * 12 + 2 * 24)
    # other paths report only the minimal bytes
    assert bench.ll_wire_bytes(runner("two_shot", "ll", 1024)) is None
    assert bench.ll_wire_bytes(runner("one_shot", "hb", 1024)) is None
    assert bench.ll_wire_bytes(runner("one_shot", "ll", 1024, transport=ar.AR_LL_CLUSTER)) is None


def test_cpu_model_is_named():
    name = bench.cpu_model()
    assert isinstance(name, str) and name.strip()


def test_function_source_takes_definitions_not_calls():
    src = bench.strip_comments(
        "int g(int x); int h() { return g(1); }\n"
        "int g(int x) { if (x) { return 1; } return 0; }  // done\n"
        "int gg(int x) { return x; }")
    assert bench.function_source(src, "g") == "g(int x) { if (x) { return 1; } return 0; }"
    assert bench.function_source(src, "gg") == "gg(int x) { return x; }"
    with pytest.raises(KeyError):
        bench.function_source(src, "missing")


def test_digest_follows_only_the_named_kernels(tmp_path, monkeypatch):
    import shutil
    csrc = os.path.join(bench.ROOT, "all_reduce_reduction_gb300", "csrc")
    copy = tmp_path / "all_reduce_reduction_gb300" / "csrc"
    shutil.copytree(csrc, copy)
    one = bench.kernel_source_digest("one_shot_ll_global_r8_n1_bf16")
    two = bench.kernel_source_digest("two_shot_ll_r8_n1_bf16")
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    assert bench.kernel_source_digest("one_shot_ll_global_r8_n1_bf16") == one
    src = (copy / "ar_ll.cu").read_text()
    # a change inside the two-shot kernel leaves the one-shot digest alone
    i = src.index("k_ll2_staged(const __grid_constant__")
    j = src.index("const uint32_t tid = threadIdx.x;", i)
    (copy / "ar_ll.cu").write_text(src[:j] + "const uint32_t tid = threadIdx.x + 0;" +
                                   src[j + len("const uint32_t tid = threadIdx.x;"):])
    assert bench.kernel_source_digest("one_shot_ll_global_r8_n1_bf16") == one
    assert bench.kernel_source_digest("two_shot_ll_r8_n1_bf16") != two
    # a change to a helper before the kernels reaches both
    (copy / "ar_ll.cu").write_text(src.replace("ld.global.L1::no_allocate.v2.u32",
                                               "ld.global.v2.u32", 1))
    assert bench.kernel_source_digest("one_shot_ll_global_r8_n1_bf16") != one


def test_workloads_match_the_configurations():
    """The bench's workloads have the sizes, dtypes and value recipes of the
    configurations they stand for, and the algorithmic bytes 2*R*N*s."""
    _, sweep = bench.workload_cases("sweep")
    assert [(c["w"].R, c["w"].n, c["w"].dtype, c["w"].dist) for c in sweep] == \
        [(8, 1 << i, "bf16", "uniform") for i in range(9, 19)]
    assert all(c["algo"] == "one_shot" and c["proto"] == "ll" and c["calls"] == 10 and c["flush"]
               for c in sweep)
    assert [bench.case_bytes(c) for c in sweep] == [2 * 8 * (1 << i) * 2 for i in range(9, 19)]
    _, decode = bench.workload_cases("decode")
    assert [(c["w"].R, c["w"].n, c["w"].dist) for c in decode] == \
        [(8, 8192 * b, "normal") for b in (1, 8, 32, 128, 256)]
    _, prefill = bench.workload_cases("prefill")
    (p,) = prefill
    assert (p["w"].R, p["w"].n, p["w"].dtype, p["algo"], p["proto"], p["flush"]) == \
        (16, 8192 * 8192, "bf16", "two_shot", "hb", False)
    assert bench.case_bytes(p) == 4 << 30                  # 4 GiB per call, far above L2
    _, edge = bench.workload_cases("edge")
    (e,) = edge
    assert (e["w"].R, e["w"].n, e["w"].dtype, e["w"].dist) == (32, 4097 * 4096 + 3, "fp32",
                                                               "loguniform")
    assert bench.case_bytes(e) == 2 * 32 * (4097 * 4096 + 3) * 4
    _, comb = bench.workload_cases("combine")
    assert [(c["w"].K, c["w"].T, c["w"].H) for c in comb] == [(8, t, 8192) for t in (1, 16, 128, 4096)]
    assert bench.case_bytes(comb[-1]) == 9 * 4096 * 8192 * 2 + 4 * 4096 * 8


def test_clock_rows_with_timestamps_bin_by_replay_window():
    """Rows carrying nvidia-smi's timestamp give a (time, MHz) series; each
    replay window takes the sample nearest its middle, if one is close."""
    row = ("00000000:1B:00.0, {sm}, 2070, 900.5, 0x0, Not Active, Not Active, Not Active, "
           "Not Active, 2026/12/03 05:29:{sec}")
    lines = [row.format(sm=m, sec=t) for m, t in ((2070, "26.000"), (1800, "26.050"),
                                                   (1500, "26.100"), (2070, "27.500"))]
    c = bench.parse_clock_rows(lines, "1B:00.0")
    t0 = bench.parse_smi_time("2026/12/03 05:29:26.000")
    assert [round(t - t0, 3) for t, _ in c["series"]] == [0.0, 0.05, 0.1, 1.5]
    assert [m for _, m in c["series"]] == [2070.0, 1800.0, 1500.0, 2070.0]
    win = [(t0 + 0.045, t0 + 0.055), (t0 + 0.095, t0 + 0.101), (t0 + 0.8, t0 + 0.801)]
    got = bench.clocks_for_windows(c["series"], win)
    assert got == {"sm_mhz_median": 1650.0, "replays_with_sample": 2}
    assert bench.clocks_for_windows([], win) == {"sm_mhz_median": None, "replays_with_sample": 0}
    assert bench.parse_smi_time("not a time") is None


def test_replay_stats():
    # replays of 10 calls: 30..39 us per replay -> 3.0..3.9 us per call
    st = bench.replay_stats([(30 + i) * 1e-3 for i in (9, 0, 5, 1, 8, 2, 7, 3, 6, 4)], 10)
    assert st == {"us_p50": 3.45, "us_p90": 3.8, "us_min": 3.0, "us_max": 3.9, "replays": 10}
    assert bench.replay_stats([0.005], 1) == {"us_p50": 5.0, "us_p90": 5.0, "us_min": 5.0,
                                              "us_max": 5.0, "replays": 1}
    assert bench.replay_stats([], 10) == {}


def test_bench_options_parse():
    a = bench.make_parser().parse_args(["--no-hbm", "--steps", "3", "--warmup", "3"])
    assert a.no_hbm and a.workload == "sweep" and a.staging == "auto"
    assert bench.HBM_WORKLOADS == ("prefill", "edge")
    b = bench.make_parser().parse_args(["--workload", "custom", "--staging", "tma"])
    assert bench.STAGINGS[b.staging] == 1
    desc, _ = bench.workload_cases("custom", b)
    assert "staging: tma" in desc
