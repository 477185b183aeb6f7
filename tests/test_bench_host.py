"""Host-side logic of bench.py (no GPU): the FLOP and byte counts it reports, and
its multi-rank path -- max-over-ranks timing and whole-job throughput -- run as two
gloo ranks on the CPU."""
from __future__ import annotations

import os
import socket

import numpy as np
import torch.multiprocessing as mp

import bench
from split_kv_attention_flash_gb300 import workloads as wl


def test_flop_counts_of_the_workloads():
    # 2 * Sq * Sk_visible * H * (D_QK + D_V) over visible (query, key) pairs
    assert bench.flops_of(wl.TARGET_SHAPE) == 2 * 4096 * 42700 * 12 * 320
    assert abs(bench.flops_of(wl.LONG_VARLEN) - 7.7856768e12) < 1e3
    assert bench.flops_of(wl.TINY_CAUSAL) == 2 * 2 * (64 * 65 // 2) * 128
    causal = bench.flops_of(wl.MASKED_F16)                      # keys <= min(q, 3000)
    assert causal == 2 * 16 * 256 * (2048 * 2049 // 2)
    prefix = bench.flops_of(wl.MASKED_F16.with_(mask=wl.MASK_PREFIX_CAUSAL, prefix_offset=2048))
    vis = np.minimum(np.arange(2048) + 2048, 3000) + 1
    assert prefix == 2 * 16 * 256 * int(vis.sum())
    fully_masked = wl.MASKED_F16.with_(mask=wl.MASK_PREFIX_CAUSAL, prefix_offset=-256)
    assert bench.flops_of(fully_masked) == 2 * 16 * 256 * sum(max(0, q - 256 + 1) for q in range(2048))


def test_flop_count_with_window_and_padding():
    w = wl.Workload("w", H=1, seqlens_q=(10,), seqlens_k=(20,), d_qk=64, d_v=64, dtype="bf16",
                    seed=0, mask=wl.MASK_PREFIX_CAUSAL, prefix_offset=5, window_left=3,
                    seqused_k=(12,))
    vis = sum(len([j for j in range(12) if q + 5 - 3 <= j <= q + 5]) for q in range(10))
    assert bench.flops_of(w) == 2 * vis * 128


def test_combine_bytes():
    w = wl.TARGET_SHAPE
    counts = np.full(w.total_q, 3, dtype=np.int32)
    b = bench.combine_bytes(w, counts, with_lse=False)
    assert b == w.H * w.total_q * (3 * (4 * 128 + 4) + 128 * 2) + 4 * w.total_q


def test_pages_baseline_figure():
    # the split-3 time printed for this shape (2.269 ms) as TFLOP/s
    assert abs(bench.PAGES_SPLIT3_TFLOPS - 591.99) < 0.1


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, queue):
    import torch.distributed as dist
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        local = [1.0 + rank, 5.0 - 2 * rank]          # per-rank step and e2e times, ms
        ms, e2e = bench.max_over_ranks(local)
        dist.barrier()
        queue.put((rank, ms, e2e, bench.whole_job_tflops(1e12, world, ms)))
    finally:
        dist.destroy_process_group()


def test_max_over_ranks_with_two_gloo_ranks():
    ctx = mp.get_context("spawn")
    queue = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, queue)) for r in range(2)]
    for p in procs:
        p.start()
    results = sorted(queue.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, ms, e2e, tflops in results:
        assert ms == 2.0 and e2e == 5.0            # both ranks see the slowest rank
        assert abs(tflops - 2 * 1e12 / 2e-3 / 1e12) < 1e-9


def test_single_process_is_identity():
    assert bench.max_over_ranks([3.0, 4.5]) == [3.0, 4.5]


def test_reference_arm_runs_on_rank_zero_only():
    class Args:
        workload, steps, warmup, cpu_seconds, gpus = "tiny", 1, 3, 1.0, 2
    assert bench.run_reference(Args, rank=1) is None


def test_recorded_traffic_lines_name_existing_sources():
    """Every profiles/traffic.txt line names sources that exist; a line whose sources still
    hash to its recorded prefix yields its bytes (scaled for another workload), any other
    line yields None rather than a stale number."""
    path = os.path.join(bench.ROOT, "profiles", "traffic.txt")
    for line in open(path):
        f = dict(kv.split("=", 1) for kv in line.split() if "=" in kv)
        srcs = f["source"].split(",")
        assert all(os.path.exists(os.path.join(bench.ROOT, s)) for s in srcs)
        got = bench.recorded_traffic(f["kernel"], f["workload"])
        if bench.sources_sha(srcs) == f["sha256"]:
            assert got == float(f["dram_bytes_per_launch"])
        else:
            assert got is None
    assert bench.recorded_traffic("partial_tc", "no such workload") is None


def test_vs_baseline_only_for_the_pages_workload():
    assert abs(bench.vs_pages("target", bench.PAGES_SPLIT3_TFLOPS) - 1.0) < 1e-12
    for name in wl.ALL:
        if name != "target":
            assert bench.vs_pages(name, 123.0) is None


def test_roofline_bound_follows_the_arithmetic_intensity():
    peaks = {"bf16": 1890.1, "hbm": 6770.5}
    for name, hbm in (("target", False), ("varlen", False), ("decode", True), ("decode_mq", True),
                      ("decode_small", True)):
        w = wl.ALL[name]
        assert bench.hbm_bound(bench.flops_of(w), bench.kv_bytes_of(w), peaks) == hbm, name


def test_code_hash_ignores_comments_and_whitespace():
    a = "int f(int x) {\n    return x + 1;  // one more\n}\n/* block\n   comment */\n"
    b = "int f(int x) { return x + 1; }\n"
    c = "int f(int x) { return x + 2; }\n"
    assert bench.code_text(a) == bench.code_text(b)
    assert bench.code_text(b) != bench.code_text(c)


def test_roofline_entry_reports_burst_and_sustained_fractions():
    peaks = {"bf16": 1890.1, "bf16_sustained": 1692.7, "hbm": 6770.5, "source": "measured"}
    w = wl.TARGET_SHAPE
    fl = bench.flops_of(w)
    loop = {"mean_ms": 0.8, "median_ms": 0.79, "launches": 1250, "seconds": 1.0}
    r = bench.roofline_of(w, "partial_tc", fl, loop, peaks, None, {"sm_mhz": 2000})
    assert r["bound"] == "tensor" and r["unit"] == "TFLOP/s"
    assert abs(r["achieved"] - fl / 0.8e-3 / 1e12) < 1e-6
    assert abs(r["frac"] - r["achieved"] / 1890.1) < 1e-12
    assert abs(r["frac_sustained"] - r["achieved"] / 1692.7) < 1e-12
    d = bench.roofline_of(wl.DECODE, "partial_tc", bench.flops_of(wl.DECODE), loop, peaks, None, {})
    assert d["bound"] == "hbm" and d["unit"] == "GB/s"
    assert abs(d["achieved"] - bench.kv_bytes_of(wl.DECODE) / 0.8e-3 / 1e9) < 1e-6
