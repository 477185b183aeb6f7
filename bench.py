"""Benchmark of the split-KV attention forward on GB300.

One step = one sk_attn_fwd over the workload (partial kernel -> combine, which
evaluates the split-count formula itself), inputs resident in HBM. Default workload: the long-context varlen
prefill target shape (bf16, Sq 4096, Sk 42700, H 12, D_QK 192, D_V 128,
non-causal, split_kv automatic -> 3). Inputs (347 MB) are larger than L2.

Prints one JSON line. Besides the step throughput it reports, measured live:
  roofline      the partial kernel's TFLOP/s (CUDA events on its stream) against
                the measured dense bf16 peak, plus ncu DRAM traffic from profiles/
  combine       the combine kernel's HBM GB/s (back-to-back launches over rotating copies of
                the partials that together exceed L2 three times)
  e2e           the same metric through the library's host-buffer call (sk_attn_fwd_host),
                host<->device copies inside the timed region (steps alternate between two
                streams, so one step's copies overlap the other's compute)
  cpu_baseline  the CPU oracle on a bounded sample of the same workload
  clocks        nvidia-smi samples taken during the timed work

--impl reference times the CPU oracle as the reference arm (rank 0 only).
Multi-GPU (torchrun): every rank runs the same workload (replicas, weak scaling),
barrier + max-over-ranks timing, value = all ranks' FLOPs / that time.
"""
from __future__ import annotations

import argparse
import hashlib
import re
import json
import os
import statistics
import subprocess
import sys
import time

import numpy as np
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from split_kv_attention_flash_gb300 import workloads as wl  # noqa: E402

METRIC = "split-KV attn fwd TFLOP/s (bf16, Sq4096 Sk42.7K H12); combine HBM GB/s"
UNIT = "TFLOP/s"
# The pages' split-3 time on MI325X for this exact shape (2.269 ms) as TFLOP/s.
PAGES_SPLIT3_TFLOPS = 2 * 4096 * 42700 * 12 * (192 + 128) / 2.269e-3 / 1e12
L2_BYTES = 129 * 1024 * 1024


def vs_pages(workload: str, value: float):
    """value / the pages' split-3 throughput, for the one workload the pages time (the
    target shape); None for every other workload."""
    return value / PAGES_SPLIT3_TFLOPS if workload == "target" else None


def flops_of(w, rows=None) -> float:
    """4 * Sq * Sk_visible * H * (D_QK + D_V) / 2 over visible (row, key) pairs."""
    total = 0
    for b in range(w.B):
        sq, sk = w.seqlens_q[b], w.seqlens_k[b]
        if w.seqused_k is not None:
            sk = min(sk, max(w.seqused_k[b], 0))
        last = sk - 1 if w.last_valid_kv_index < 0 else min(w.last_valid_kv_index, sk - 1)
        qs = np.arange(sq) if rows is None else np.asarray(
            [r - w.cu_seqlens_q[b] for r in rows if w.cu_seqlens_q[b] <= r < w.cu_seqlens_q[b + 1]])
        if len(qs) == 0:
            continue
        if w.mask == wl.MASK_NONE:
            vis = np.full(len(qs), last + 1)
        else:
            off = w.prefix_offset if w.mask == wl.MASK_PREFIX_CAUSAL else 0
            hi = np.minimum(qs + off, last)
            lo = np.maximum(qs + off - w.window_left, 0) if w.window_left >= 0 else 0
            vis = np.clip(hi - lo + 1, 0, None)
        total += int(vis.sum())
    return 2.0 * total * w.H * (w.d_qk + w.d_v)


def combine_bytes(w, counts: np.ndarray, with_lse: bool) -> float:
    es = 2 if w.dtype != "f32" else 4
    per_row = counts.astype(np.int64) * (4 * w.d_v + 4) + w.d_v * es + (4 if with_lse else 0)
    return float(per_row.sum() * w.H + 4 * w.total_q)


def max_over_ranks(values, device=None) -> list:
    """Element-wise maximum of `values` over all ranks (identity without a process
    group). The slowest rank's time is the job's time."""
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()):
        return [float(v) for v in values]
    t = torch.tensor([float(v) for v in values], dtype=torch.float64,
                     device=device if device is not None else "cpu")
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return [float(v) for v in t.tolist()]


def whole_job_tflops(flop_per_rank: float, world: int, ms: float) -> float:
    """Throughput of the whole job: every rank's FLOPs over the slowest rank's time."""
    return world * flop_per_rank / (ms * 1e-3) / 1e12


def measured_peaks() -> dict:
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        d = json.load(open(path))
        return {"hbm": d["hbm_gbs"], "bf16": d["bf16_tflops"],
                "bf16_sustained": d.get("bf16_tflops_sustained"), "source": "measured"}
    return {"hbm": 6800.0, "bf16": 1900.0, "bf16_sustained": 1700.0, "source": "fallback"}


def code_text(text: str) -> str:
    """C / C++ source without its comments, whitespace collapsed: what the compiler sees,
    so that editing a comment does not retire a measurement of unchanged code."""
    text = re.sub(r"/\*.*?\*/", " ", text, flags=re.S)
    text = re.sub(r"//[^\n]*", " ", text)
    return " ".join(text.split())


def sources_sha(paths: list[str]) -> str | None:
    """sha256 prefix of the concatenated code of the files (a kernel's source and the
    headers it includes, comments stripped), or None when one is missing."""
    h = hashlib.sha256()
    for rel in paths:
        src = os.path.join(ROOT, rel)
        if not os.path.exists(src):
            return None
        h.update(code_text(open(src, encoding="utf-8").read()).encode())
        h.update(b"\0")
    return h.hexdigest()[:16]


def recorded_traffic(kernel: str, workload: str):
    """DRAM bytes per launch from a committed ncu summary (profiles/traffic.txt), valid
    only while the kernel's sources are unchanged (the sha256 prefix of its source and
    headers, `source=` a comma-separated list, is recorded beside the number). A line
    for another workload of the same kernel carries `scale_<workload>=` factors when
    the traffic grows in proportion to the work."""
    path = os.path.join(ROOT, "profiles", "traffic.txt")
    if not os.path.exists(path):
        return None
    for line in open(path):
        f = dict(kv.split("=", 1) for kv in line.split() if "=" in kv)
        if f.get("kernel") != kernel or "source" not in f:
            continue
        if f.get("workload") == workload:
            scale = 1.0
        elif f"scale_{workload}" in f:
            scale = float(f[f"scale_{workload}"])
        else:
            continue
        if sources_sha(f["source"].split(",")) != f.get("sha256"):
            return None
        return float(f["dram_bytes_per_launch"]) * scale
    return None


def hbm_bound(flop: float, kv_bytes: float, peaks: dict) -> bool:
    """Whether the partial kernel's roofline is HBM: fewer FLOPs per byte of K and V than
    the ratio of the measured bf16 peak to the measured HBM copy bandwidth (decode shapes,
    a few queries per sequence), rather than the tensor cores (prefill shapes)."""
    return flop / max(kv_bytes, 1.0) < peaks["bf16"] * 1e12 / (peaks["hbm"] * 1e9)


def kv_bytes_of(w) -> float:
    """Bytes of K and V a streaming kernel reads once: every used key of every head."""
    keys = 0
    for b in range(w.B):
        sk = w.seqlens_k[b] if w.seqused_k is None else min(w.seqlens_k[b], max(w.seqused_k[b], 0))
        keys += sk
    return float(keys * w.H * (w.d_qk + w.d_v) * (4 if w.dtype == "f32" else 2))


class ClockSampler:
    """nvidia-smi samples (every 50 ms) of one GPU while the `with` block runs. Entering
    waits (up to 5 s) for the first sample, so that a loop of about a second is sampled
    from its start."""
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,utilization.gpu,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index: int, keep_first: bool = False, trailing: bool = False):
        self.idx = device_index
        self.proc = None
        self.lines = []
        self.keep_first = keep_first  # keep the samples taken before the work started
        self.trailing = trailing      # wait for one sample after the work (short loops)

    def _read(self):
        for line in self.proc.stdout:
            if line.strip():
                self.lines.append(line)

    def __enter__(self):
        import threading
        self.lines = []
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.idx}", f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "50"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
            return self
        self.reader = threading.Thread(target=self._read, daemon=True)
        self.reader.start()
        t0 = time.time()
        while not self.lines and time.time() - t0 < 5.0 and self.proc.poll() is None:
            time.sleep(0.01)
        self.first = 0 if self.keep_first else len(self.lines)
        return self

    def __exit__(self, *exc):
        if self.proc is not None:
            if self.trailing:
                n, t0 = len(self.lines), time.time()
                while len(self.lines) == n and time.time() - t0 < 1.0 and self.proc.poll() is None:
                    time.sleep(0.005)
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
                self.proc.wait()
            self.reader.join(timeout=5)
            self.lines = self.lines[self.first:]

    def summary(self):
        rows = []
        for l in self.lines:
            f = [x.strip() for x in l.split(",")]
            try:
                rows.append((float(f[1]), float(f[2]), float(f[4]), f[5:9]))
            except (ValueError, IndexError):
                continue
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"], "samples": 0}
        loaded = [r for r in rows if r[2] >= 50] or rows
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in loaded for i, v in enumerate(r[3]) if v == "Active"})
        return {"sm_mhz": statistics.median(r[0] for r in loaded),
                "sm_max_mhz": max(r[1] for r in rows), "reasons": reasons,
                "samples": len(loaded)}


# ------------------------------------------------------------------ CPU oracle

def time_oracle(w, target_s: float, seed: int = 0, inputs=None):
    """The oracle, as it is, on a bounded random sample of rows (all heads)."""
    import oracle
    q, k, v = inputs if inputs is not None else w.make_inputs("cpu")
    prob = oracle.Problem(cu_q=w.cu_seqlens_q, cu_k=w.cu_seqlens_k, H=w.H, d_qk=w.d_qk,
                          d_v=w.d_v, mask=w.mask, prefix_offset=w.prefix_offset,
                          last_valid_kv_index=w.last_valid_kv_index, n_per_block=w.n_per_block)
    cores = os.cpu_count() or 1
    rng = np.random.default_rng(seed)
    n = max(cores, 16)
    rows = np.sort(rng.choice(w.total_q, size=n, replace=False)).astype(np.int32)
    t0 = time.perf_counter()
    oracle.attention(prob, q, k, v, rows=rows, nthreads=cores)
    dt = time.perf_counter() - t0
    n2 = int(min(w.total_q, max(n, n * target_s / max(dt, 1e-3))))
    n2 = max(cores, (n2 // cores) * cores)
    rows = np.sort(rng.choice(w.total_q, size=n2, replace=False)).astype(np.int32)
    t0 = time.perf_counter()
    oracle.attention(prob, q, k, v, rows=rows, nthreads=cores)
    dt = time.perf_counter() - t0
    fl = flops_of(w, rows.tolist())
    return {"value": fl / dt / 1e12, "unit": UNIT, "cores": cores, "kind": "oracle",
            "sample": f"{n2} random query rows x {w.H} heads of {w.name} "
                      f"({fl:.3g} FLOP in {dt:.1f} s, f64, {cores} threads)"}


# ------------------------------------------------------------------- our arm

def timed_chunks(run_chunk, per_chunk: int, min_s: float, stream) -> dict:
    """Back-to-back chunks of `per_chunk` launches for at least `min_s` seconds of device
    time, each chunk bracketed by CUDA events on `stream`; the host enqueues every chunk
    before it waits. mean_ms = total time / launches (the average launch duration);
    median_ms = median over chunks of the chunk's time per launch."""
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    e0.record(stream)
    run_chunk()
    e1.record(stream)
    torch.cuda.synchronize()
    n = max(10, int(min_s / max(e0.elapsed_time(e1) * 1e-3, 1e-6)) + 1)
    evs = [torch.cuda.Event(enable_timing=True) for _ in range(n + 1)]
    evs[0].record(stream)
    for i in range(n):
        run_chunk()
        evs[i + 1].record(stream)
    torch.cuda.synchronize()
    ms = [evs[i].elapsed_time(evs[i + 1]) for i in range(n)]
    return {"mean_ms": sum(ms) / (n * per_chunk), "median_ms": statistics.median(ms) / per_chunk,
            "launches": n * per_chunk, "seconds": sum(ms) * 1e-3}


def time_back_to_back(launch, min_s: float, stream, rotate: int = 1) -> dict:
    """Device time per launch of `launch(i)` (i picks one of `rotate` buffer sets) run back
    to back for at least `min_s` seconds. Launches shorter than 0.2 ms are captured into a
    CUDA graph of a few milliseconds of launches and replayed, so that the host's call
    overhead (a ctypes call takes some 10-20 us) cannot leave gaps between them."""
    for i in range(3):
        launch(i % rotate)
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    launch(0)
    e1.record(stream)
    torch.cuda.synchronize()
    one_ms = e0.elapsed_time(e1)
    if one_ms < 0.2:
        per = max(rotate, int(2.0 / max(one_ms, 1e-3)))
        per = rotate * -(-per // rotate)
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph):
            for i in range(per):
                launch(i % rotate)
        graph.replay()
        r = timed_chunks(graph.replay, per, min_s, stream)
        r["graph_launches"] = per
        del graph
        return r
    state = {"i": 0}

    def one():
        launch(state["i"] % rotate)
        state["i"] += 1
    return timed_chunks(one, 1, min_s, stream)


def roofline_of(w, kname: str, fl: float, loop: dict, peaks: dict, traffic, clocks) -> dict:
    """The partial kernel's roofline entry: tensor-bound (TFLOP/s against the measured dense
    bf16 peak, burst and sustained) for prefill shapes, HBM-bound (K and V bytes per second
    against the measured copy bandwidth) for decode shapes."""
    ms = loop["mean_ms"]
    common = {"kernel": kname, "ms_per_launch": ms, "ms_per_launch_median": loop["median_ms"],
              "launches": loop["launches"], "seconds": loop["seconds"], "traffic": traffic,
              "clocks": clocks}
    if hbm_bound(fl, kv_bytes_of(w), peaks):   # a stream over K and V: bound by HBM
        gbs = kv_bytes_of(w) / (ms * 1e-3) / 1e9
        return {"bound": "hbm", "achieved": gbs, "peak": peaks["hbm"], "unit": "GB/s",
                "frac": gbs / peaks["hbm"], "peak_source": f"{peaks['source']} HBM copy",
                "bytes_per_launch": kv_bytes_of(w), **common}
    tf = fl / (ms * 1e-3) / 1e12
    out = {"bound": "tensor", "achieved": tf, "peak": peaks["bf16"], "unit": "TFLOP/s",
           "frac": tf / peaks["bf16"], "peak_source": f"{peaks['source']} dense bf16 burst",
           "flop_per_launch": fl, **common}
    if peaks.get("bf16_sustained"):
        out["peak_sustained"] = peaks["bf16_sustained"]
        out["frac_sustained"] = tf / peaks["bf16_sustained"]
    return out


def kernel_blocks(skv, w, p, q, k, v, S: int, kname: str, peaks: dict, min_s: float, dev, stream):
    """The partial kernel alone and the combine alone, each timed back to back for at least
    `min_s` seconds with the clocks sampled during its loop. The combine runs over rotating
    copies of the partials that together exceed L2 three times, so that every launch reads
    its inputs from HBM."""
    fl = flops_of(w)
    o_part = torch.empty(w.H, S, w.total_q, w.d_v, dtype=torch.float32, device=dev)
    l_part = torch.empty(w.H, S, w.total_q, dtype=torch.float32, device=dev)
    with ClockSampler(dev.index) as cs:
        loop = time_back_to_back(lambda i: skv.sk_attn_partial_fwd(p, q, k, v, o_part, l_part),
                                 min_s, stream)
    roof = roofline_of(w, kname, fl, loop, peaks, None, cs.summary())
    comb = None
    counts = torch.empty(w.total_q, dtype=torch.int32, device=dev)
    skv.sk_valid_split_counts(p, counts)
    if S > 1:
        out = torch.empty(w.total_q, w.H, w.d_v, dtype=q.dtype, device=dev)
        part_bytes = (o_part.numel() + l_part.numel()) * 4
        n_copies = max(2, -(-3 * L2_BYTES // max(part_bytes, 1)))
        copies = [(o_part, l_part)] + [(o_part.clone(), l_part.clone()) for _ in range(n_copies - 1)]
        with ClockSampler(dev.index) as cs:
            cl = time_back_to_back(lambda i: skv.sk_combine(p, *copies[i], counts, out, None),
                                   min_s, stream, rotate=n_copies)
        cbytes = combine_bytes(w, counts.cpu().numpy(), with_lse=False)
        gbs = cbytes / (cl["mean_ms"] * 1e-3) / 1e9
        comb = {"achieved": gbs, "unit": "GB/s", "peak": peaks["hbm"], "frac": gbs / peaks["hbm"],
                "bytes": cbytes, "us_per_launch": cl["mean_ms"] * 1e3,
                "us_per_launch_median": cl["median_ms"] * 1e3, "launches": cl["launches"],
                "seconds": cl["seconds"], "clocks": cs.summary(),
                "l2": f"back-to-back launches (CUDA graph of {cl.get('graph_launches', 1)}) over "
                      f"{n_copies} rotating partial copies >= 3x L2"}
        del copies
    return roof, comb, counts


def run_ours(args, rank: int, world: int, dist_on: bool):
    import split_kv_attention_flash_gb300 as skv
    from split_kv_attention_flash_gb300 import _build
    if rank == 0 or not dist_on:
        _build.build()
    if dist_on:
        torch.distributed.barrier()
    dev = torch.device("cuda", int(os.environ.get("LOCAL_RANK", 0)))
    torch.cuda.set_device(dev)
    w = wl.ALL[args.workload]
    if args.split is not None:
        w = w.with_(split_kv=args.split)
    q, k, v = w.make_inputs(dev)
    p = skv.params_for(w, dev)
    S = skv.sk_auto_split_kv(p)
    p.split_kv = S
    p.fuse_combine = int(args.fuse_combine)
    out = torch.empty(w.total_q, w.H, w.d_v, dtype=q.dtype, device=dev)
    lse = None
    ws = torch.empty(max(skv.sk_workspace_bytes(p), 1), dtype=torch.uint8, device=dev)
    kname = skv.sk_partial_kernel_name(p, q, k, v)
    fl = flops_of(w)
    stream = torch.cuda.current_stream()
    peaks = measured_peaks()

    def step():
        skv.sk_attn_fwd(p, q, k, v, out, lse, ws)

    fused = bool(p.fuse_combine) and kname.startswith("partial_tc") and S <= 8
    launches_per_step = 1 if S == 1 or fused else 2   # partial, combine
    # the timed steps may last only milliseconds: keep every sample from the warm-up on and
    # one taken right after the last step
    sampler = ClockSampler(dev.index, keep_first=True, trailing=True)
    with sampler:
        for _ in range(args.warmup):
            step()
        torch.cuda.synchronize()
        if dist_on:
            torch.distributed.barrier()
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(args.steps):
            step()
        e1.record(stream)
        torch.cuda.synchronize()
        if dist_on:
            torch.distributed.barrier()
        ms = e0.elapsed_time(e1) / args.steps
    clocks = sampler.summary()
    if args.step_only:  # profiling runs: the timed steps and nothing else
        ms = max_over_ranks([ms], device=dev if dist_on else None)[0]
        if rank != 0:
            return None
        return {"metric": METRIC, "value": whole_job_tflops(fl, world, ms), "unit": UNIT,
                "n_gpus": world, "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms,
                "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
                "dtype": "bf16" if w.dtype == "bf16" else w.dtype, "data": "synthetic",
                "config": {**shape_config(w), "split_kv": S, "step_only": True},
                "gpu_launches": launches_per_step * args.steps, "clocks": clocks}

    # the dominant kernel and the combine, each alone, seconds-long loops
    roof, comb, counts = kernel_blocks(skv, w, p, q, k, v, S, kname, peaks, args.loop_seconds,
                                       dev, stream)
    roof["traffic"] = recorded_traffic(kname, args.workload)
    if launches_per_step == 1 and not fused:
        roof["note"] = "split 1: a step is this kernel writing the output directly"

    e2e = None
    if not args.no_e2e:
        e2e = e2e_block(skv, p, q, k, v, out, ws, w, world, fl, stream, dev, args)
    ms = max_over_ranks([ms], device=dev if dist_on else None)[0]
    varlen = None
    if world == 1 and args.workload != "varlen" and not args.no_varlen:
        del q, k, v, ws, out
        torch.cuda.empty_cache()
        varlen = varlen_block(skv, args, peaks, dev, stream)
    if rank != 0:
        return None

    line = {
        "metric": METRIC, "value": whole_job_tflops(fl, world, ms), "unit": UNIT,
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms,
        "higher_is_better": True, "scaling": "weak",
        "vs_baseline": vs_pages(args.workload, whole_job_tflops(fl, world, ms)),
        "dtype": "bf16" if w.dtype == "bf16" else w.dtype, "data": "synthetic",
        "config": {**shape_config(w),
                   "split_kv": S, "fuse_combine": p.fuse_combine,
                   "block_m": skv.sk_default_block_m(w.d_qk, w.d_v),
                   "l2": "inputs larger than L2 "
                   f"({(w.total_q * w.d_qk + w.total_k * (w.d_qk + w.d_v)) * w.H * (4 if w.dtype == 'f32' else 2) / 1e6:.0f} MB)",
                   "parallelism": f"replicas x{world}" if world > 1 else "single GPU"},
        "roofline": roof,
        "combine": comb,
        "e2e": e2e,
        "gpu_launches": launches_per_step * args.steps,
        "clocks": clocks,
    }
    if varlen is not None:
        line["varlen"] = varlen
    if world == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = time_oracle(w, args.cpu_seconds)
    return line


def e2e_block(skv, p, q, k, v, out, ws, w, world, fl, stream, dev, args) -> dict:
    """The step end to end through the library's host-buffer call, sk_attn_fwd_host: every step
    copies its Q, K, V in from pinned host memory, runs the forward pass and copies its output
    back, all enqueued by the one call. Steps alternate between two streams with a device buffer
    each, so that one step's copies overlap the other's compute."""
    code = {"bf16": skv.SK_BF16, "f16": skv.SK_F16, "f32": skv.SK_F32}[w.dtype]
    hq, hk, hv = (t.cpu().pin_memory() for t in (q, k, v))
    hout = [torch.empty(out.shape, dtype=out.dtype).pin_memory() for _ in range(2)]
    nbytes = skv.sk_host_buffer_bytes(p, code, False)
    bufs = [torch.empty(nbytes, dtype=torch.uint8, device=dev) for _ in range(2)]
    streams = [torch.cuda.Stream(device=dev) for _ in range(2)]

    def run(n_steps):
        start = torch.cuda.Event()
        start.record(stream)
        for st in streams:
            st.wait_event(start)
        for i in range(n_steps):
            skv.sk_attn_fwd_host(p, hq, hk, hv, hout[i % 2], None, bufs[i % 2], stream=streams[i % 2])
        for st in streams:
            stream.wait_stream(st)

    run(4)
    torch.cuda.synchronize()
    # enough steps that the one step whose copy is not overlapped (the first) and the one whose
    # compute and read-back trail (the last) do not weigh on the per-step figure
    n_e2e = max(args.steps, 24)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    run(n_e2e)
    e1.record(stream)
    torch.cuda.synchronize()
    e2e_ms = max_over_ranks([e0.elapsed_time(e1) / n_e2e],
                            device=dev if torch.distributed.is_initialized() else None)[0]
    h2d_bytes = int(sum(t.numel() * t.element_size() for t in (hq, hk, hv)))
    return {"value": whole_job_tflops(fl, world, e2e_ms), "unit": UNIT,
            "h2d_bytes_per_step": h2d_bytes,
            "d2h_bytes_per_step": int(hout[0].numel() * hout[0].element_size()),
            "ms_per_step": e2e_ms, "call": "sk_attn_fwd_host",
            "overlap": "steps alternate between two streams, each with its own device buffer"}


def varlen_block(skv, args, peaks: dict, dev, stream) -> dict:
    """The long-context packed varlen prefill (4 x Sq 4096, Sk 8192 / 42700 / 65536 / 131072,
    H 12, D 192/128, split automatic): the whole step, the partial kernel alone against the
    dense bf16 peak and the combine alone against HBM, in the same run as the main line."""
    w = wl.LONG_VARLEN
    q, k, v = w.make_inputs(dev)
    p = skv.params_for(w, dev)
    S = skv.sk_auto_split_kv(p)
    p.split_kv = S
    out = torch.empty(w.total_q, w.H, w.d_v, dtype=q.dtype, device=dev)
    ws = torch.empty(max(skv.sk_workspace_bytes(p), 1), dtype=torch.uint8, device=dev)
    kname = skv.sk_partial_kernel_name(p, q, k, v)
    fl = flops_of(w)
    with ClockSampler(dev.index) as cs:
        st = time_back_to_back(lambda i: skv.sk_attn_fwd(p, q, k, v, out, None, ws),
                               args.loop_seconds, stream)
    roof, comb, _ = kernel_blocks(skv, w, p, q, k, v, S, kname, peaks, args.loop_seconds, dev,
                                  stream)
    roof["traffic"] = recorded_traffic(kname, "varlen")
    return {"workload": w.name, "split_kv": S, "flop_per_step": fl,
            "ms_per_step": st["mean_ms"], "step_tflops": fl / (st["mean_ms"] * 1e-3) / 1e12,
            "steps": st["launches"], "step_clocks": cs.summary(), "partial": roof,
            "combine": comb}


def shape_config(w) -> dict:
    """The workload's shape keys of the JSON line's config, shared by both arms."""
    return {"workload": w.name, "sequences": w.B, "seq_len_q": list(w.seqlens_q),
            "seq_len_k": list(w.seqlens_k), "heads": w.H, "d_qk": w.d_qk, "d_v": w.d_v,
            "n_per_block": w.n_per_block, "flop_per_step": flops_of(w)}


def run_reference(args, rank: int):
    """The reference arm: the CPU oracle as it stands, on host cores, rank 0 only."""
    if rank != 0:
        return None
    w = wl.ALL[args.workload]
    import oracle
    oracle.build()
    per_step = max(args.cpu_seconds / max(args.steps + args.warmup, 1), 0.5)
    inputs = w.make_inputs("cpu")
    vals = []
    base = None
    for i in range(args.warmup + args.steps):
        r = time_oracle(w, per_step, seed=i, inputs=inputs)
        if i >= args.warmup:
            vals.append(r["value"])
            base = r
    value = statistics.mean(vals)
    return {"metric": METRIC, "value": value, "unit": UNIT, "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": vs_pages(args.workload, value), "dtype": "f64",
            "data": "synthetic", "impl": "reference",
            "config": {**shape_config(w), "parallelism": "host cores (the f64 oracle, unsplit)"},
            "cpu_baseline": {"value": value, "unit": UNIT, "cores": base["cores"],
                             "kind": "oracle", "sample": base["sample"] + " per step"},
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=300)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", choices=sorted(wl.ALL), default="target")
    ap.add_argument("--split", type=int, default=None, help="force split_kv (default: auto)")
    ap.add_argument("--fuse-combine", action="store_true",
                    help="merge the splits inside the tensor-core kernel (sk_params.fuse_combine)")
    ap.add_argument("--cpu-seconds", type=float, default=15.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--loop-seconds", type=float, default=1.0,
                    help="device time of each kernel-alone loop (partial kernel, combine)")
    ap.add_argument("--no-varlen", action="store_true",
                    help="skip the long-context varlen block of the JSON line")
    ap.add_argument("--no-e2e", action="store_true",
                    help="skip the end-to-end (host buffers) measurement")
    ap.add_argument("--step-only", action="store_true",
                    help="time the steps only (no kernel loops, end-to-end, varlen block or CPU "
                         "baseline): the command the profiler captures")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    dist_on = world > 1
    if args.impl == "reference":
        line = run_reference(args, rank)
        if line is not None:
            print(json.dumps(line), flush=True)
        return
    if dist_on:
        torch.distributed.init_process_group("nccl")
    try:
        line = run_ours(args, rank, world, dist_on)
        if line is not None:
            print(json.dumps(line), flush=True)
    finally:
        if dist_on:
            torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()
