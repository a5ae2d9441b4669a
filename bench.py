"""Benchmark: one step of the paged prefix-reuse hot path on synthetic data.

A step is the whole path over one batch: copy-on-write block copies, slot
indexing, append of the new tokens' K/V, prefix attention of the prefill
chunks and decode attention of the decode batch (whichever the workload has).
The default workload is the long-context prefix batch, the largest of the
five shapes (Hq=64, Hkv=8, d=128, bf16; 4 requests, each a 32768-token
cached prefix at random physical placement plus a 2048-token new chunk).
Its step has no decode sequences, so the same run also times the decode
batch of the multi-turn continuous-batching shape (Qwen2.5-32B-shaped
layer: 64 sequences, cached contexts lognormal around 2048 tokens) and
reports it in a ``decode`` object: tokens/s and HBM GB/s against the
measured copy bandwidth.

Prints ONE JSON line.  ``value`` is the algorithmic prefix-attention
TFLOP/s of the whole step (4*d*Hq*sum(N*P + N(N+1)/2) per step, divided by
the device time of the step), with inputs resident in HBM and L2 flushed
between timed steps.  ``e2e`` is the same metric measured through the C ABI
with pinned host buffers: the step's inputs are copied host->device and its
outputs device->host inside the timed region, the sequences in groups on
their own streams so that copies overlap kernels (``step.HostStep``),
replayed as one CUDA graph that includes the copies.

    python bench.py [--steps K] [--warmup W] [--workload NAME] [--decode-workload NAME] [--impl kvp|reference]
    python bench.py --op block_swap|decode_q [--bits 8|4]|blockmgr|cacheblend

With several GPUs (torchrun), every rank runs an independent replica (the
path has no exchange step) and the slowest rank's time is reported.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import workloads as wl  # noqa: E402

METRIC = "paged prefix-attn TFLOP/s + decode tok/s; % of GB300 tensor/HBM roofline"
WORKLOADS = {
    "shared_system_prompt": 2,
    "rag_chunk_reuse": 3,
    "continuous_batching_step": 4,
    "long_context_prefix": 5,
    # one request of the long-context shape in a 4096-block pool: a small case
    # for detailed profiler captures of the same kernel
    "long_context_prefix_b1": 5,
}
WORKLOAD_ARGS = {"long_context_prefix_b1": {"B": 1, "num_blocks": 4096}}
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
L2_FLUSH_BYTES = 512 << 20


# ---------------------------------------------------------------------------
# algorithmic work (the FLOP and byte conventions of the measurement)
# ---------------------------------------------------------------------------
def prefill_flops(w) -> float:
    """4 * d * Hq * sum_s (N_s * P_s + N_s (N_s + 1) / 2) over the prefill chunks."""
    n = w.new_lens[: w.num_prefill].astype(np.float64)
    p = w.prefix_lens[: w.num_prefill].astype(np.float64)
    return float(4.0 * w.head_dim * w.num_q_heads * np.sum(n * p + n * (n + 1) / 2))


def decode_kv_bytes(w) -> float:
    """Unique K+V bytes read by the decode batch (each sequence's context)."""
    L = w.context_lens[w.num_prefill :].astype(np.float64)
    return float(np.sum(L) * w.num_kv_heads * w.head_dim * 2 * 2)


def row_flops(w, rows) -> float:
    """Algorithmic flops of the given flat prefill rows t * Hq + h: 4 d (p + 1)."""
    cu = w.cu_seqlens_q
    t = np.asarray(rows) // w.num_q_heads
    s = np.searchsorted(cu, t, side="right") - 1
    pos = w.context_lens[s] - w.new_lens[s] + (t - cu[s])
    return float(np.sum(4.0 * w.head_dim * (pos + 1)))


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        try:
            with open(path) as f:
                d = json.load(f)
            return d, "measured"
        except Exception:
            pass
    return dict(FALLBACK_PEAKS), "fallback"


def _peak_value(peaks, *keys):
    for k in keys:
        v = peaks.get(k)
        if isinstance(v, (int, float)) and v > 0:
            return float(v)
        if isinstance(v, dict):
            for kk in ("value", "burst", "gbs", "tflops"):
                if isinstance(v.get(kk), (int, float)):
                    return float(v[kk])
    return None


# Workloads too large for a full ncu capture under the size rule take their
# DRAM traffic from a smaller capture of the same kernel, scaled by the units
# processed: long_context_prefix is four independent copies of the B=1 case
# (own block tables, Q and O), so its traffic is four times B=1's.
TRAFFIC_PROXY = {"long_context_prefix": ("long_context_prefix_b1", 4.0)}
# The source files a kernel's code comes from (besides kvp_internal.cuh).
KERNEL_SOURCES = {"prefix": ["kvp_prefix.cu", "kvp_prefix_impl.cuh"], "decode": ["kvp_decode.cu", "kvp_decode_impl.cuh"],
                  "decode_q_int8": ["kvp_quant.cu", "kvp_decode_impl.cuh"],
                  "decode_q_int4": ["kvp_quant.cu", "kvp_decode_impl.cuh"],
                  "prefix_q_int8": ["kvp_prefix_q.cu", "kvp_prefix_impl.cuh"],
                  "prefix_q_int4": ["kvp_prefix_q.cu", "kvp_prefix_impl.cuh"], "deviation": ["kvp_cacheblend.cu"],
                  "block_swap": ["kvp_cache.cu"], "append": ["kvp_cache.cu"]}


def committed_traffic(kernel: str, workload: str):
    if workload in TRAFFIC_PROXY:
        proxy, factor = TRAFFIC_PROXY[workload]
        t = _committed_traffic(kernel, proxy)
        return None if t is None else t * factor
    return _committed_traffic(kernel, workload)


def code_digest(paths) -> str:
    """sha256 (16 hex digits) of the files' code with their // comments and
    blank lines removed: a comment edit leaves a kernel, and its counters,
    unchanged.  (The CUDA sources hold no string literal containing //.)"""
    h = hashlib.sha256()
    for path in paths:
        for line in open(path, encoding="utf-8"):
            code = line.split("//", 1)[0].rstrip()
            if code:
                h.update(code.encode() + b"\n")
    return h.hexdigest()[:16]


def _committed_traffic(kernel: str, workload: str):
    """DRAM bytes per launch from the committed ncu summary, if that summary
    was taken on the kernel code as it is now -- the kernel's source files and
    the shared kvp_internal.cuh, hashed together without comments -- else
    None."""
    path = os.path.join(ROOT, "profiles", f"{kernel}_{workload}.txt")
    csrc = os.path.join(ROOT, "paged_prefix_reuse_gb300", "csrc")
    srcs = [os.path.join(csrc, f) for f in KERNEL_SOURCES.get(kernel, [f"kvp_{kernel}.cu"])]
    srcs.append(os.path.join(csrc, "kvp_internal.cuh"))
    if not (os.path.exists(path) and all(os.path.exists(f) for f in srcs)):
        return None
    digest = code_digest(srcs)
    vals = {}
    for line in open(path):
        if ":" in line:
            k, v = line.split(":", 1)
            vals[k.strip()] = v.strip()
    if vals.get("source_sha256_16") != digest:
        return None
    try:
        return float(vals["dram_bytes_per_launch"])
    except (KeyError, ValueError):
        return None


# ---------------------------------------------------------------------------
# clocks during the timed region
# ---------------------------------------------------------------------------
class ClockSampler:
    FIELDS = ("clocks.sm,clocks.max.sm,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index: int):
        self.proc = None
        self.idx = device_index

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits", "-lms", "20",
                 "-i", str(self.idx)], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except Exception:
            self.proc.kill()
            out, _ = self.proc.communicate()
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in out.strip().splitlines():
            parts = [x.strip() for x in line.split(",")]
            if len(parts) < 6:
                continue
            try:
                sm.append(float(parts[0]))
                mx.append(float(parts[1]))
            except ValueError:
                continue
            for n, v in zip(names, parts[2:6]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "reasons": sorted(reasons),
                "samples": len(sm), "window": "untimed pre-roll steps + the timed steps"}


# ---------------------------------------------------------------------------
# distributed bookkeeping (replicas only)
# ---------------------------------------------------------------------------
def dist_setup():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def max_over_ranks(value: float, device=None) -> float:
    """The largest per-rank value (a time) over the process group, or the value
    itself with one process.  Replicas end when the slowest rank does."""
    import torch
    import torch.distributed as dist

    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return float(value)
    t = torch.tensor([float(value)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_rate(units_per_rank: float, world: int, ms: float) -> float:
    """Whole-job throughput: every rank processed units_per_rank in at most ms."""
    return world * units_per_rank / (ms * 1e-3)


def cpu_oracle_sample(w, budget_s: float, seed: int = 0):
    """Time the fp64 oracle on a bounded random sample of prefill rows (and
    decode rows) of the workload; returns (tflops, seconds, rows, threads)."""
    import oracle

    rng = np.random.default_rng(seed)
    tq = int(w.cu_seqlens_q[w.num_prefill])
    all_rows = tq * w.num_q_heads
    cu = w.cu_seqlens_q[: w.num_prefill + 1]
    ctx = w.context_lens[: w.num_prefill]
    bt = w.block_tables[: w.num_prefill]
    n = 16
    spent, flops, done = 0.0, 0.0, 0
    while spent < budget_s and done < all_rows:
        rows = rng.integers(0, all_rows, size=n)
        t0 = time.perf_counter()
        oracle.prefix_attn(w.dtype, w.k_pool, w.v_pool, w.q[:tq], cu, ctx, bt, w.softmax_scale, rows)
        dt = time.perf_counter() - t0
        spent += dt
        flops += row_flops(w, rows)
        done += n
        if dt < budget_s / 8:
            n *= 2
    return flops / spent / 1e12, spent, done, oracle.num_threads()


# ---------------------------------------------------------------------------
# arms
# ---------------------------------------------------------------------------
def run_reference(args):
    world, rank, _ = dist_setup()
    if rank != 0:
        return 0
    w = wl.make_config(WORKLOADS[args.workload], **WORKLOAD_ARGS.get(args.workload, {}))
    flops = prefill_flops(w)
    per_step_budget = max(1.0, 60.0 / max(1, args.steps + args.warmup))
    for _ in range(args.warmup):
        cpu_oracle_sample(w, per_step_budget / 4)
    vals, secs, rows_done, threads = [], 0.0, 0, 1
    for i in range(args.steps):
        v, s, r, threads = cpu_oracle_sample(w, per_step_budget, seed=i + 1)
        vals.append(v)
        secs += s
        rows_done += r
    value = float(np.mean(vals))
    ms = flops / (value * 1e12) * 1e3
    sample = (f"{rows_done} random (query token, head) rows of the prefill batch over {args.steps} steps, "
              f"{secs:.1f} s of CPU time; value scales the sample's algorithmic flops to the whole step")
    line = {
        "impl": "reference",
        "metric": METRIC,
        "value": value,
        "unit": "TFLOP/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": ms,
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "f64",
        "data": "synthetic",
        "config": {"workload": args.workload},
        "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": threads, "kind": "oracle", "sample": sample},
        "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


def time_decode(st, stream, flush_l2, warmup, steps):
    """Device time (ms) of the decode call of ``st`` (kvp_decode_attn plus the
    split merge), replayed from a CUDA graph after an L2 flush, like the
    per-kernel times of the step."""
    import torch

    with torch.cuda.stream(stream):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            st.run_decode()
        times = []
        for i in range(warmup + steps):
            flush_l2()
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(stream)
            g.replay()
            b.record(stream)
            stream.synchronize()
            if i >= warmup:
                times.append(a.elapsed_time(b))
    return float(np.mean(times))


def decode_block(w, st, ms, peaks, peak_src, workload, launches, steps):
    """The decode half of the metric: tokens/s of one decode call over the
    batch and its K/V bytes per second against the measured HBM copy rate."""
    hbm = _peak_value(peaks, "hbm_gbs", "hbm_GBps") or FALLBACK_PEAKS["hbm_gbs"]
    byts = decode_kv_bytes(w)
    gbs = byts / (ms * 1e-3) / 1e9
    return {
        "workload": workload,
        "sequences": int(w.num_decode),
        "tok_s": w.num_decode / (ms * 1e-3),
        "ms": ms,
        "kv_bytes": byts,
        "achieved_gbs": gbs,
        "peak_gbs": hbm,
        "frac": gbs / hbm,
        "peak_source": f"{peak_src} HBM copy",
        "splits": int(st.decode_splits),
        "gpu_launches": launches * steps,
        "l2": "flushed before every timed call",
        "traffic": committed_traffic("decode", workload),
    }


def run_kvp(args):
    import torch

    world, rank, local = dist_setup()
    if world > 1:
        import torch.distributed as dist

        torch.cuda.set_device(local)
        dist.init_process_group("nccl")
    else:
        torch.cuda.set_device(0)
    dev = torch.device("cuda", torch.cuda.current_device())

    from paged_prefix_reuse_gb300 import build as kvp_build

    kvp_build.build_library()
    import paged_prefix_reuse_gb300 as kvp
    from paged_prefix_reuse_gb300.step import DeviceStep

    kvp.load_library()
    kvp.kvp_set_launch_options(kvp.LAUNCH_PDL if args.pdl else 0)
    w = wl.make_config(WORKLOADS[args.workload], **WORKLOAD_ARGS.get(args.workload, {}))
    st = DeviceStep(w, device=dev, prefix_splits=args.prefix_splits, decode_splits=args.decode_splits)
    stream = torch.cuda.Stream(device=dev)
    flops = prefill_flops(w)
    dec_bytes = decode_kv_bytes(w)
    flush = torch.empty(L2_FLUSH_BYTES // 4, dtype=torch.int32, device=dev)
    flush_sink = torch.empty(1, dtype=torch.int32, device=dev)

    def flush_l2():
        """Write a buffer 4x the L2 size, then read it back: the write evicts
        every line of the workload, the read makes L2 write back the dirty
        lines of the fill before the timed step starts (so the step does not
        pay for the flush's own write-backs)."""
        flush.zero_()
        torch.amax(flush, dim=0, out=flush_sink[0])

    # kernels launched per step (ours, counted from the calls the step makes)
    launches = 0
    launches += 1 if st.pairs.shape[0] else 0
    launches += 2 if st.T else 0  # slot mapping + append
    if st.npf:
        launches += 1 + (1 if st.prefix_splits > 1 else 0)
    if st.ndec:
        launches += 1 + (1 if st.decode_splits > 1 else 0)

    def barrier():
        if world > 1:
            import torch.distributed as dist

            dist.barrier()

    # ---- device-resident timing ----
    # The step's kernels are enqueued once through the C ABI inside a CUDA
    # graph capture; each timed step replays that graph (the launch-bound
    # step then pays no per-call host overhead).  L2 is flushed before every
    # timed step, outside the timed events.
    with torch.cuda.stream(stream):
        for _ in range(args.warmup):
            st.run(stream)
        stream.synchronize()
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph, stream=stream):
            st.run()
        for _ in range(args.warmup):
            graph.replay()
        stream.synchronize()
        ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
        clocks = ClockSampler(dev.index if world == 1 else local)
        barrier()
        torch.cuda.synchronize()
        # nvidia-smi samples every 20 ms: keep the GPU busy with untimed steps
        # for a short pre-roll so the samples cover the load the timed steps see.
        clocks.start()
        t_pre = time.perf_counter()
        while time.perf_counter() - t_pre < args.preroll_s:
            for _ in range(8):
                flush_l2()
                graph.replay()
            stream.synchronize()
        t_wall = time.perf_counter()
        for i in range(args.steps):
            flush_l2()
            ev[i][0].record(stream)
            graph.replay()
            ev[i][1].record(stream)
        stream.synchronize()
        torch.cuda.synchronize()
        barrier()
        wall = time.perf_counter() - t_wall
        clk = clocks.stop()
        # Per-kernel device times for the roofline: each call is captured in a
        # graph of its own and timed by events around its replay, so the
        # duration is the kernel's, not the host's launch latency.
        calls = {"copy": st.run_copy, "slots": st.run_slots, "append": st.run_append, "prefill": st.run_prefill,
                 "decode": st.run_decode}
        has_work = {"copy": bool(st.pairs.shape[0]), "slots": st.T > 0, "append": st.T > 0,
                    "prefill": st.npf > 0 and st.tq > 0, "decode": st.ndec > 0}
        kern_ms = {}
        for k, call in calls.items():
            if not has_work[k]:
                kern_ms[k] = 0.0
                continue
            gk = torch.cuda.CUDAGraph()
            with torch.cuda.graph(gk, stream=stream):
                call()
            times = []
            for i in range(args.warmup + args.steps):
                flush_l2()
                a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                a.record(stream)
                gk.replay()
                b.record(stream)
                stream.synchronize()
                if i >= args.warmup:
                    times.append(a.elapsed_time(b))
            kern_ms[k] = float(np.mean(times))
        stream.synchronize()
    # The decode half of the metric, when the step itself has no decode
    # batch: the decode sequences of another workload, appended once, then
    # their decode call timed alone.
    dec_w = dec_st = None
    dec_ms = 0.0
    if not st.ndec and args.decode_workload != "none":
        dec_w = wl.make_config(WORKLOADS[args.decode_workload], **WORKLOAD_ARGS.get(args.decode_workload, {}))
        dec_st = DeviceStep(dec_w, device=dev, decode_splits=args.decode_splits)
        if dec_st.ndec:
            with torch.cuda.stream(stream):
                dec_st.run_copy(stream)
                dec_st.run_slots(stream)
                dec_st.run_append(stream)
            stream.synchronize()
            dec_ms = time_decode(dec_st, stream, flush_l2, args.warmup, args.steps)
        torch.cuda.synchronize()
        if dec_st.pool.errors():
            raise RuntimeError(f"decode workload: device error word {dec_st.pool.errors():#x}")
    step_ms = [a.elapsed_time(b) for a, b in ev]
    ms = max_over_ranks(float(np.mean(step_ms)), dev)

    # ---- end to end through the C ABI with pinned host buffers ----
    # HostStep: the same calls per group of sequences, each group's copies
    # overlapping the other groups' kernels.
    from paged_prefix_reuse_gb300.step import HostStep

    hs = HostStep(st, groups=args.e2e_groups)
    h2d, d2h = hs.h2d_bytes, hs.d2h_bytes
    e2e_ms = []
    with torch.cuda.stream(stream):
        hgraph = hs.capture(stream)
        for i in range(args.warmup + args.steps):
            flush_l2()
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(stream)
            hgraph.replay()
            b.record(stream)
            stream.synchronize()
            if i >= args.warmup:
                e2e_ms.append(a.elapsed_time(b))
    e2e = max_over_ranks(float(np.mean(e2e_ms)), dev)

    if rank != 0:
        return 0
    peaks, peak_src = load_peaks()
    value = job_rate(flops, world, ms) / 1e12
    line = {
        "metric": METRIC,
        "value": value,
        "unit": "TFLOP/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": ms,
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "bf16" if w.dtype == "bf16" else "f16",
        "data": "synthetic",
        "config": {
            "workload": args.workload,
            "B": w.B,
            "num_q_heads": w.num_q_heads,
            "num_kv_heads": w.num_kv_heads,
            "head_dim": w.head_dim,
            "block_size": w.block_size,
            "num_blocks": w.num_blocks,
            "prefill_tokens": int(w.cu_seqlens_q[w.num_prefill]),
            "decode_seqs": int(w.num_decode),
            "prefix_splits": int(getattr(st, "prefix_splits", 0)),
            "decode_splits": int(getattr(st, "decode_splits", 0)),
            "l2": "flushed before every timed step (512 MB write, then read back)",
            "launch": "CUDA graph replay of the step; the graph holds the kernels the C-ABI calls enqueued",
            "parallelism": f"replicas x{world}",
            "pdl": bool(args.pdl),
        },
        "gpu_launches": launches * args.steps,
        "kernel_ms": kern_ms,
        "wall_s": wall,
        "e2e": {"value": job_rate(flops, world, e2e) / 1e12, "unit": "TFLOP/s", "ms_per_step": e2e,
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "groups": len(hs.groups)},
        "clocks": clk,
    }
    if st.npf:
        peak = _peak_value(peaks, "bf16_tflops", "bf16_tflops_burst") or FALLBACK_PEAKS["bf16_tflops"]
        achieved = flops / (kern_ms["prefill"] * 1e-3) / 1e12
        line["roofline"] = {
            "kernel": "prefix_attn" + (" + lse_merge" if st.prefix_splits > 1 else ""),
            "bound": "tensor",
            "achieved": achieved,
            "peak": peak,
            "unit": "TFLOP/s",
            "frac": achieved / peak,
            "peak_source": f"{peak_src} bf16 dense (burst)" + (", fp16 taken equal to bf16" if w.dtype == "f16" else ""),
            "traffic": committed_traffic("prefix", args.workload),
        }
    dec_launches = lambda s: 1 + (1 if s.decode_splits > 1 else 0)
    if st.ndec:
        hbm = _peak_value(peaks, "hbm_gbs", "hbm_GBps") or FALLBACK_PEAKS["hbm_gbs"]
        gbs = dec_bytes / (kern_ms["decode"] * 1e-3) / 1e9
        line["decode"] = decode_block(w, st, kern_ms["decode"], peaks, peak_src, args.workload, dec_launches(st),
                                      args.steps)
        if not st.npf:
            line["roofline"] = {"kernel": "decode_attn", "bound": "hbm", "achieved": gbs, "peak": hbm,
                                "unit": "GB/s", "frac": gbs / hbm, "peak_source": peak_src,
                                "traffic": committed_traffic("decode", args.workload)}
    elif dec_st is not None and dec_st.ndec:
        line["decode"] = decode_block(dec_w, dec_st, dec_ms, peaks, peak_src, args.decode_workload,
                                      dec_launches(dec_st), args.steps)
    if not args.no_cpu_baseline and world >= 1:
        v, s, r, threads = cpu_oracle_sample(w, args.cpu_seconds)
        line["cpu_baseline"] = {
            "value": v,
            "unit": "TFLOP/s",
            "cores": threads,
            "kind": "oracle",
            "sample": f"{r} random (query token, head) rows of the prefill batch, {s:.1f} s; "
                      f"flops of the sample / CPU time",
        }
    print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist

        dist.destroy_process_group()
    return 0


def run_swap(args):
    """Host <-> device block swap: move N scattered pages (K and V) of the
    mixed-batch pool to a pinned host page pool and back, through the C ABI.
    The denominator is one contiguous pinned copy of the same bytes
    (cudaMemcpyAsync through torch), measured in the same run: the host
    link's practical rate."""
    import numpy as np
    import torch

    torch.cuda.set_device(0)
    dev = torch.device("cuda", 0)
    from paged_prefix_reuse_gb300 import build as kvp_build

    kvp_build.build_library()
    import paged_prefix_reuse_gb300 as kvp
    from paged_prefix_reuse_gb300.step import DeviceStep

    kvp.load_library()
    kvp.kvp_set_launch_options(kvp.LAUNCH_PDL if args.pdl else 0)
    w = wl.make_config(4)
    st = DeviceStep(w, device=dev)
    pool = st.pool
    n = min(1024, pool.num_blocks)
    host = kvp.HostKVPool.like(pool, n)
    rng = np.random.default_rng(0)
    src = rng.choice(pool.num_blocks, size=n, replace=False)
    out_pairs = torch.from_numpy(np.stack([src, np.arange(n)], 1).astype(np.int32)).to(dev)
    in_pairs = torch.from_numpy(np.stack([np.arange(n), src], 1).astype(np.int32)).to(dev)
    page_bytes = 2 * pool.num_kv_heads * pool.block_size * pool.head_dim * pool.k.element_size()
    moved = n * page_bytes
    stream = torch.cuda.Stream(device=dev)
    flush = torch.empty(L2_FLUSH_BYTES // 4, dtype=torch.int32, device=dev)
    dbuf = torch.empty(moved, dtype=torch.uint8, device=dev)
    hbuf = torch.empty(moved, dtype=torch.uint8, pin_memory=True)

    def timed(fn):
        ts = []
        with torch.cuda.stream(stream):
            for i in range(args.warmup + args.steps):
                flush.zero_()
                e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                e0.record(stream)
                fn()
                e1.record(stream)
                e1.synchronize()
                if i >= args.warmup:
                    ts.append(e0.elapsed_time(e1) / 1e3)
        return sorted(ts)[len(ts) // 2]

    t_out = timed(lambda: kvp.kvp_block_swap(pool, host, out_pairs, kvp.HostKVPool.SWAP_OUT, stream=stream))
    t_in = timed(lambda: kvp.kvp_block_swap(pool, host, in_pairs, kvp.HostKVPool.SWAP_IN, stream=stream))
    t_d2h = timed(lambda: hbuf.copy_(dbuf, non_blocking=True))
    t_h2d = timed(lambda: dbuf.copy_(hbuf, non_blocking=True))
    gbs = lambda t: moved / t / 1e9
    value = 2 * moved / (t_out + t_in) / 1e9
    peak = 2 * moved / (t_d2h + t_h2d) / 1e9
    line = {
        "metric": "block swap GB/s (scattered K+V pages, GPU pool to pinned host pool and back)",
        "value": value, "unit": "GB/s", "n_gpus": 1, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": (t_out + t_in) * 1e3, "higher_is_better": True, "op": "block_swap",
        "dtype": "bf16", "data": "synthetic",
        "config": {"workload": "continuous_batching_step pool", "pages": n, "page_bytes": page_bytes,
                   "bytes_each_way": moved, "l2": "flushed before every timed call"},
        "out_gbs": gbs(t_out), "in_gbs": gbs(t_in), "gpu_launches": 2,
        "roofline": {"bound": "host link", "achieved": value, "peak": peak, "unit": "GB/s", "frac": value / peak,
                     "peak_source": "one contiguous pinned cudaMemcpyAsync of the same bytes each way, this run",
                     "memcpy_d2h_gbs": gbs(t_d2h), "memcpy_h2d_gbs": gbs(t_h2d),
                     # device DRAM bytes of one swap-out launch (the host side is not device DRAM)
                     "traffic": committed_traffic("block_swap", "continuous_batching_step_swap_out")},
    }
    print(json.dumps(line), flush=True)
    return 0


def run_decode_q(args):
    """Decode over a quantized cached prefix: the mixed batch's decode
    sequences with every complete page moved to an 8- or 4-bit pool (the
    trailing partial page stays 16-bit), timed against the 16-bit decode of
    the same batch.  Bytes are the pages each kernel reads: quantized pages at
    their packed size (codes and fp16 scales), 16-bit pages whole."""
    import numpy as np
    import torch

    torch.cuda.set_device(0)
    dev = torch.device("cuda", 0)
    from paged_prefix_reuse_gb300 import build as kvp_build

    kvp_build.build_library()
    import paged_prefix_reuse_gb300 as kvp
    from paged_prefix_reuse_gb300.step import DeviceStep

    kvp.load_library()
    kvp.kvp_set_launch_options(kvp.LAUNCH_PDL if args.pdl else 0)
    w = wl.make_config(4)
    st = DeviceStep(w, device=dev)
    st.run_slots()
    st.run_append()
    torch.cuda.synchronize()
    pool = st.pool
    bs, hkv, d = pool.block_size, pool.num_kv_heads, pool.head_dim
    ctx = st.ctx[st.npf:].cpu().numpy()
    bt = st.bt[st.npf:].cpu().numpy().copy()
    qpages = (ctx // bs).astype(np.int32)
    pairs = []
    for b in range(len(ctx)):
        for pg in range(int(qpages[b])):
            pairs.append((int(bt[b, pg]), len(pairs)))
            bt[b, pg] = len(pairs) - 1
    qp = kvp.QuantKVPool.like(pool, len(pairs), args.bits)
    tpairs = torch.tensor(pairs, dtype=torch.int32, device=dev)
    kvp.kvp_quantize_blocks(pool, qp, tpairs)
    torch.cuda.synchronize()
    tq = torch.from_numpy(qpages).to(dev)
    tbt = torch.from_numpy(bt).to(dev)
    q = st.q[st.tq:]
    ctx_d = st.ctx[st.npf:]
    bt16 = st.bt[st.npf:]
    stream = torch.cuda.Stream(device=dev)
    flush = torch.empty(L2_FLUSH_BYTES // 4, dtype=torch.int32, device=dev)

    def timed(fn):
        ts = []
        with torch.cuda.stream(stream):
            for i in range(args.warmup + args.steps):
                flush.zero_()
                e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                e0.record(stream)
                fn()
                e1.record(stream)
                e1.synchronize()
                if i >= args.warmup:
                    ts.append(e0.elapsed_time(e1) / 1e3)
        return sorted(ts)[len(ts) // 2]

    mctx = int(ctx.max())
    # the write-back of the cached pages in quantized form (one call over all pairs)
    t_quant = timed(lambda: kvp.kvp_quantize_blocks(pool, qp, tpairs, stream=stream))
    t16 = timed(lambda: kvp.kvp_decode_attn(pool, q, ctx_d, bt16, mctx, w.softmax_scale, stream=stream))
    tqz = timed(lambda: kvp.kvp_decode_attn_q(pool, qp, tq, q, ctx_d, tbt, mctx, w.softmax_scale, stream=stream))
    npages = (ctx + bs - 1) // bs
    page16 = hkv * bs * d * 2 * 2
    pageq = hkv * (2 * bs * d * args.bits // 8 + 4 * d + 4 * bs)
    bytes16 = float(npages.sum() * page16)
    bytesq = float(qpages.sum() * pageq + (npages - qpages).sum() * page16)
    peaks, peak_src = load_peaks()
    hbm = _peak_value(peaks, "hbm_gbs") or FALLBACK_PEAKS["hbm_gbs"]
    gbs = bytesq / tqz / 1e9
    line = {
        "metric": f"decode over an int{args.bits} cached prefix: sequences/s (GB/s of quantized pages read)",
        "value": len(ctx) / tqz, "unit": "seq/s", "n_gpus": 1, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": tqz * 1e3, "higher_is_better": True, "op": "decode_q", "dtype": w.dtype, "data": "synthetic",
        "config": {"workload": "continuous_batching_step decode batch", "B": int(len(ctx)), "bits": args.bits,
                   "quantized_pages": int(qpages.sum()), "pages_16bit": int((npages - qpages).sum()),
                   "l2": "flushed before every timed call"},
        "decode_16bit_ms": t16 * 1e3, "speedup_vs_16bit": t16 / tqz, "bytes_read": bytesq,
        "quantize_ms": t_quant * 1e3,
        "quantize_gbs": len(pairs) * (page16 + pageq) / t_quant / 1e9,  # 16-bit pages read + quantized written
        "bytes_read_16bit": bytes16, "gpu_launches": 1 + (1 if kvp.kvp_decode_num_splits(
            len(ctx), hkv, bs, mctx) > 1 else 0),
        "roofline": {"kernel": "decode_attn_q", "bound": "hbm", "achieved": gbs, "peak": hbm, "unit": "GB/s",
                     "frac": gbs / hbm, "peak_source": f"{peak_src} HBM copy",
                     "traffic": committed_traffic(f"decode_q_int{args.bits}",
                                                  f"continuous_batching_step_int{args.bits}_prefix")},
    }
    print(json.dumps(line), flush=True)
    return 0


def run_prefix_q(args):
    """Prefix attention over a quantized cached prefix: the workload's
    prefill chunks with every complete page of their cached prefixes moved to
    an 8- or 4-bit pool (a block shared by several tables is quantized once),
    timed against the 16-bit prefix attention of the same batch.  The FLOP
    count is the prefill's (quantization changes where K/V come from, not the
    work)."""
    import numpy as np
    import torch

    torch.cuda.set_device(0)
    dev = torch.device("cuda", 0)
    from paged_prefix_reuse_gb300 import build as kvp_build

    kvp_build.build_library()
    import paged_prefix_reuse_gb300 as kvp
    from paged_prefix_reuse_gb300.step import DeviceStep

    kvp.load_library()
    kvp.kvp_set_launch_options(kvp.LAUNCH_PDL if args.pdl else 0)
    w = wl.make_config(WORKLOADS[args.workload], **WORKLOAD_ARGS.get(args.workload, {}))
    st = DeviceStep(w, device=dev)
    st.run_copy()
    st.run_slots()
    st.run_append()
    torch.cuda.synchronize()
    pool = st.pool
    bs = pool.block_size
    npf = st.npf
    bt = st.bt[:npf].cpu().numpy().copy()
    prefix = (w.context_lens[:npf] - w.new_lens[:npf]).astype(np.int64)
    qpages = (prefix // bs).astype(np.int32)
    qid = {}
    for s_ in range(npf):
        for pg in range(int(qpages[s_])):
            src = int(bt[s_, pg])
            if src not in qid:
                qid[src] = len(qid)
            bt[s_, pg] = qid[src]
    pairs = np.array(list(qid.items()), dtype=np.int32).reshape(-1, 2)
    qp = kvp.QuantKVPool.like(pool, max(1, len(qid)), args.bits)
    for i in range(0, len(pairs), 65535):
        kvp.kvp_quantize_blocks(pool, qp, torch.from_numpy(pairs[i:i + 65535]).to(dev))
    torch.cuda.synchronize()
    tq, tbt = torch.from_numpy(qpages).to(dev), torch.from_numpy(bt).to(dev)
    q, cu, ctx = st.q[: st.tq], st.cu[: npf + 1], st.ctx[:npf]
    out = torch.empty_like(q)
    lse = torch.empty((w.num_q_heads, st.tq), dtype=torch.float32, device=dev)
    stream = torch.cuda.Stream(device=dev)
    flush = torch.empty(L2_FLUSH_BYTES // 4, dtype=torch.int32, device=dev)

    def timed(fn):
        with torch.cuda.stream(stream):
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=stream):
                fn()
            ts = []
            for i in range(args.warmup + args.steps):
                flush.zero_()
                e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                e0.record(stream)
                g.replay()
                e1.record(stream)
                e1.synchronize()
                if i >= args.warmup:
                    ts.append(e0.elapsed_time(e1) / 1e3)
        return float(np.mean(ts))

    t16 = timed(lambda: kvp.kvp_prefix_attn(pool, q, cu, ctx, st.bt[:npf], st.max_q_pf, st.max_ctx_pf, st.scale,
                                            num_splits=st.prefix_splits, out=out, lse=lse, workspace=st.ws_pf,
                                            stream=stream))
    tqz = timed(lambda: kvp.kvp_prefix_attn_q(pool, qp, tq, q, cu, ctx, tbt, st.max_q_pf, st.max_ctx_pf, st.scale,
                                              num_splits=st.prefix_splits, out=out, lse=lse, workspace=st.ws_pf,
                                              stream=stream))
    if pool.errors():
        raise RuntimeError(f"device error word {pool.errors():#x}")
    flops = prefill_flops(w)
    peaks, peak_src = load_peaks()
    peak = _peak_value(peaks, "bf16_tflops") or FALLBACK_PEAKS["bf16_tflops"]
    hkv, d = pool.num_kv_heads, pool.head_dim
    page16 = hkv * bs * d * 2 * 2
    pageq = hkv * (2 * bs * d * args.bits // 8 + 4 * d + 4 * bs)
    line = {
        "metric": f"prefix attention over an int{args.bits} cached prefix: TFLOP/s",
        "value": flops / tqz / 1e12, "unit": "TFLOP/s", "n_gpus": 1, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": tqz * 1e3, "higher_is_better": True, "op": "prefix_q", "dtype": w.dtype,
        "data": "synthetic",
        "config": {"workload": args.workload, "bits": args.bits, "quantized_pages": int(len(qid)),
                   "cached_prefix_bytes_16bit": float(len(qid) * page16),
                   "cached_prefix_bytes_quantized": float(len(qid) * pageq),
                   "splits": int(st.prefix_splits), "l2": "flushed before every timed call",
                   "launch": "CUDA graph replay of the one call"},
        "prefix_16bit_ms": t16 * 1e3, "speed_vs_16bit": t16 / tqz,
        "gpu_launches": 1 + (1 if st.prefix_splits > 1 else 0),
        "roofline": {"kernel": "prefix_attn_q", "bound": "tensor", "achieved": flops / tqz / 1e12, "peak": peak,
                     "unit": "TFLOP/s", "frac": flops / tqz / 1e12 / peak,
                     "peak_source": f"{peak_src} bf16 dense (burst); the products run in fp16 (same nominal rate)",
                     "traffic": committed_traffic(f"prefix_q_int{args.bits}", args.workload)},
    }
    print(json.dumps(line), flush=True)
    return 0


def run_blockmgr(args):
    """Host block manager throughput through the public binding: chunk
    hashing (SHA-256 chain) and a request stream -- admit a prompt that shares
    a 1024-token system prompt (8 cached chunks after the first request),
    8 decode appends, finish -- with the reference (plain Python) timed on a
    sample of the same stream as the CPU baseline."""
    import time

    import numpy as np

    from paged_prefix_reuse_gb300 import build as kvp_build

    kvp_build.build_library()
    import paged_prefix_reuse_gb300 as kvp

    kvp.load_library()
    kvp.kvp_set_launch_options(kvp.LAUNCH_PDL if args.pdl else 0)
    rng = np.random.default_rng(0)
    toks = rng.integers(0, 50000, size=1 << 20).astype(np.int32)
    kvp.kvp_hash_chunks(toks[:4096], 128)
    t0 = time.perf_counter()
    kvp.kvp_hash_chunks(toks, 128)
    t_hash = time.perf_counter() - t0
    system = rng.integers(0, 50000, size=1024).astype(np.int32)
    n_req = 2000
    prompts = [np.concatenate([system, rng.integers(0, 50000, size=256).astype(np.int32)]) for _ in range(n_req)]

    def stream(m, reqs, base):
        for i, p in enumerate(reqs):
            sid = base + i
            m.admit(sid, p)
            for _ in range(8):
                m.append(sid, 1)
            m.finish(sid, np.concatenate([p, np.full(8, 7, np.int32)]))

    native = kvp.BlockManager(65536, 16, 128)
    stream(native, prompts[:20], 10**6)  # warm: registers the system prompt's chunks
    t0 = time.perf_counter()
    stream(native, prompts, 0)
    t_native = time.perf_counter() - t0
    assert native.audit()
    from oracle import blockmgr as ref_bm

    model = ref_bm.BlockManager(65536, 16, 128)
    stream(model, prompts[:20], 10**6)
    k = 100
    t0 = time.perf_counter()
    stream(model, prompts[:k], 0)
    t_ref = time.perf_counter() - t0
    # a decode step of 64 running sequences: one batched call per step
    dec = kvp.BlockManager(65536, 16, 128)
    ids = np.arange(64, dtype=np.int64)
    for i in ids:
        dec.admit(int(i), prompts[int(i)])
    ones = np.ones(64, dtype=np.int32)
    dec.append_batch(ids, ones, max_blocks=256)
    t0 = time.perf_counter()
    n_steps = 1000
    for _ in range(n_steps):
        dec.append_batch(ids, ones, max_blocks=256)
    t_step = (time.perf_counter() - t0) / n_steps
    line = {
        "metric": "host block manager: requests/s (admit 1280 tokens with a shared 1024-token prefix, 8 appends, "
                  "finish)",
        "value": n_req / t_native, "unit": "req/s", "n_gpus": 0, "steps": n_req, "warmup": 20,
        "ms_per_step": 1e3 * t_native / n_req, "higher_is_better": True, "op": "blockmgr", "data": "synthetic",
        "config": {"workload": "shared 1024-token system prompt + 256 own tokens, chunk 128, block 16",
                   "num_blocks": 65536},
        "decode_step_us_64_seqs": t_step * 1e6,  # one append_batch call, 256-page tables
        "hash_mtokens_per_s": len(toks) / t_hash / 1e6,
        "hash_gbs": len(toks) * 4 * 2 / t_hash / 1e9,
        "gpu_launches": 0,
        "cpu_baseline": {"value": k / t_ref, "unit": "req/s", "cores": 1, "kind": "oracle",
                         "sample": f"{k} requests of the same stream through the plain-Python reference"},
    }
    print(json.dumps(line), flush=True)
    return 0


def run_cacheblend(args):
    """CacheBlend recompute selection on the RAG shape: every cached token of
    16 requests (8 retrieved 256-token chunks each, 32 kv heads, d=96, fp16)
    has its pool K/V compared with fresh K/V (deviation), the ~15% most
    deviated per request are selected and overwritten.  The deviation kernel
    is HBM-bound: it reads the cached and the fresh K and V of every token."""
    import numpy as np
    import torch

    torch.cuda.set_device(0)
    dev = torch.device("cuda", 0)
    from paged_prefix_reuse_gb300 import build as kvp_build

    kvp_build.build_library()
    import paged_prefix_reuse_gb300 as kvp
    from paged_prefix_reuse_gb300.step import DeviceStep

    kvp.load_library()
    kvp.kvp_set_launch_options(kvp.LAUNCH_PDL if args.pdl else 0)
    w = wl.make_config(3)
    st = DeviceStep(w, device=dev)
    pool = st.pool
    bs, hkv, d = pool.block_size, pool.num_kv_heads, pool.head_dim
    P = w.prefix_lens.astype(np.int64)
    slots = np.concatenate([w.block_tables[s][np.arange(P[s]) // bs].astype(np.int64) * bs + np.arange(P[s]) % bs
                            for s in range(w.B)])
    T = len(slots)
    cu = torch.from_numpy(np.concatenate([[0], np.cumsum(P)]).astype(np.int32)).to(dev)
    ts = torch.from_numpy(slots).to(dev)
    g = torch.Generator(device=dev).manual_seed(0)
    kf = torch.randn((T, hkv, d), generator=g, device=dev).half()
    vf = torch.randn((T, hkv, d), generator=g, device=dev).half()
    devv = torch.empty(T, dtype=torch.float32, device=dev)
    stream = torch.cuda.Stream(device=dev)
    flush = torch.empty(L2_FLUSH_BYTES // 4, dtype=torch.int32, device=dev)
    kp0, vp0 = pool.k.clone(), pool.v.clone()

    def timed(fn, reset=False):
        ts_ = []
        with torch.cuda.stream(stream):
            for i in range(args.warmup + args.steps):
                if reset:
                    pool.k.copy_(kp0)
                    pool.v.copy_(vp0)
                flush.zero_()
                e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                e0.record(stream)
                fn()
                e1.record(stream)
                e1.synchronize()
                if i >= args.warmup:
                    ts_.append(e0.elapsed_time(e1) / 1e3)
        return sorted(ts_)[len(ts_) // 2]

    t_dev = timed(lambda: kvp.kvp_kv_deviation(pool, kf, vf, ts, out=devv, stream=stream))
    sel = {}

    def do_sel():
        sel["rs"], sel["c"] = kvp.kvp_select_recompute(devv, ts, cu, 150, stream=stream)

    t_sel = timed(do_sel)
    t_ovw = timed(lambda: kvp.kvp_cache_append(pool, kf, vf, sel["rs"], stream=stream), reset=True)

    def whole():
        kvp.kvp_kv_deviation(pool, kf, vf, ts, out=devv, stream=stream)
        rs, _ = kvp.kvp_select_recompute(devv, ts, cu, 150, stream=stream)
        kvp.kvp_cache_append(pool, kf, vf, rs, stream=stream)

    t_all = timed(whole, reset=True)
    dev_bytes = 4.0 * T * hkv * d * 2  # cached K,V + fresh K,V
    nsel = int(sel["c"].sum().item())
    peaks, peak_src = load_peaks()
    hbm = _peak_value(peaks, "hbm_gbs") or FALLBACK_PEAKS["hbm_gbs"]
    gbs = dev_bytes / t_dev / 1e9
    line = {
        "metric": "CacheBlend selection: cached tokens/s (deviation + top-15% select + overwrite)",
        "value": T / t_all, "unit": "tokens/s", "n_gpus": 1, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": t_all * 1e3, "higher_is_better": True, "op": "cacheblend", "dtype": w.dtype,
        "data": "synthetic",
        "config": {"workload": "rag_chunk_reuse cached prefixes", "tokens": T, "selected": nsel,
                   "l2": "flushed before every timed call"},
        "deviation_ms": t_dev * 1e3, "select_ms": t_sel * 1e3, "overwrite_ms": t_ovw * 1e3, "gpu_launches": 3,
        "roofline": {"kernel": "kv_deviation", "bound": "hbm", "achieved": gbs, "peak": hbm, "unit": "GB/s",
                     "frac": gbs / hbm, "peak_source": f"{peak_src} HBM copy",
                     "traffic": committed_traffic("deviation", "rag_chunk_reuse_cached")},
    }
    print(json.dumps(line), flush=True)
    return 0


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1, help="GPUs of the run (replicas; launch N > 1 with torchrun)")
    ap.add_argument("--steps", type=int, default=20, help="timed steps")
    ap.add_argument("--warmup", type=int, default=5, help="untimed warm-up steps (at least 3)")
    ap.add_argument("--impl", choices=["kvp", "reference"], default="kvp",
                    help="kvp: the CUDA library; reference: the fp64 oracle on the host cores")
    ap.add_argument("--workload", choices=sorted(WORKLOADS), default="long_context_prefix",
                    help="synthetic batch shape (default: the long-context prefix batch, the largest)")
    ap.add_argument("--decode-workload", choices=sorted(WORKLOADS) + ["none"], default="continuous_batching_step",
                    help="when the workload has no decode sequences, time the decode batch of this one too "
                         "(reported as the line's decode object; none: skip)")
    ap.add_argument("--prefix-splits", type=int, default=0, help="split-KV count of prefix attention (0: the library's)")
    ap.add_argument("--decode-splits", type=int, default=0, help="split-KV count of decode (0: the library's)")
    ap.add_argument("--cpu-seconds", type=float, default=15.0, help="CPU time of the oracle baseline sample")
    ap.add_argument("--no-cpu-baseline", action="store_true", help="skip the timed oracle sample")
    ap.add_argument("--preroll-s", type=float, default=0.4,
                    help="seconds of untimed steps before timing, so the clock samples see load")
    ap.add_argument("--op", choices=["step", "block_swap", "decode_q", "prefix_q", "blockmgr", "cacheblend"],
                    default="step",
                    help="step: the prefill/decode step (default); block_swap: host <-> device page swap; "
                         "decode_q: decode over a quantized cached prefix; prefix_q: prefix attention over a "
                         "quantized cached prefix (--workload's prefill); blockmgr: host block manager; "
                         "cacheblend: CacheBlend recompute selection")
    ap.add_argument("--bits", type=int, choices=[8, 4], default=8,
                    help="quantized pool width for --op decode_q and --op prefix_q")
    ap.add_argument("--e2e-groups", type=int, default=0,
                    help="sequence groups of the host-buffer (e2e) step, each on its own stream (0: auto)")
    ap.add_argument("--pdl", type=int, choices=[0, 1], default=1,
                    help="1: programmatic dependent launch between the step's kernels (kvp_set_launch_options)")
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3
    if args.op == "block_swap":
        return run_swap(args)
    if args.op == "decode_q":
        return run_decode_q(args)
    if args.op == "prefix_q":
        return run_prefix_q(args)
    if args.op == "blockmgr":
        return run_blockmgr(args)
    if args.op == "cacheblend":
        return run_cacheblend(args)
    if args.impl == "reference":
        return run_reference(args)
    return run_kvp(args)


if __name__ == "__main__":
    sys.exit(main())
