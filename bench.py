"""Benchmark of the paged chunked-prefill hot path on GB300.

One step = slot mapping and KV append (one fused kernel) + paged extend
attention (device work planning, the tensor-core kernel and the split-KV row
kernel) over one batch
of the GQA chunked-prefill workload (Qwen3-8B-like attention: B=8, 32 query /
8 KV heads, head_dim 128, page_size 16, chunk 512, prefix ~U[0, 8192],
scattered pages), inputs resident in HBM.  The metric is effective TFLOP/s:
4 * head_dim * n_q_heads * (visible query/key pairs per head) per step -- only
unmasked QK^T and PV work counts.

Prints one JSON line.  Extra keys: roofline of the tensor-core kernel, the
oracle timed on the host cores (cpu_baseline), an end-to-end figure through
the C ABI with host buffers, the decode-row and KV-append bandwidths, and
the SM clocks sampled during the timed region.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "extend-attn effective TFLOP/s"
UNIT = "TFLOP/s"


def visible_pairs(prefix_lens, chunk_lens, window: int) -> int:
    """Query/key pairs one head attends to (closed form per sequence)."""
    total = 0
    for P, c in zip(np.asarray(prefix_lens, np.int64), np.asarray(chunk_lens, np.int64)):
        p = P + np.arange(c, dtype=np.int64)
        n = p + 1
        if window > 0:
            n = np.minimum(n, window)
        total += int(n.sum())
    return total


def rows_pairs(batch, tok, head) -> int:
    """Visible pairs of selected (row, head) samples."""
    b_of = np.searchsorted(batch.qo_indptr, tok, side="right") - 1
    p = batch.prefix_lens[b_of].astype(np.int64) + (tok - batch.qo_indptr[b_of])
    n = p + 1
    if batch.window > 0:
        n = np.minimum(n, batch.window)
    return int(n.sum())


# DRAM traffic (dram__bytes_read.sum + dram__bytes_write.sum) of one launch of
# the dominant kernel, from an ncu capture of this bench on the named workload.
# It is reported only while the sources that build, plan and launch that
# kernel hash to the value the capture ran with; after a change there the key
# reads null until the counters are taken again.
NCU_TRAFFIC = {
    ("gqa_prefill", "extend_tc_kernel<128>"): {
        "bytes": 197.944576e6 + 13.285120e6,
        "sources_sha256": "65866cc5b44b23d79dfe5db669164ad2",
    },
    ("long_context", "extend_tc_kernel<128>"): {
        "bytes": 4086.055936e6 + 532.024576e6,
        "sources_sha256": "65866cc5b44b23d79dfe5db669164ad2",
    },
    ("mixed", "extend_tc_kernel<128>"): {
        "bytes": 307.345408e6 + 3.377408e6,
        "sources_sha256": "65866cc5b44b23d79dfe5db669164ad2",
    },
    ("decode_rows", "row_attn_kernel<128>"): {
        "bytes": 275.760384e6 + 0.564736e6,
        "sources_sha256": "706c6fde763ecf2d3b22a9ec4691b98e",
    },
}

# The sources behind a kernel's counters: its own file, the planner (item
# order and split), the host side that sets up its launch, and the shared
# device headers.
COMMON_SOURCES = ("pcp_api.cu", "pcp_plan.cu", "pcp_device.cuh", "pcp_internal.h",
                  "pcp_launch.h")
KERNEL_SOURCES = {"extend_tc_kernel": "pcp_extend_tc.cu", "row_attn_kernel": "pcp_rows.cu"}


def sources_sha256(kernel: str) -> str:
    """Hash of the sources behind one kernel's counters (kernel named with or
    without its template arguments)."""
    import hashlib
    d = os.path.join(ROOT, "paged_chunked_prefill_gb300", "csrc")
    h = hashlib.sha256()
    for name in sorted(COMMON_SOURCES + (KERNEL_SOURCES[kernel.split("<")[0]],)):
        h.update(name.encode())
        with open(os.path.join(d, name), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:32]


def ncu_traffic(workload: str, kernel: str):
    rec = NCU_TRAFFIC.get((workload, kernel))
    if rec is None or rec["sources_sha256"] != sources_sha256(kernel):
        return None
    return rec["bytes"]


def to_device(batch, dev):
    """The workload's arrays as device tensors (bf16 bit patterns and int32)."""
    import torch
    t16 = lambda a: torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(
        torch.bfloat16).to(dev)
    i32 = lambda a: torch.from_numpy(np.ascontiguousarray(a, dtype=np.int32)).to(dev)
    nonempty = lambda a: a if len(a) else np.zeros(1, np.int32)
    return dict(q=t16(batch.q), k_new=t16(batch.k_new), v_new=t16(batch.v_new),
                k_pool=t16(batch.k_pool), v_pool=t16(batch.v_pool),
                qo_indptr=i32(batch.qo_indptr), kv_indptr=i32(batch.kv_indptr),
                kv_indices=i32(nonempty(batch.kv_indices)),
                prefix_lens=i32(nonempty(batch.prefix_lens)))


def row_max_chunk(batch) -> int:
    """Longest chunk the split-KV row kernel takes (decode-shaped rows)."""
    G = batch.n_q_heads // batch.n_kv_heads
    return 16 // G if G <= 16 else 0


def split_work(batch):
    """(visible pairs per head of the chunks the tensor-core kernel takes,
    algorithmic bytes of the decode-shaped rows the row kernel takes: the K/V
    of every visible key once per KV head, q, out, lse and page ids)."""
    c = batch.chunk_lens.astype(np.int64)
    P = batch.prefix_lens.astype(np.int64)
    rmax = row_max_chunk(batch)
    tc = c > rmax
    tc_pairs = visible_pairs(P[tc], c[tc], batch.window)
    rows = (c > 0) & ~tc
    D, Hkv, Hq = batch.head_dim, batch.n_kv_heads, batch.n_q_heads
    first = np.maximum(0, P[rows] - batch.window + 1) if batch.window > 0 else 0 * P[rows]
    keys = (P[rows] + c[rows] - first).sum()
    pages = 0
    for b in np.nonzero(rows)[0]:
        pages += -(-(int(P[b] + c[b])) // batch.page_size)
    n_rows = int(c[rows].sum())
    row_bytes = int(keys) * Hkv * D * 2 * 2 + n_rows * Hq * (D * 2 * 2 + 4) + 4 * pages
    return tc_pairs, row_bytes


def launches_per_step(batch, rows_on_tensor_cores: bool = False) -> int:
    """Library kernels one step (the attention call with the step's new K/V
    rows and host copies of qo_indptr and prefix_lens) launches: the planner
    with the append beside it, or the append alone when the row kernel plans
    a decode-only call of at most 512 sequences itself; the tensor-core
    kernel for chunks above the row path's size; the row kernel and the
    combine for decode-shaped chunks unless they joined the tensor cores."""
    G = batch.n_q_heads // batch.n_kv_heads
    rmax = 16 // G if G <= 16 else 0
    c = np.diff(batch.qo_indptr)
    tc = bool((c > rmax).any())
    rows = bool(((c > 0) & (c <= rmax)).any()) and not rows_on_tensor_cores
    return 1 + int(tc) + 2 * int(rows)


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        d = json.load(open(path))
        return d, "measured"
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}, "fallback"


class ClockSampler:
    """nvidia-smi clocks and throttle reasons, sampled every 200 ms."""

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.path = None

    def __enter__(self):
        fd, self.path = tempfile.mkstemp(suffix=".csv")
        os.close(fd)
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index),
                 "--query-gpu=clocks.sm,clocks.max.sm,clocks_event_reasons.active,"
                 "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
                 "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap",
                 "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None
        time.sleep(0.3)
        return self

    def __exit__(self, *a):
        if self.proc is not None:
            time.sleep(0.25)
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()

    def summary(self):
        if self.proc is None or self.path is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unavailable"]}
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in open(self.path):
            f = [x.strip() for x in line.split(",")]
            if len(f) < 7:
                continue
            try:
                sm.append(float(f[0]))
                mx.append(float(f[1]))
            except ValueError:
                continue
            for n, v in zip(names, f[3:7]):
                if v.lower() == "active":
                    reasons.add(n)
        os.unlink(self.path)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx),
                "reasons": sorted(reasons), "samples": len(sm)}


class L2Flush:
    """Flush of the 129 MB L2 before a timed step: write a 256 MB buffer, then
    read it back, so nothing of the previous step stays in L2 and no dirty
    line of the flush is left for the timed step to write back."""

    def __init__(self, torch, dev):
        self.torch = torch
        self.buf = torch.empty(256 * 1024 * 1024 // 4, dtype=torch.float32, device=dev)
        self.out = torch.empty((), dtype=torch.float32, device=dev)

    def __call__(self):
        self.buf.zero_()
        self.torch.sum(self.buf, dim=0, out=self.out)


def max_over_ranks(torch, value: float, world: int, device) -> float:
    """The largest of every rank's value (all_reduce MAX; the value itself on
    one rank).  Used for step times: the whole job is as slow as its slowest
    rank."""
    if world <= 1:
        return float(value)
    t = torch.tensor([float(value)], dtype=torch.float64, device=device)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return float(t.item())


def whole_job_rate(units_per_rank: float, world: int, ms: float) -> float:
    """Units per second of the whole job: every rank processes its own
    replica's units (weak scaling) in at most `ms` milliseconds."""
    return world * units_per_rank / (ms * 1e-3)


def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def oracle_sample(batch, seconds_target: float, seed: int = 0, detail: bool = False):
    """Time the FP64 oracle on a bounded sample of rows of `batch` (appended
    pools).  Returns (TFLOP/s of effective work, threads, sample text), plus
    the seconds spent and the (row, head) pairs done with detail=True."""
    import oracle
    loc = oracle.out_cache_loc(batch.qo_indptr, batch.kv_indptr, batch.kv_indices,
                               batch.prefix_lens, batch.page_size, batch.num_pages)
    kp, vp = batch.k_pool.copy(), batch.v_pool.copy()
    oracle.kv_append(batch.k_new, batch.v_new, loc, kp, vp)
    rng = np.random.default_rng(seed)
    D, Hq = batch.head_dim, batch.n_q_heads
    n = 64
    elapsed, done_flops, rows = 0.0, 0, 0
    while elapsed < seconds_target:
        tok = rng.integers(0, batch.total_q, size=n)
        head = rng.integers(0, Hq, size=n).astype(np.int32)
        t0 = time.perf_counter()
        oracle.paged_extend_attn(batch.q, batch.qo_indptr, batch.kv_indptr, batch.kv_indices,
                                 batch.prefix_lens, kp, vp, batch.page_size, Hq,
                                 batch.n_kv_heads, D, batch.window, batch.sm_scale,
                                 rows=(tok, head))
        elapsed += time.perf_counter() - t0
        done_flops += 4 * D * rows_pairs(batch, tok, head)
        rows += n
        n = min(n * 2, 4096)
    res = (done_flops / elapsed / 1e12, oracle.num_threads(),
           f"{rows} random (row, head) pairs of the workload, {elapsed:.1f} s")
    return res + (elapsed, rows) if detail else res


def config_dict(batch, world: int) -> dict:
    """The workload description both arms print."""
    return {"workload": batch.name, "global_batch": batch.batch * world,
            "tokens_per_step": batch.total_q * world,
            "visible_pairs_per_head": visible_pairs(batch.prefix_lens, batch.chunk_lens,
                                                    batch.window),
            "l2": "flushed before every timed step: 256 MB written, then read back",
            "parallelism": f"replicas x{world}" if world > 1 else "single GPU"}


def run_reference(args):
    """Reference arm: the FP64 oracle on the host cores.  Each step runs the
    oracle on a bounded random sample of (row, head) pairs of the workload
    (about 60 s of oracle time over the whole run); the value is the
    effective TFLOP/s of that sample, ms_per_step the oracle time actually
    spent per step, and ms_per_step_extrapolated the time a whole step of the
    workload would take at that rate."""
    world, rank, _ = dist_env()
    if rank != 0:
        return
    import workloads as W
    batch = W.config_by_name(args.workload)
    per_step = max(1.0, 60.0 / max(1, args.steps + args.warmup))
    vals, secs, rows = [], [], []
    for i in range(args.warmup + args.steps):
        v, cores, sample, spent, n = oracle_sample(batch, per_step, seed=i, detail=True)
        if i >= args.warmup:
            vals.append(v)
            secs.append(spent)
            rows.append(n)
    value = float(np.mean(vals))
    flops = 4 * batch.head_dim * batch.n_q_heads * visible_pairs(
        batch.prefix_lens, batch.chunk_lens, batch.window)
    ms = float(np.mean(secs)) * 1e3
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT,
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": ms,
        "ms_per_step_extrapolated": flops / (value * 1e12) * 1e3,
        "ms_per_step_note": "ms_per_step is the oracle time spent per step on its sample; "
                            "ms_per_step_extrapolated is a whole step of the workload at the "
                            "sample's rate (extrapolated, not measured)",
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic",
        "config": config_dict(batch, world),
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": cores, "kind": "oracle",
                         "sample": f"per step: {int(np.mean(rows))} random (row, head) pairs "
                                   f"of the workload, {ms / 1e3:.2f} s of oracle time"},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--cpu-seconds", type=float, default=15.0)
    ap.add_argument("--no-secondary", action="store_true")
    ap.add_argument("--workload", default="gqa_prefill",
                    help="workloads.CONFIGS name (the headline line uses gqa_prefill)")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--only", default=None, choices=SECONDARY_KEYS,
                    help="run one secondary measurement alone and print it (no headline line; "
                         "for profiling its kernels)")
    args = ap.parse_args()
    if args.impl == "reference":
        return run_reference(args)

    import torch
    import paged_chunked_prefill_gb300 as pcp
    import workloads as W

    world, rank, local = dist_env()
    if world > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl")
    dev = torch.device("cuda", torch.cuda.current_device())
    args.warmup = max(args.warmup, 3)
    if args.only is not None:
        peaks, peak_kind = load_peaks()
        res = secondary(pcp, torch, W, dev, peaks, peak_kind, L2Flush(torch, dev),
                        only=args.only)
        if rank == 0:
            print(json.dumps({"only": args.only, "secondary": res}))
        return

    batch = W.config_by_name(args.workload)
    d = to_device(batch, dev)
    flops = 4 * batch.head_dim * batch.n_q_heads * visible_pairs(
        batch.prefix_lens, batch.chunk_lens, batch.window)
    ws = torch.empty(pcp.workspace_size(batch.batch, batch.total_q, batch.n_q_heads,
                                        batch.n_kv_heads, batch.head_dim),
                     dtype=torch.uint8, device=dev)
    err = torch.zeros(1, dtype=torch.int32, device=dev)
    out = torch.empty_like(d["q"])
    lse = torch.empty(batch.total_q, batch.n_q_heads, dtype=torch.float32, device=dev)
    flush = L2Flush(torch, dev)

    def step(tc_events=None):
        # one call: the append of the step's new K/V rows (in the planner's
        # launch) and the attention over the pools
        pcp.paged_extend_attn(d["q"], d["qo_indptr"], d["kv_indptr"],
                              d["kv_indices"], d["prefix_lens"], d["k_pool"], d["v_pool"],
                              batch.page_size, batch.n_q_heads, batch.n_kv_heads,
                              batch.head_dim, batch.window, batch.sm_scale, out=out, lse=lse,
                              workspace=ws, dev_err=err, qo_indptr_host=batch.qo_indptr,
                              prefix_lens_host=batch.prefix_lens, tc_events=tc_events,
                              k_new=d["k_new"], v_new=d["v_new"])

    stream = torch.cuda.current_stream(dev)
    for _ in range(args.warmup):
        # the flush too: its kernels load on first use, which must not fall
        # inside the first timed step
        flush()
        step()
    torch.cuda.synchronize()
    if pcp.read_error(err) != 0:
        raise RuntimeError(f"device error {pcp.read_error(err)} during warm-up")
    # where the decode-shaped chunks ran (the planner's header: n_row_groups)
    c = np.diff(batch.qo_indptr)
    rmax = row_max_chunk(batch)
    rows_on_tc = bool((c > rmax).any() and ((c > 0) & (c <= rmax)).any() and
                      int(ws[4:8].view(torch.int32).item()) == 0)

    # ---- timed region: L2 flushed before every step, events around each step
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True),
           torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(args.steps)]
    for e in ev:  # materialise the events before handing them to the library
        for x in e:
            x.record(stream)
    with ClockSampler(dev.index) as clocks:
        # the GPU idled while the sampler started (0.3 s): one more untimed
        # step brings its clocks back before the timed ones
        flush()
        step()
        torch.cuda.synchronize()
        if world > 1:
            torch.distributed.barrier()
        torch.cuda.synchronize()
        # (1) whole steps: nothing between the library's launches, so each
        # kernel's launch overlaps the end of the one before it.  After the
        # synchronize the host must get ahead of the GPU again before the
        # first timed step: two more untimed flushes (about 160 us of GPU
        # work) give it that lead (with one, the first step sometimes ran
        # 15-45 us long while the GPU waited for its launches)
        for i in range(args.steps):
            if i == 0:
                flush()
                flush()
            flush()
            ev[i][0].record(stream)
            step()
            ev[i][1].record(stream)
        torch.cuda.synchronize()
        # (2) the same steps again with events around the tensor-core kernel
        # (they serialise its two neighbours, so they stay out of loop 1)
        for i in range(args.steps):
            if i == 0:
                flush()
                flush()
            flush()
            step(tc_events=(ev[i][2], ev[i][3]))
        torch.cuda.synchronize()
    step_ms = [a.elapsed_time(b) for a, b, _, _ in ev]
    tc_ms = [c.elapsed_time(e) for _, _, c, e in ev]
    total_ms = float(sum(step_ms))
    total_ms = max_over_ranks(torch, total_ms, world, dev)
    if world > 1:
        torch.distributed.barrier()
    code = pcp.read_error(err)
    if code != 0:
        raise RuntimeError(f"device error {code} in the timed region")
    ms_per_step = total_ms / args.steps
    value = whole_job_rate(flops, world, ms_per_step) / 1e12

    peaks, peak_kind = load_peaks()
    tc_avg = float(np.mean(tc_ms))
    if (np.diff(batch.qo_indptr) > row_max_chunk(batch)).any():
        tc_flops = 4 * batch.head_dim * batch.n_q_heads * split_work(batch)[0]
        achieved = tc_flops / (tc_avg * 1e-3) / 1e12
        roofline = {"bound": "tensor", "achieved": achieved, "peak": peaks["bf16_tflops"],
                    "unit": UNIT, "frac": achieved / peaks["bf16_tflops"],
                    "traffic": ncu_traffic(args.workload, f"extend_tc_kernel<{batch.head_dim}>"),
                    "kernel": f"extend_tc_kernel<{batch.head_dim}>", "kernel_ms": tc_avg,
                    "peak_source": f"{peak_kind} bf16 dense (burst)"}
    else:  # decode-shaped rows only: no tensor-core launch to time
        roofline = None

    # ---- end to end through the C ABI with pinned host buffers
    e2e = None
    if not args.no_e2e:
        e2e = end_to_end(args, torch, pcp, batch, d, out, flush, stream, flops, world)

    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms_per_step,
        "ms_steps": [round(x, 4) for x in step_ms], "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": config_dict(batch, world),
        "roofline": roofline,
        "e2e": e2e,
        # the planner with the append beside it (or the append kernel), then
        # the tensor-core kernel and/or the row kernel + combine (the host
        # copy of qo_indptr skips a kernel without work), in each of the two
        # timed loops
        "gpu_launches": 2 * args.steps * launches_per_step(batch, rows_on_tc),
        "clocks": clocks.summary(),
    }

    if not args.no_secondary and rank == 0:
        line["secondary"] = secondary(pcp, torch, W, dev, peaks, peak_kind, flush)
    if rank == 0 and world == 1:
        v, cores, sample = oracle_sample(batch, args.cpu_seconds)
        line["cpu_baseline"] = {"value": v, "unit": UNIT, "cores": cores, "kind": "oracle",
                                "sample": sample}
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        torch.distributed.destroy_process_group()


def end_to_end(args, torch, pcp, batch, d, out_ref, flush, stream, flops, world):
    """The step through the public API from pinned host memory: every step
    copies its inputs (q, the chunk's K/V, the page-table metadata) host to
    device and reads out and lse back device to host, inside the timed region.

    As a serving loop runs it, the copies go on streams of their own, so step
    i's kernels overlap step i+1's input copies and step i-1's read-back.
    Three buffer sets (inputs, KV pools, outputs, workspace) rotate between
    the steps, so a step finds in L2 at most the inputs just copied for it,
    never the pools or outputs of the step before.  A set is refilled once the
    read-back of its previous step has finished; with three sets that wait
    does not chain one step's copies, kernels and read-back to the next's.

    The inputs travel as one pinned buffer and out / lse come back as one, so
    a step makes one copy each way.

    Also reported: the same step run alone (copies, kernels, read-back one
    after the other, L2 flushed before it)."""
    # one pinned input buffer (q, the chunk's K/V, the metadata) and one
    # output buffer (out, lse) per step, each moved by one copy: the copy
    # engines pay a fixed cost per copy
    inputs = ("q", "k_new", "v_new", "qo_indptr", "kv_indptr", "kv_indices", "prefix_lens")
    dev = d["q"].device

    def layout(tensors):
        offs, off = [], 0
        for t in tensors:
            offs.append(off)
            off += (t.numel() * t.element_size() + 255) // 256 * 256
        return offs, off

    def views(buf, offs, likes):
        return [buf[o:o + t.numel() * t.element_size()].view(t.dtype).view(t.shape)
                for o, t in zip(offs, likes)]

    in_offs, in_bytes = layout([d[n] for n in inputs])
    h_in = torch.empty(in_bytes, dtype=torch.uint8).pin_memory()
    for hv, n in zip(views(h_in, in_offs, [d[n] for n in inputs]), inputs):
        hv.copy_(d[n].cpu())
    h2d = in_bytes
    out_like = [torch.empty_like(d["q"]),
                torch.empty(batch.total_q, batch.n_q_heads, dtype=torch.float32, device=dev)]
    out_offs, out_bytes = layout(out_like)
    ws_bytes = pcp.workspace_size(batch.batch, batch.total_q, batch.n_q_heads, batch.n_kv_heads,
                                  batch.head_dim)
    err = torch.zeros(1, dtype=torch.int32, device=dev)
    n_sets = 3
    sets = []
    for _ in range(n_sets):
        S = {"in": torch.empty(in_bytes, dtype=torch.uint8, device=dev),
             "res": torch.empty(out_bytes, dtype=torch.uint8, device=dev),
             "h_res": torch.empty(out_bytes, dtype=torch.uint8).pin_memory()}
        S.update(zip(inputs, views(S["in"], in_offs, [d[n] for n in inputs])))
        S["out"], S["lse"] = views(S["res"], out_offs, out_like)
        S["h_out"], S["h_lse"] = views(S["h_res"], out_offs, out_like)
        S["k_pool"] = d["k_pool"].clone()
        S["v_pool"] = d["v_pool"].clone()
        S["ws"] = torch.empty(ws_bytes, dtype=torch.uint8, device=dev)
        sets.append(S)
    d2h = out_bytes

    def h2d_copies(S):
        S["in"].copy_(h_in, non_blocking=True)

    def kernels(S):
        pcp.paged_extend_attn(S["q"], S["qo_indptr"], S["kv_indptr"], S["kv_indices"],
                              S["prefix_lens"], S["k_pool"], S["v_pool"], batch.page_size,
                              batch.n_q_heads, batch.n_kv_heads, batch.head_dim, batch.window,
                              batch.sm_scale, out=S["out"], lse=S["lse"], workspace=S["ws"],
                              dev_err=err, qo_indptr_host=batch.qo_indptr,
                              prefix_lens_host=batch.prefix_lens, k_new=S["k_new"],
                              v_new=S["v_new"])

    def d2h_copies(S):
        S["h_res"].copy_(S["res"], non_blocking=True)

    s_in, s_back = torch.cuda.Stream(dev), torch.cuda.Stream(dev)

    def pipeline(n, t0=None, t1=None):
        ev_in = [torch.cuda.Event() for _ in range(n)]
        ev_run = [torch.cuda.Event() for _ in range(n)]
        ev_back = [torch.cuda.Event() for _ in range(n)]
        if t0 is not None:
            t0.record(s_in)
        for i in range(n):
            S = sets[i % n_sets]
            with torch.cuda.stream(s_in):
                if i >= n_sets:
                    s_in.wait_event(ev_back[i - n_sets])
                h2d_copies(S)
                ev_in[i].record(s_in)
            stream.wait_event(ev_in[i])
            kernels(S)
            ev_run[i].record(stream)
            with torch.cuda.stream(s_back):
                s_back.wait_event(ev_run[i])
                d2h_copies(S)
                ev_back[i].record(s_back)
        if t1 is not None:
            t1.record(s_back)

    pipeline(max(args.warmup, 3))
    torch.cuda.synchronize()
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    pipeline(args.steps, t0, t1)
    torch.cuda.synchronize()
    e2e_ms = max_over_ranks(torch, t0.elapsed_time(t1) / args.steps, world, dev)
    if pcp.read_error(err) != 0:
        raise RuntimeError("device error in the end-to-end loop")
    # the loop computed and read back what the device-resident steps did
    for S in sets:
        if not (torch.equal(S["out"], out_ref) and torch.equal(S["h_out"], out_ref.cpu())):
            raise RuntimeError("end-to-end loop output differs from the device-resident step")
    e2e_value = whole_job_rate(flops, world, e2e_ms) / 1e12

    # the same step alone: copies, kernels and read-back one after the other
    S = sets[0]
    alone = []
    for _ in range(args.steps):
        flush()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        h2d_copies(S)
        kernels(S)
        d2h_copies(S)
        b.record(stream)
        b.synchronize()
        alone.append(a.elapsed_time(b))
    alone_ms = max_over_ranks(torch, float(np.mean(alone)), world, dev)

    return {"value": e2e_value, "unit": UNIT, "h2d_bytes_per_step": int(h2d),
            "d2h_bytes_per_step": int(d2h), "ms_per_step": e2e_ms,
            "loop": "copies on their own streams overlap the neighbouring steps' kernels; "
                    "three buffer sets (inputs, KV pools, outputs) rotate",
            "alone_ms_per_step": alone_ms}


def attn_figures(pcp, torch, batch, dev, peaks, flush, err, n=20, warm=5, causal=True,
                 mask=None, pairs=None, key=None, computed_pairs=None):
    """One attention call on `batch` (its chunk's K/V appended first), L2
    flushed before each timed call: the whole call, and the tensor-core and
    row kernels alone between per-call events.  Effective FLOPs count the
    visible pairs only (`pairs` per head when a mask hides more keys).  With
    a boolean mask the kernel still multiplies every pair its causal range
    holds and drops the masked ones in the softmax: `computed_pairs` (per
    head) gives that figure too, the rate at which the tensor cores work."""
    d = to_device(batch, dev)
    loc = pcp.compute_out_cache_loc(d["qo_indptr"], d["kv_indptr"], d["kv_indices"],
                                    d["prefix_lens"], batch.page_size, batch.num_pages)
    pcp.kv_append(d["k_new"], d["v_new"], loc, d["k_pool"], d["v_pool"], dev_err=err)
    out = torch.empty_like(d["q"])
    lse = torch.empty(batch.total_q, batch.n_q_heads, dtype=torch.float32, device=dev)
    ws = torch.empty(pcp.workspace_size(batch.batch, batch.total_q, batch.n_q_heads,
                                        batch.n_kv_heads, batch.head_dim),
                     dtype=torch.uint8, device=dev)
    mask_t = None if mask is None else torch.from_numpy(mask).to(dev)

    def call(tc_ev=None, row_ev=None):
        pcp.paged_extend_attn(d["q"], d["qo_indptr"], d["kv_indptr"], d["kv_indices"],
                              d["prefix_lens"], d["k_pool"], d["v_pool"], batch.page_size,
                              batch.n_q_heads, batch.n_kv_heads, batch.head_dim, batch.window,
                              batch.sm_scale, out=out, lse=lse, workspace=ws, dev_err=err,
                              qo_indptr_host=batch.qo_indptr,
                              prefix_lens_host=batch.prefix_lens, causal=causal, mask=mask_t,
                              tc_events=tc_ev, rows_events=row_ev)
    tc_pairs, row_bytes = split_work(batch)
    all_pairs = visible_pairs(batch.prefix_lens, batch.chunk_lens, batch.window)
    # the plan the call made (workspace header: n_tc_items, n_row_groups;
    # written by the planner kernel, which a call with tensor-core work
    # runs): decode-shaped chunks that joined the tensor-core queue count there
    call()
    n_tc_items, n_row_groups = (int(x) for x in ws[:8].view(torch.int32).cpu().tolist())
    absorbed = tc_pairs > 0 and row_bytes > 0 and n_row_groups == 0
    if absorbed:
        tc_pairs, row_bytes = all_pairs, 0
    if pairs is not None:  # a mask or non-causal call: all its work is on the tensor cores
        all_pairs = tc_pairs = pairs
    D, Hq = batch.head_dim, batch.n_q_heads
    ms = time_calls(torch, lambda ev: call(), flush, n=n, warm=warm)
    r = {"workload": batch.name, "ms": ms,
         "TFLOP/s": 4 * D * Hq * all_pairs / (ms * 1e-3) / 1e12,
         "what": "whole call (planner, kernels, combine), effective FLOPs of visible pairs",
         **({"tc_items": n_tc_items, "row_groups": n_row_groups} if tc_pairs > 0 else {})}
    if absorbed:
        r["decode_rows_on_tensor_cores"] = True
    r["frac_bf16"] = r["TFLOP/s"] / peaks["bf16_tflops"]
    if tc_pairs > 0:
        kms = time_calls(torch, lambda ev: call(tc_ev=ev), flush, n=n, warm=warm, events=True)
        tf = 4 * D * Hq * tc_pairs / (kms * 1e-3) / 1e12
        r["tc_kernel"] = {"bound": "tensor", "kernel": f"extend_tc_kernel<{D}>",
                          "kernel_ms": kms, "achieved": tf, "peak": peaks["bf16_tflops"],
                          "unit": "TFLOP/s", "frac": tf / peaks["bf16_tflops"],
                          "visible_pairs_per_head": int(tc_pairs),
                          "traffic": ncu_traffic(key, f"extend_tc_kernel<{D}>") if key else None}
        if computed_pairs is not None:
            ctf = 4 * D * Hq * computed_pairs / (kms * 1e-3) / 1e12
            r["tc_kernel"].update({
                "computed_pairs_per_head": int(computed_pairs), "computed_TFLOP/s": ctf,
                "frac_computed": ctf / peaks["bf16_tflops"],
                "what_computed": "every causal pair multiplied, masked ones included: the "
                                 "tensor-core rate; frac counts the kept pairs only"})
    if row_bytes > 0 and pairs is None:
        kms = time_calls(torch, lambda ev: call(row_ev=ev), flush, n=n, warm=warm, events=True)
        gbs = row_bytes / (kms * 1e-3) / 1e9
        r["row_kernel"] = {"bound": "hbm", "kernel": f"row_attn_kernel<{D}>", "kernel_ms": kms,
                           "achieved": gbs, "peak": peaks["hbm_gbs"], "unit": "GB/s",
                           "frac": gbs / peaks["hbm_gbs"], "bytes": int(row_bytes),
                           "traffic": ncu_traffic(key, f"row_attn_kernel<{D}>") if key else None}
    return r


SECONDARY_KEYS = ("decode_rows", "decode_step", "kv_append", "kv_append_long",
                  "long_context_attn", "mixed_attn", "gqa_prefill_ps1", "stress_ps1_w4096",
                  "stress_ps1_w0", "stress_ps16_w4096", "stress_ps16_w0", "masked",
                  "chunk_planner", "cow_page_copy")


def decode_step_secondary(pcp, torch, db, dev, peaks, flush, err, res):
    """The decode rows as a serving decode step: one attention call with
    their new tokens, appended by the append kernel ahead of the row kernel
    (which plans the call while the append runs)."""
    _, nbytes = split_work(db)
    g = to_device(db, dev)
    dout = torch.empty_like(g["q"])
    dlse = torch.empty(db.total_q, db.n_q_heads, dtype=torch.float32, device=dev)
    dws = torch.empty(pcp.workspace_size(db.batch, db.total_q, db.n_q_heads, db.n_kv_heads,
                                         db.head_dim), dtype=torch.uint8, device=dev)

    def dstep(ev):
        pcp.paged_extend_attn(g["q"], g["qo_indptr"], g["kv_indptr"], g["kv_indices"],
                              g["prefix_lens"], g["k_pool"], g["v_pool"], db.page_size,
                              db.n_q_heads, db.n_kv_heads, db.head_dim, db.window, db.sm_scale,
                              out=dout, lse=dlse, workspace=dws, dev_err=err,
                              qo_indptr_host=db.qo_indptr, prefix_lens_host=db.prefix_lens,
                              k_new=g["k_new"], v_new=g["v_new"])
    ms = time_calls(torch, dstep, flush)
    sbytes = nbytes + 2 * 2 * db.total_q * db.n_kv_heads * db.head_dim * 2
    gbs = sbytes / (ms * 1e-3) / 1e9
    res["decode_step"] = {"workload": db.name, "ms": ms, "GB/s": gbs,
                          "frac_hbm": gbs / peaks["hbm_gbs"], "bytes": sbytes,
                          "what": "the attention call with the rows' new tokens appended in it"}
    del g, dout, dlse, dws


def secondary(pcp, torch, W, dev, peaks, peak_kind, flush, only=None):
    """Per-kernel figures on every workload the benchmark does not time as
    its headline, L2 flushed before each call (`only`: one of
    SECONDARY_KEYS, e.g. to profile its kernels alone)."""
    res = {"peak_source": f"{peak_kind} (MEASURED_PEAKS.json when present): bf16 dense "
                          f"burst {peaks['bf16_tflops']} TFLOP/s, HBM copy {peaks['hbm_gbs']} GB/s"}
    err = torch.zeros(1, dtype=torch.int32, device=dev)

    def want(key):
        return only is None or only == key

    # decode rows: the 31 decode rows of the mixed batch as a decode-only call
    db = W.decode_rows()
    if want("decode_rows"):
        r = attn_figures(pcp, torch, db, dev, peaks, flush, err, key="decode_rows")
        _, nbytes = split_work(db)
        gbs = nbytes / (r["ms"] * 1e-3) / 1e9
        res["decode_rows"] = {"workload": db.name, "ms": r["ms"], "GB/s": gbs,
                              "frac_hbm": gbs / peaks["hbm_gbs"], "bytes": nbytes,
                              "what": "whole call: row kernel (planning its own split), "
                                      "split-KV combine"}
        res["decode_rows_kernel"] = r["row_kernel"]
    if want("decode_step"):
        decode_step_secondary(pcp, torch, db, dev, peaks, flush, err, res)


    # the KV append of the GQA chunk (4096 tokens) and of the long-context
    # chunk (32768 tokens): the fused slot mapping + append the step runs, and
    # the append alone from a precomputed out_cache_loc
    for key, bf in (("kv_append", W.gqa_prefill), ("kv_append_long", W.long_context)):
        if not want(key):
            continue
        b = bf()
        g = to_device(b, dev)
        loc = pcp.compute_out_cache_loc(g["qo_indptr"], g["kv_indptr"], g["kv_indices"],
                                        g["prefix_lens"], b.page_size, b.num_pages)
        kv_bytes = 2 * 2 * b.total_q * b.n_kv_heads * b.head_dim * 2
        what = f"{b.total_q} tokens x {b.n_kv_heads} KV heads x D {b.head_dim}"
        ms = time_calls(torch, lambda ev: pcp.kv_append_paged(
            g["qo_indptr"], g["kv_indptr"], g["kv_indices"], g["prefix_lens"], b.page_size,
            g["k_new"], g["v_new"], g["k_pool"], g["v_pool"], dev_err=err), flush)
        gbs = kv_bytes / (ms * 1e-3) / 1e9
        res[key] = {"workload": what, "ms": ms, "GB/s": gbs,
                    "frac_hbm": gbs / peaks["hbm_gbs"], "bytes": kv_bytes,
                    "what": "pcp_kv_append_paged: slot mapping and append in one kernel"}
        ms = time_calls(torch, lambda ev: pcp.kv_append(g["k_new"], g["v_new"], loc,
                                                        g["k_pool"], g["v_pool"], dev_err=err),
                        flush)
        nbytes = kv_bytes + 8 * b.total_q
        gbs = nbytes / (ms * 1e-3) / 1e9
        res[key + "_from_loc"] = {"workload": what, "ms": ms, "GB/s": gbs,
                                  "frac_hbm": gbs / peaks["hbm_gbs"], "bytes": nbytes,
                                  "what": "pcp_kv_append from a precomputed out_cache_loc"}
        del g, loc

    # the long-context batch, the mixed scheduler batch (prompt chunks on the
    # tensor cores beside decode rows in one call), the GQA workload over the
    # flat one-slot-per-token pool (page size 1), and the page-boundary and
    # window stress batches
    if want("long_context_attn"):
        res["long_context_attn"] = attn_figures(pcp, torch, W.long_context(), dev, peaks, flush,
                                                err, n=5, warm=2, key="long_context")
    if want("mixed_attn"):
        res["mixed_attn"] = attn_figures(pcp, torch, W.mixed_batch(), dev, peaks, flush, err,
                                         key="mixed")
    if want("gqa_prefill_ps1"):
        res["gqa_prefill_ps1"] = attn_figures(pcp, torch, W.gqa_prefill(page_size=1), dev,
                                              peaks, flush, err, n=10, warm=3)
    for name in ("stress_ps1_w4096", "stress_ps1_w0", "stress_ps16_w4096", "stress_ps16_w0"):
        if want(name):
            res[name] = attn_figures(pcp, torch, W.config_by_name(name), dev, peaks, flush,
                                     err, n=10, warm=3)

    # non-causal attention and a 2-D key mask (keep 1/2) on the GQA workload
    if want("masked"):
        res.update(masked_secondary(pcp, torch, W, dev, peaks, flush, err))

    if want("chunk_planner"):
        res["chunk_planner"] = planner_secondary(pcp)
    if want("cow_page_copy"):
        res["cow_page_copy"] = cow_secondary(pcp, torch, dev, peaks, flush)
    if pcp.read_error(err) != 0:
        raise RuntimeError("device error in secondary measurements")
    return res


def planner_secondary(pcp, n_decode=240, n_prompt=16, steps=200):
    """Host time of one planned step (pcp_schedule_step through the binding)
    in a serving loop of n_decode decoding requests and n_prompt incoming
    2000-token prompts, token budget 8192, page size 16."""
    rng = np.random.default_rng(11)
    pg = pcp.Pager(200_000, 16)
    # the loop's state lives in int arrays, as a serving loop keeps it
    ids = np.arange(n_decode + n_prompt, dtype=np.int64)
    total = np.concatenate([rng.integers(100, 4000, size=n_decode),
                            np.full(n_prompt, 2000)]).astype(np.int32)
    comp = np.concatenate([total[:n_decode] - 1, np.zeros(n_prompt, np.int32)]).astype(np.int32)
    # the decoding requests already hold their pages
    pg.schedule_step(ids[:n_decode], total[:n_decode], np.zeros(n_decode, np.int32), 1 << 30)
    times = []
    for _ in range(steps):
        t0 = time.perf_counter()
        st = pg.schedule_step(ids, total, comp, 8192)
        times.append(time.perf_counter() - t0)
        rows = st["row_req"]
        comp[rows] += np.diff(st["qo_indptr"]).astype(np.int32)
        total[rows[st["sample"]]] += 1
    return {"workload": f"{n_decode} decoding + {n_prompt} prefilling requests, budget 8192, "
                        f"page size 16", "us_per_step": float(np.median(times) * 1e6),
            "what": "host time of pcp_schedule_step through the Python binding (median)"}


def cow_secondary(pcp, torch, dev, peaks, flush, n_copies=2048, page_size=16, hkv=8, d=128):
    """pcp_copy_page_slots on 2048 whole pages (K and V) of a pool of 8192."""
    num_pages = 4 * n_copies
    g = torch.Generator(device=dev)
    g.manual_seed(3)
    kp = torch.randn(num_pages * page_size, hkv, d, device=dev, generator=g).to(torch.bfloat16)
    vp = torch.randn(num_pages * page_size, hkv, d, device=dev, generator=g).to(torch.bfloat16)
    perm = torch.randperm(num_pages, device=dev, generator=g).to(torch.int32)
    src, dst = perm[:n_copies].contiguous(), perm[n_copies:2 * n_copies].contiguous()
    nsl = torch.full((n_copies,), page_size, dtype=torch.int32, device=dev)
    ms = time_calls(torch, lambda ev: pcp.copy_page_slots(kp, vp, page_size, src, dst, nsl,
                                                           check=False), flush)
    nbytes = 2 * 2 * n_copies * page_size * hkv * d * 2
    gbs = nbytes / (ms * 1e-3) / 1e9
    return {"workload": f"{n_copies} whole pages of {page_size} slots x {hkv} KV heads x D {d}",
            "ms": ms, "GB/s": gbs, "frac_hbm": gbs / peaks["hbm_gbs"], "bytes": nbytes}


def masked_secondary(pcp, torch, W, dev, peaks, flush, err):
    """Non-causal and 2-D-masked calls on the GQA chunked-prefill workload;
    effective FLOPs count the visible pairs only."""
    gb = W.gqa_prefill()
    mask_np = W.random_mask(gb, "2d", seed=5, keep=0.5)
    P = gb.prefix_lens.astype(np.int64)
    C = gb.chunk_lens
    keep = np.cumsum(mask_np, axis=1)   # kept keys among 0..j
    masked_pairs = 0
    for b in range(gb.batch):
        masked_pairs += int(keep[b, P[b] + np.arange(C[b])].sum())
    nc = attn_figures(pcp, torch, gb, dev, peaks, flush, err, n=10, warm=3, causal=False,
                      pairs=int((C * (P + C)).sum()))
    nc["workload"] += ", non-causal"
    mk = attn_figures(pcp, torch, gb, dev, peaks, flush, err, n=10, warm=3, mask=mask_np,
                      pairs=masked_pairs,
                      computed_pairs=visible_pairs(gb.prefix_lens, gb.chunk_lens, 0))
    mk["workload"] += ", causal + 2-D key mask keeping 1/2"
    return {"non_causal_attn": nc, "masked_2d_attn": mk}


def time_calls(torch, fn, flush, n=20, warm=5, events=False):
    """Median ms of fn(ev) between CUDA events, L2 flushed before each call.
    With events=False the events bracket the whole call (fn gets None); with
    events=True fn gets the (before, after) pair to hand to the library, which
    records it around one kernel."""
    stream = torch.cuda.current_stream()
    for _ in range(warm):
        flush()
        fn(None)
    torch.cuda.synchronize()
    ms = []
    for _ in range(n):
        flush()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        if not events:
            a.record(stream)
            fn(None)
            b.record(stream)
        else:
            a.record(stream)  # creates the events before the library records them
            b.record(stream)
            fn((a, b))
        b.synchronize()
        ms.append(a.elapsed_time(b))
    return float(np.median(ms))


if __name__ == "__main__":
    main()
