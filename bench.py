#!/usr/bin/env python
"""Benchmark of the block-sparse (Splash) masked attention forward hot path.

One step = one pass of the whole hot path on one batch of seeded synthetic
input: the MaskInfo build (classification, compaction, pattern dedup) into a
reused handle, then the attention forward.  The default workload is the
dense-causal GQA configuration (B=2, Hq=32, Hkv=8, L=4096, d=128, 128x128
blocks).  Inputs are resident in HBM when the timed region starts; L2 is
flushed (a 256 MiB write) between timed steps, outside the timed events.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

With N > 1 (launched by torch.distributed.run) every rank runs the same
workload on its own GPU (independent replicas, weak scaling); the timing is
the max over ranks.  `--impl reference` times the CPU oracle (the plain f64
implementation) on the host cores, on bounded samples of the same workload.
Prints one JSON line on rank 0.
"""
import argparse
import dataclasses
import json
import math
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "masked attn fwd useful TFLOP/s & % of GB300 BF16 tensor peak; ms per call"
L2_FLUSH_BYTES = 256 << 20


def parse_args(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=1000)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", type=int, default=2)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-per-workload", action="store_true",
                    help="skip the sparse workloads timed beside the headline one")
    ap.add_argument("--sustain-s", type=float, default=2.0,
                    help="seconds of back-to-back attention calls for the clock-normalised figures (0: skip)")
    ap.add_argument("--shard", choices=["replicas", "heads"], default="replicas",
                    help="N > 1: every rank runs the whole workload (replicas, weak scaling) or its own range "
                         "of (batch, KV head) groups of one workload (heads, strong scaling)")
    ap.add_argument("--gather", action="store_true",
                    help="with --shard heads: gather every rank's O / LSE slice to rank 0 after timing and "
                         "check that they tile the whole output")
    ap.add_argument("--splits", type=int, default=1,
                    help="split-KV forward with this many splits per row, then the LSE merge")
    ap.add_argument("--backward", action="store_true",
                    help="time the backward pass (MaskInfo rebuild + gradients) instead of the forward")
    ap.add_argument("--pattern-source", choices=["stored", "positions"], default="stored",
                    help="partial-block masks from the stored patterns or computed from positions")
    ap.add_argument("--bq", type=int, default=None,
                    help="override the workload's query block (e.g. 256: two 128-row tiles of one head "
                         "share each K / V tile)")
    ap.add_argument("--max-logit", type=float, default=None,
                    help="Max Logit Estimate: fix every row's softmax reference at this constant "
                         "(e.g. the workload's soft cap)")
    return ap.parse_args(argv)


def bench_workload(args):
    import dataclasses
    import workloads
    w = workloads.workload(args.workload)
    return dataclasses.replace(w, bq=args.bq) if args.bq else w


# --------------------------------------------------------------------- accounting
def flop_counts(w, counts, batch_rows):
    """Useful FLOPs (unmasked (q, k) pairs only) and executed FLOPs (every
    element of every active block) of one forward pass."""
    per_pair = 2 * (w.dqk + w.dv)
    rep = w.Hq * (w.B if batch_rows == 1 else 1)
    useful = per_pair * counts["allowed_pairs"] * rep
    executed = per_pair * w.bq * w.bk * counts["num_active"] * rep
    return float(useful), float(executed)


def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            d = json.load(f)
        return d, "measured"
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}, "fallback"


def kernel_source_sha():
    """sha256 prefix of the attention kernel's sources (kernel + PTX header)."""
    import hashlib
    h = hashlib.sha256()
    for name in ("attention_fwd.cu", "sm103_ptx.cuh"):
        with open(os.path.join(ROOT, "block_sparse_flash_gb300", "csrc", name), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def recorded_traffic(workload_index):
    """DRAM bytes per attention launch from the committed ncu summary, or None
    when the kernel source has changed since those counters were taken."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(path):
        return None
    with open(path) as f:
        rec = json.load(f).get(f"workload{workload_index}")
    if not rec:
        return None
    return rec.get("bytes_per_launch") if kernel_source_sha() == rec.get("kernel_sha256_prefix") else None


def percentiles(xs, qs=(10, 50, 90)):
    """Nearest-rank percentiles of a list of times."""
    ys = sorted(xs)
    return [ys[min(len(ys) - 1, max(0, int(math.ceil(q / 100 * len(ys))) - 1))] for q in qs]


def mask_info_rate(w, counts, shape, build_ms, peaks):
    """The MaskInfo build against HBM: algorithmic bytes = segment IDs read
    (4 (Lq + Lk) per table batch row, with segment IDs), block_mask (1 byte
    per block), row_ptr (4 (R + 1)), the active lists (3 int32 + 2 flag bytes
    per active block) and the bit-packed patterns (bq*bk/8 bytes each)
    written; divided by the median build time."""
    R = shape["batch_rows"] * shape["nq"]
    nk = shape["nk"]
    seg = 4 * (w.q_len + w.L) * shape["batch_rows"] if w.documents else 0
    P = counts["num_patterns"]
    nbytes = seg + R * nk + 4 * (R + 1) + counts["num_active"] * (3 * 4 + 2) + P * w.bq * w.bk // 8
    med = percentiles(build_ms)[1]
    hbm = float(peaks.get("hbm_gbs", 6800.0))
    gbs = nbytes / (med * 1e-3) / 1e9
    return {"ms_p50": round(med, 5), "bytes": int(nbytes), "gbs": round(gbs, 2), "hbm_peak_gbs": hbm,
            "frac_of_hbm": round(gbs / hbm, 5),
            "note": "launch- and latency-bound at these sizes: the table is KB to a few MB"}


def reduce_max(value, world, device=None):
    """Max of a float over ranks (identity for one rank)."""
    if world <= 1:
        return float(value)
    import torch
    import torch.distributed as dist
    t = torch.tensor([float(value)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def whole_job_throughput(flop_per_step_per_rank, world, ms_per_step_max):
    """Aggregate over ranks: every rank processes its own copy of the workload."""
    return world * flop_per_step_per_rank / (ms_per_step_max * 1e-3) / 1e12


def sum_over_ranks(value, world, device=None):
    """Sum of a float over ranks (identity for one rank)."""
    if world <= 1:
        return float(value)
    import torch
    import torch.distributed as dist
    t = torch.tensor([float(value)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.SUM)
    return float(t.item())


def gather_shards(pieces, B, Hq, Hkv, Lq, dv):
    """Assembles the ranks' (begin, end, out, lse) slices of (batch, KV head)
    groups into out [B, Hq, Lq, dv] and lse [B, Hq, Lq] (host tensors), and a
    coverage count per (batch, query head) that must be 1 everywhere."""
    import torch
    G = Hq // Hkv
    out = torch.zeros((B, Hq, Lq, dv), dtype=pieces[0][2].dtype)
    lse = torch.zeros((B, Hq, Lq), dtype=torch.float32)
    cover = torch.zeros((B * Hkv, G), dtype=torch.int32)
    for b0, b1, o, l in pieces:
        out.view(B * Hkv, G, Lq, dv)[b0:b1] = o.reshape(b1 - b0, G, Lq, dv)
        lse.view(B * Hkv, G, Lq)[b0:b1] = l.reshape(b1 - b0, G, Lq)
        cover[b0:b1] += 1
    return out, lse, cover.view(B, Hq)


# --------------------------------------------------------------------- clocks
class ClockSampler:
    """Samples SM clocks and throttle reasons with nvidia-smi while running."""
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index):
        self.device_index = device_index
        self.proc = None
        self.path = None

    def start(self):
        try:
            fd, self.path = tempfile.mkstemp(prefix="clocks", suffix=".csv")
            os.close(fd)
            self.fh = open(self.path, "w")
            self.proc = subprocess.Popen(["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                                          "-i", str(self.device_index), "-lms", "50"], stdout=self.fh,
                                         stderr=subprocess.DEVNULL)
            # the timed region starts only once sampling runs (nvidia-smi takes
            # a few hundred ms to start; a short region would otherwise see at
            # most the sample taken after it)
            t0 = time.time()
            while time.time() - t0 < 3.0 and self.proc.poll() is None and os.path.getsize(self.path) == 0:
                time.sleep(0.01)
        except Exception:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unavailable"], "samples": 0}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        self.fh.close()
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        with open(self.path) as f:
            for line in f:
                parts = [p.strip() for p in line.split(",")]
                if len(parts) < 9:
                    continue
                try:
                    sm.append(float(parts[1]))
                    smax.append(float(parts[2]))
                except ValueError:
                    continue
                for name, val in zip(names, parts[5:9]):
                    if val.lower().startswith("active"):
                        reasons.add(name)
        os.unlink(self.path)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(smax) if smax else None,
                "reasons": sorted(reasons), "samples": len(sm)}


# --------------------------------------------------------------------- CPU oracle timing
def oracle_sample_rate(w, inp, nrows, seed, nthreads=0):
    """Times the oracle on `nrows` seeded random query rows of the workload;
    returns (useful FLOP of those rows, seconds, threads)."""
    import numpy as np
    import oracle
    rng = np.random.default_rng(seed)
    nq_rows = w.B * w.Hq * w.q_len
    rows = np.sort(rng.choice(nq_rows, size=min(nrows, nq_rows), replace=False))
    seg = inp.segment_ids.numpy() if inp.segment_ids is not None else None
    spec = oracle.MaskSpec(w.causal, w.window_left, w.window_right, seg, seg)
    nth = nthreads or oracle.default_threads()
    t0 = time.perf_counter()
    oracle.attention(inp.q, inp.k, inp.v, spec, w.scale, w.softcap, rows=rows, nthreads=nth)
    dt = time.perf_counter() - t0
    # allowed keys of each sampled row, counted from the mask definition: the
    # band [lo, hi] of the causal / window part, intersected with the row's
    # document when segment IDs are given (contiguous documents)
    i = (rows % w.q_len).astype(np.int64)
    b = (rows // (w.Hq * w.q_len)).astype(np.int64)
    lo = np.maximum(0, i - w.window_left) if w.window_left >= 0 else np.zeros_like(i)
    hi = i.copy() if w.causal else np.full_like(i, w.L - 1)
    if w.window_right >= 0:
        hi = np.minimum(hi, i + w.window_right)
    if seg is not None:
        starts = np.zeros_like(seg, dtype=np.int64)
        ends = np.zeros_like(seg, dtype=np.int64)
        for r in range(seg.shape[0]):
            change = np.flatnonzero(np.diff(seg[r]) != 0) + 1
            bounds = np.concatenate([[0], change, [seg.shape[1]]])
            doc = np.repeat(np.arange(len(bounds) - 1), np.diff(bounds))
            starts[r] = bounds[doc]
            ends[r] = bounds[doc + 1] - 1
        lo = np.maximum(lo, starts[b, i])
        hi = np.minimum(hi, ends[b, i])
    allowed = np.maximum(hi - lo + 1, 0)
    return 2.0 * (w.dqk + w.dv) * float(allowed.sum()), dt, nth, len(rows)


def cpu_baseline(w, inp, target_s=12.0):
    flop, dt, nth, n = oracle_sample_rate(w, inp, 256, 7)
    rate = n / max(dt, 1e-6)
    nrows = int(min(w.B * w.Hq * w.q_len, max(256, rate * target_s)))
    flop, dt, nth, n = oracle_sample_rate(w, inp, nrows, 8)
    return {"value": flop / dt / 1e12, "unit": "TFLOP/s", "cores": nth, "kind": "oracle",
            "sample": f"{n} seeded random query rows of the workload (all heads/batches), f64 oracle, "
                      f"{dt:.1f} s wall; useful FLOPs of those rows / time"}



# --------------------------------------------------------------------- sparse workloads and sustained load
# bf16 dense FLOPs one SM's tensor unit retires per clock: a 128x128x16 MMA
# (65,536 FLOPs) executes in 64 cycles when the pipe is kept full (single-CTA
# clock64 microbenchmark on this GPU).
TENSOR_FLOP_PER_CLK_PER_SM = 2 * 128 * 128 * 16 / 64


def tile_units(w, counts, batch_rows):
    """Active (batch, query head, 128x128 tile) units of one forward pass."""
    rep = w.Hq * (w.B if batch_rows == 1 else 1)
    return counts["num_active"] * rep * (w.bq // 128 if w.bq >= 128 else 1) * (w.bk // 128 if w.bk >= 128 else 1)


def time_forward_steps(bsf, w, inp, dev, K, warmup, flush):
    """The headline step (MaskInfo rebuild + attention) on workload w, timed
    like the headline: L2 flushed between steps outside the events.  Returns
    (attention ms list, build ms list, counts, batch_rows)."""
    import torch
    q, k, v = inp.q.to(dev), inp.k.to(dev), inp.v.to(dev)
    seg = inp.segment_ids.to(dev) if inp.segment_ids is not None else None
    spec = bsf.MaskSpec(w.causal, w.window_left, w.window_right, seg, seg)
    mi = bsf.build_mask_info(spec, w.q_len, w.L, w.bq, w.bk)
    counts, batch_rows = mi.counts(), mi.shape()["batch_rows"]
    out = torch.empty((w.B, w.Hq, w.q_len, w.dv), dtype=torch.bfloat16, device=dev)
    lse = torch.empty((w.B, w.Hq, w.q_len), dtype=torch.float32, device=dev)
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(K)]
    for i in range(warmup + K):
        flush.zero_()
        e = ev[i - warmup] if i >= warmup else None
        if e:
            e[0].record()
        mi.rebuild(spec, w.q_len, w.L, w.bq, w.bk)
        if e:
            e[1].record()
        bsf.attention_fwd(q, k, v, mi, w.scale, w.softcap, seg, seg, out=out, lse=lse)
        if e:
            e[2].record()
    torch.cuda.synchronize()
    bsf.check_device_error()
    mi.close()
    attn = [e[1].elapsed_time(e[2]) for e in ev]
    build = [e[0].elapsed_time(e[1]) for e in ev]
    return attn, build, counts, batch_rows


def per_workload(bsf, dev, K, warmup, flush, peak, indices=(3, 4, 5)):
    """Attention time against active tile units on the sparse and wide-head
    workloads, to show time proportional to the active blocks."""
    import workloads
    res = {}
    for idx in indices:
        w = workloads.workload(idx)
        inp = workloads.make_inputs(w)
        attn, build, counts, batch_rows = time_forward_steps(bsf, w, inp, dev, K, warmup, flush)
        useful, executed = flop_counts(w, counts, batch_rows)
        units = tile_units(w, counts, batch_rows)
        p50 = percentiles(attn)[1]
        res[f"workload{idx}"] = {
            "workload": w.describe(), "attention_ms_p50": round(p50, 5),
            "mask_build_ms_p50": round(percentiles(build)[1], 5),
            "active_blocks": counts["num_active"], "active_tile_units": int(units),
            "ns_per_unit": round(p50 * 1e6 / units, 3),
            "ns_per_unit_d128_equiv": round(p50 * 1e6 / (executed / (2 * 128 * 128 * 256)), 3),
            "executed_frac_of_burst": round(executed / (p50 * 1e-3) / 1e12 / peak, 4),
            "useful_frac_of_burst": round(useful / (p50 * 1e-3) / 1e12 / peak, 4)}
        del inp
    return res


def sustained_figures(bsf, w, q, k, v, mi, out, lse, dev, seconds, peaks, local, seg=None):
    """Back-to-back attention calls for `seconds` (no flush, no rebuild) with
    the clock sampler running: executed TFLOP/s against the sustained cuBLAS
    peak, the median SM clock of the samples, and the tensor fraction at that
    clock (executed FLOPs / (time x clock x FLOP per clock per SM x SMs))."""
    import torch
    counts = mi.counts()
    _, executed = flop_counts(w, counts, mi.shape()["batch_rows"])
    sms = torch.cuda.get_device_properties(dev).multi_processor_count
    # calls per chunk from one timed call
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record()
    bsf.attention_fwd(q, k, v, mi, w.scale, w.softcap, seg, seg, out=out, lse=lse)
    b.record()
    torch.cuda.synchronize()
    per_chunk = max(1, int(50.0 / max(a.elapsed_time(b), 1e-3)))  # ~50 ms chunks
    clocks = ClockSampler(local)
    clocks.start()
    chunks, calls, total_ms = [], 0, 0.0
    t0 = time.time()
    while time.time() - t0 < seconds:
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record()
        for _ in range(per_chunk):
            bsf.attention_fwd(q, k, v, mi, w.scale, w.softcap, seg, seg, out=out, lse=lse)
        b.record()
        chunks.append((a, b))
        calls += per_chunk
        b.synchronize()
    torch.cuda.synchronize()
    clk = clocks.stop()
    bsf.check_device_error()
    total_ms = sum(x.elapsed_time(y) for x, y in chunks)
    tflops = executed * calls / (total_ms * 1e-3) / 1e12
    res = {"seconds": round(total_ms * 1e-3, 3), "calls": calls, "ms_per_call": round(total_ms / calls, 5),
           "executed_tflops": round(tflops, 2),
           "peak_sustained": float(peaks.get("bf16_tflops_sustained", 1700.0)),
           "frac_of_sustained": round(tflops / float(peaks.get("bf16_tflops_sustained", 1700.0)), 4),
           "clocks": clk}
    if clk.get("sm_mhz"):
        clock_peak = clk["sm_mhz"] * 1e6 * TENSOR_FLOP_PER_CLK_PER_SM * sms / 1e12
        res["tensor_peak_at_median_clock_tflops"] = round(clock_peak, 1)
        res["clock_normalised_tensor_frac"] = round(tflops / clock_peak, 4)
        res["clock_normalised_note"] = (f"{TENSOR_FLOP_PER_CLK_PER_SM:.0f} bf16 FLOP per clock per SM x {sms} SMs "
                                        "x median SM clock of the samples")
    return res

# --------------------------------------------------------------------- our arm
def run_ours(args):
    import torch
    import torch.distributed as dist

    import block_sparse_flash_gb300 as bsf
    from block_sparse_flash_gb300 import build as libbuild
    import workloads

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        dist.init_process_group("nccl")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if rank == 0 or world == 1:
        libbuild.build()
    if world > 1:
        dist.barrier()
    bsf.lib()

    w_full = bench_workload(args)
    inp_full = workloads.make_inputs(w_full)
    w, inp, shard = w_full, inp_full, None
    if args.shard == "heads":
        # this rank's (batch, KV head) groups of the one workload, as a problem
        # of (end - begin) batch rows with Hq / Hkv query heads and one KV head
        if world > w_full.B * w_full.Hkv:
            raise SystemExit("--shard heads needs at least one (batch, KV head) group per rank")
        shard = bsf.shard_items(w_full.B, w_full.Hkv, world, rank)
        sv = bsf.shard_views(inp_full.q, inp_full.k, inp_full.v, shard[0], shard[1],
                             segment_ids=inp_full.segment_ids)
        w = dataclasses.replace(w_full, B=shard[1] - shard[0], Hq=w_full.Hq // w_full.Hkv, Hkv=1)
        inp = workloads.Inputs(sv["q"].contiguous(), sv["k"].contiguous(), sv["v"].contiguous(),
                               sv.get("segment_ids"))
    q, k, v = inp.q.to(dev), inp.k.to(dev), inp.v.to(dev)
    seg = inp.segment_ids.to(dev) if inp.segment_ids is not None else None
    spec = bsf.MaskSpec(w.causal, w.window_left, w.window_right, seg, seg)
    mi = bsf.build_mask_info(spec, w.q_len, w.L, w.bq, w.bk)
    if args.pattern_source != "stored":
        mi.set_pattern_source(args.pattern_source)
    counts = mi.counts()
    batch_rows = mi.shape()["batch_rows"]
    useful, executed = flop_counts(w, counts, batch_rows)
    # FLOPs of one step of the whole job: every rank's own copy (replicas), or
    # the sum of the ranks' shares of one workload (heads)
    job_useful = sum_over_ranks(useful, world, dev) if shard else world * useful
    out = torch.empty((w.B, w.Hq, w.q_len, w.dv), dtype=torch.bfloat16, device=dev)
    lse = torch.empty((w.B, w.Hq, w.q_len), dtype=torch.float32, device=dev)
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)

    S = args.splits
    if S > 1 and args.max_logit is not None:
        raise SystemExit("--max-logit applies to the one-pass forward only")
    if S > 1:
        o_part = torch.empty((S, w.B, w.Hq, w.q_len, w.dv), dtype=torch.float32, device=dev)
        lse_part = torch.empty((S, w.B, w.Hq, w.q_len), dtype=torch.float32, device=dev)

    def step(attn_events=None, merge_events=None):
        mi.rebuild(spec, w.q_len, w.L, w.bq, w.bk)
        if attn_events:
            attn_events[0].record()
        if S > 1:
            bsf.attention_fwd_split(q, k, v, mi, w.scale, w.softcap, S, seg, seg, o_part=o_part, lse_part=lse_part)
            if merge_events:
                merge_events[0].record()
            bsf.attention_merge(o_part, lse_part, out=out, lse=lse)
            if merge_events:
                merge_events[1].record()
        else:
            bsf.attention_fwd(q, k, v, mi, w.scale, w.softcap, seg, seg, out=out, lse=lse,
                              max_logit=args.max_logit)
        if attn_events:
            attn_events[1].record()

    for _ in range(args.warmup):
        flush.zero_()
        step()
    torch.cuda.synchronize()
    bsf.check_device_error()

    K = args.steps
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(K)]
    ea = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(K)]
    em = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(K)]
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    clocks = ClockSampler(local)
    clocks.start()
    launches0 = bsf.kernel_launches()
    for i in range(K):
        flush.zero_()
        ev[i][0].record()
        step(ea[i], em[i] if S > 1 else None)
        ev[i][1].record()
    torch.cuda.synchronize()
    launches = bsf.kernel_launches() - launches0
    if world > 1:
        dist.barrier()
    clk = clocks.stop()
    bsf.check_device_error()
    step_ms = [a.elapsed_time(b) for a, b in ev]
    attn_ms = [a.elapsed_time(b) for a, b in ea]
    build_ms = [a[0].elapsed_time(b[0]) for a, b in zip(ev, ea)]  # step start -> attention start
    ms_step = reduce_max(statistics.mean(step_ms), world, dev)
    ms_attn = reduce_max(statistics.mean(attn_ms), world, dev)
    value = job_useful / (ms_step * 1e-3) / 1e12

    peaks, peak_src = measured_peaks()
    peak = float(peaks["bf16_tflops"])
    ms_merge = reduce_max(statistics.mean([a.elapsed_time(b) for a, b in em]), world, dev) if S > 1 else 0.0
    achieved = executed / ((ms_attn - ms_merge) * 1e-3) / 1e12
    roofline = {"bound": "tensor", "achieved": round(achieved, 2), "peak": peak, "unit": "TFLOP/s",
                "frac": round(achieved / peak, 4), "traffic": None,
                "kernel": "splash_fwd_kernel", "peak_source": f"{peak_src} bf16 burst (cuBLAS)",
                "achieved_is": "executed FLOPs of the active blocks per launch / mean launch time (CUDA events)"}
    roofline["traffic"] = recorded_traffic(args.workload) if args.bq is None else None

    e2e = None
    if not args.no_e2e:
        e2e = run_e2e(bsf, w, inp, spec, mi, dev, K=max(3, min(K, 20)), world=world, job_useful=job_useful,
                      max_logit=args.max_logit)

    result = {
        "metric": METRIC, "value": round(value, 3), "unit": "TFLOP/s", "n_gpus": world, "steps": K,
        "warmup": args.warmup, "ms_per_step": round(ms_step, 5), "higher_is_better": True,
        "scaling": "strong" if shard else "weak",
        "vs_baseline": None, "dtype": "bf16", "data": "synthetic (seeded N(0,1) bf16, see workloads/)",
        "config": {"workload": w_full.describe(), "step": "MaskInfo rebuild + attention forward",
                   "l2": "flushed between timed steps (256 MiB write, outside the timed events)",
                   "active_blocks": counts["num_active"], "partial_blocks": counts["num_partial"],
                   "patterns": counts["num_patterns"],
                   "parallelism": (f"(batch, KV head) groups split over {world} ranks" if shard
                                   else f"replicas x{world}")},
        "attention_ms": round(ms_attn, 5),
        "mask_build_ms": round(ms_step - ms_attn, 5),
        "attention_ms_p10_p50_p90": [round(x, 5) for x in percentiles(attn_ms)],
        "mask_info": mask_info_rate(w, counts, mi.shape(), build_ms, peaks),
        "attention_useful_tflops": round(useful / (ms_attn * 1e-3) / 1e12, 2),
        "attention_executed_tflops": round(achieved, 2),
        "pct_of_bf16_peak_useful": round(100 * useful / (ms_attn * 1e-3) / 1e12 / peak, 2),
        "pct_of_bf16_peak_executed": round(100 * achieved / peak, 2),
        "roofline": roofline,
        "gpu_launches": int(launches),
        "clocks": clk,
    }
    if S > 1:
        rows = w.B * w.Hq * w.q_len
        mbytes = S * rows * (4 * w.dv + 4) + rows * (2 * w.dv + 4)
        gbs = mbytes / (ms_merge * 1e-3) / 1e9
        hbm = float(peaks.get("hbm_gbs", 6800.0))
        result["split_kv"] = {
            "splits": S, "split_kernel_ms": round(ms_attn - ms_merge, 5), "merge_ms": round(ms_merge, 5),
            "merge_roofline": {"bound": "hbm", "achieved": round(gbs, 1), "peak": hbm, "unit": "GB/s",
                               "frac": round(gbs / hbm, 4), "bytes": int(mbytes)},
            "note": "attention_ms = split kernel + merge; roofline.achieved uses the split kernel alone"}
    if args.max_logit is not None:
        result["config"]["max_logit"] = args.max_logit
    if args.pattern_source != "stored":
        result["config"]["pattern_source"] = args.pattern_source
    if e2e:
        result["e2e"] = e2e
    if world == 1 and S == 1 and args.max_logit is None and args.sustain_s > 0:
        result["sustained"] = sustained_figures(bsf, w, q, k, v, mi, out, lse, dev, args.sustain_s, peaks, local,
                                                seg)
    if world == 1 and not shard and args.workload == 2 and S == 1 and args.bq is None \
            and args.max_logit is None and args.pattern_source == "stored" and not args.no_per_workload:
        pw = per_workload(bsf, dev, K, args.warmup, flush, peak)
        pw["workload2"] = {
            "workload": w.describe(), "attention_ms_p50": round(percentiles(attn_ms)[1], 5),
            "mask_build_ms_p50": round(percentiles(build_ms)[1], 5), "active_blocks": counts["num_active"],
            "active_tile_units": int(tile_units(w, counts, batch_rows)),
            "ns_per_unit": round(percentiles(attn_ms)[1] * 1e6 / tile_units(w, counts, batch_rows), 3),
            "ns_per_unit_d128_equiv": round(percentiles(attn_ms)[1] * 1e6 / (executed / (2 * 128 * 128 * 256)), 3),
            "executed_frac_of_burst": round(executed / (percentiles(attn_ms)[1] * 1e-3) / 1e12 / peak, 4),
            "useful_frac_of_burst": round(useful / (percentiles(attn_ms)[1] * 1e-3) / 1e12 / peak, 4)}
        result["per_workload"] = dict(sorted(pw.items()))
        result["per_workload_note"] = ("same step, events and L2 flush as the headline; unit = one active "
                                       "(batch, query head, 128x128 tile); d128_equiv divides by the executed "
                                       "FLOPs of a d=128 tile (2*128*128*256)")
    if shard:
        result["config"]["rank0_groups"] = list(shard)
        if args.gather and world > 1:
            # host gather of every rank's slice (outside the timed region)
            pieces = [None] * world
            dist.all_gather_object(pieces, (shard[0], shard[1], out.cpu(), lse.cpu()))
            full_out, full_lse, cover = gather_shards(pieces, w_full.B, w_full.Hq, w_full.Hkv, w_full.q_len,
                                                      w_full.dv)
            result["gather"] = {"tiles_exactly": bool((cover == 1).all()),
                                "finite": bool(torch.isfinite(full_lse).all())}
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        result["cpu_baseline"] = cpu_baseline(w_full, inp_full)
    if rank == 0:
        print(json.dumps(result), flush=True)
    mi.close()
    if world > 1:
        dist.destroy_process_group()


def run_e2e(bsf, w, inp, spec, mi, dev, K, world, job_useful, max_logit=None):
    """Same metric through the public API with host buffers: pinned host ->
    device copies of the inputs, the step, device -> host copies of O and LSE,
    all inside the timed region (splash_attention_fwd_host, which pipelines
    the copies with the attention in chunks)."""
    import torch
    qh, kh, vh = inp.q.pin_memory(), inp.k.pin_memory(), inp.v.pin_memory()
    segh = inp.segment_ids.pin_memory() if inp.segment_ids is not None else None
    q = torch.empty_like(qh, device=dev)
    k = torch.empty_like(kh, device=dev)
    v = torch.empty_like(vh, device=dev)
    seg = spec.q_segment_ids
    out = torch.empty((w.B, w.Hq, w.q_len, w.dv), dtype=torch.bfloat16, device=dev)
    lse = torch.empty((w.B, w.Hq, w.q_len), dtype=torch.float32, device=dev)
    outh = torch.empty(out.shape, dtype=out.dtype).pin_memory()
    lseh = torch.empty(lse.shape, dtype=lse.dtype).pin_memory()
    h2d = qh.numel() * 2 + kh.numel() * 2 + vh.numel() * 2 + (segh.numel() * 4 if segh is not None else 0)
    d2h = outh.numel() * 2 + lseh.numel() * 4
    times = []
    for i in range(K + 2):
        torch.cuda.synchronize()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record()
        if segh is not None:
            seg.copy_(segh, non_blocking=True)
        mi.rebuild(spec, w.q_len, w.L, w.bq, w.bk)
        if max_logit is None:
            # the library's host-buffer entry: copies and attention pipelined in chunks
            bsf.attention_fwd_host(qh, kh, vh, mi, w.scale, w.softcap, out_host=outh, lse_host=lseh,
                                   q=q, k=k, v=v, out=out, lse=lse, q_segment_ids=seg, kv_segment_ids=seg)
        else:
            q.copy_(qh, non_blocking=True)
            k.copy_(kh, non_blocking=True)
            v.copy_(vh, non_blocking=True)
            bsf.attention_fwd(q, k, v, mi, w.scale, w.softcap, seg, seg, out=out, lse=lse, max_logit=max_logit)
            outh.copy_(out, non_blocking=True)
            lseh.copy_(lse, non_blocking=True)
        b.record()
        torch.cuda.synchronize()
        if i >= 2:
            times.append(a.elapsed_time(b))
    ms = reduce_max(statistics.mean(times), world, dev)
    return {"value": round(job_useful / (ms * 1e-3) / 1e12, 3), "unit": "TFLOP/s",
            "ms_per_step": round(ms, 4), "h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": int(d2h)}


# --------------------------------------------------------------------- reference arm
def run_reference(args):
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    import workloads
    w = bench_workload(args)
    inp = workloads.make_inputs(w)
    # the rate from a sample large enough that thread start-up is small
    # against it; each step's sample is at least 512 rows for the same reason
    _, dt, nth, n = oracle_sample_rate(w, inp, 1024, 3)
    rate = n / max(dt, 1e-6)
    per_step = int(min(8192, max(512, rate * 90.0 / max(1, args.steps + args.warmup))))
    for i in range(args.warmup):
        oracle_sample_rate(w, inp, per_step, 100 + i)
    flops, secs = 0.0, 0.0
    for i in range(args.steps):
        f, dt, nth, n = oracle_sample_rate(w, inp, per_step, 1000 + i)
        flops += f
        secs += dt
    value = flops / secs / 1e12
    sample = (f"{per_step} seeded random query rows per step (all heads/batches) of the workload, f64 oracle "
              f"on {nth} host threads; useful FLOPs of the rows / wall time")
    res = {"impl": "reference", "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": world,
           "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * secs / max(1, args.steps),
           "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
           "data": "synthetic (seeded N(0,1) bf16, see workloads/)",
           "config": {"workload": w.describe(), "step": f"oracle on {per_step} sampled rows"},
           "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": nth, "kind": "oracle", "sample": sample},
           "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(res), flush=True)


# --------------------------------------------------------------------- backward
def bwd_flop_counts(w, counts, batch_rows):
    """Backward FLOPs: per (query, key) pair five products of the forward's
    size class: S, dP, dV, dK, dQ = 2 * (3 * dqk + 2 * dv)."""
    per_pair = 2 * (3 * w.dqk + 2 * w.dv)
    rep = w.Hq * (w.B if batch_rows == 1 else 1)
    return (float(per_pair * counts["allowed_pairs"] * rep),
            float(per_pair * w.bq * w.bk * counts["num_active"] * rep))


def run_backward(args):
    """One step = MaskInfo rebuild + the backward call (transposed table, D,
    main kernel, dq conversion) for the workload's forward outputs, which are
    computed once before timing; dout is seeded N(0, 1) bf16."""
    import torch

    import block_sparse_flash_gb300 as bsf
    from block_sparse_flash_gb300 import build as libbuild
    import workloads

    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    libbuild.build()
    w = bench_workload(args)
    inp = workloads.make_inputs(w)
    q, k, v = inp.q.to(dev), inp.k.to(dev), inp.v.to(dev)
    dout = workloads.normal_bf16((w.B, w.Hq, w.q_len, w.dv), 1000 * w.index + 5).to(dev)
    seg = inp.segment_ids.to(dev) if inp.segment_ids is not None else None
    spec = bsf.MaskSpec(w.causal, w.window_left, w.window_right, seg, seg)
    mi = bsf.build_mask_info(spec, w.q_len, w.L, w.bq, w.bk)
    counts = mi.counts()
    useful, executed = bwd_flop_counts(w, counts, mi.shape()["batch_rows"])
    out, lse = bsf.attention_fwd(q, k, v, mi, w.scale, w.softcap)
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    ws = torch.empty(bsf.attention_bwd_workspace_size(w.B, w.Hq, w.q_len, w.dqk), dtype=torch.uint8, device=dev)
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)

    def step(ev=None):
        mi.rebuild(spec, w.q_len, w.L, w.bq, w.bk)
        if ev:
            ev[0].record()
        bsf.attention_bwd(q, k, v, out, lse, dout, mi, w.scale, w.softcap, dq=dq, dk=dk, dv=dv, workspace=ws)
        if ev:
            ev[1].record()

    for _ in range(args.warmup):
        flush.zero_()
        step()
    torch.cuda.synchronize()
    bsf.check_device_error()
    K = args.steps
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(K)]
    eb = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(K)]
    torch.cuda.synchronize()
    clocks = ClockSampler(0)
    clocks.start()
    launches0 = bsf.kernel_launches()
    for i in range(K):
        flush.zero_()
        ev[i][0].record()
        step(eb[i])
        ev[i][1].record()
    torch.cuda.synchronize()
    launches = bsf.kernel_launches() - launches0
    clk = clocks.stop()
    bsf.check_device_error()
    ms_step = statistics.mean(a.elapsed_time(b) for a, b in ev)
    ms_bwd = statistics.mean(a.elapsed_time(b) for a, b in eb)
    peaks, peak_src = measured_peaks()
    peak = float(peaks["bf16_tflops"])
    achieved = executed / (ms_bwd * 1e-3) / 1e12
    result = {
        "metric": "masked attn bwd useful TFLOP/s & % of GB300 BF16 tensor peak; ms per call",
        "value": round(useful / (ms_step * 1e-3) / 1e12, 3), "unit": "TFLOP/s", "n_gpus": 1, "steps": K,
        "warmup": args.warmup, "ms_per_step": round(ms_step, 5), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16", "data": "synthetic (seeded N(0,1) bf16, see workloads/)",
        "config": {"workload": w.describe(), "step": "MaskInfo rebuild + attention backward",
                   "l2": "flushed between timed steps (256 MiB write, outside the timed events)",
                   "active_blocks": counts["num_active"], "parallelism": "replicas x1"},
        "backward_ms": round(ms_bwd, 5),
        "backward_useful_tflops": round(useful / (ms_bwd * 1e-3) / 1e12, 2),
        "backward_executed_tflops": round(achieved, 2),
        "roofline": {"bound": "tensor", "achieved": round(achieved, 2), "peak": peak, "unit": "TFLOP/s",
                     "frac": round(achieved / peak, 4), "traffic": None, "kernel": "whole backward call",
                     "peak_source": f"{peak_src} bf16 burst (cuBLAS)",
                     "achieved_is": "executed backward FLOPs of the active blocks / mean time of the whole "
                                    "backward call (its 7 kernels, CUDA events)"},
        "gpu_launches": int(launches), "clocks": clk,
    }
    print(json.dumps(result), flush=True)
    mi.close()


def main(argv=None):
    args = parse_args(argv)
    if args.impl == "reference":
        run_reference(args)
    elif args.backward:
        run_backward(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
