#!/usr/bin/env python3
"""Throughput of causal GQA prefill (TFLOP/s) and paged decode (KV-read GB/s)
on GB300, through the libgqa C ABI.

Default line (one JSON object on stdout, rank 0):
  * main metric -- bf16 ragged prefill: B=4, H_q=32, H_kv=8, d_h=128, padded
    n=2048, valid lengths ~U{512..2048} (seeded), right padded, N(0,1) inputs.
    One step = attn_prefill (host checks, then one launch: causal attention
    with the cache write fused and the padding rows zeroed) + kv_truncate of
    every sequence back to 0, so each step starts from an empty cache.  L2 is flushed (512 MiB write) before
    every timed step; only the step is inside the CUDA events.
  * "decode" -- bf16 paged decode: B=64, H_q=32, H_kv=8, d_h=128, cache
    lengths ~U{1024..8192} including the step's own entry, pages placed by a
    seeded random permutation.  One step = attn_decode_append (one token
    per sequence appended and attended in one call) + kv_truncate back.  The 1.2 GB of K/V is larger
    than L2, so no flush is needed.
  * "wide_gqa" -- B=1, H_q=48, H_kv=8, prefill T=8192 (TFLOP/s, roofline),
    then 256 attn_decode_append steps: kernel time L2-resident, per-step time
    with and without an L2 flush.
  * "prefix_reuse" -- a 4096-token prefix shared by 8 forks, each prefilling
    512 tokens over it; fork 0 edited at m=2000 (truncate + re-prefill).
  (--no-extra skips the last two.)  Each object carries a roofline for its
  dominant kernel and, on rank 0 at N=1, a bounded fp64-oracle sample.
  "clocks" comes from nvidia-smi samples taken while the headline step runs
  back to back for 0.6 s right after its event-timed region.
Work counts: prefill flops = 4 d_h H_q sum_b causal_pairs; decode bytes =
sum_b L_b * 2 * H_kv * d_h * 2 (each KV head read once).

Multi-GPU: replicas only (the workloads are independent per GPU); a barrier
and a max over ranks bracket the timed region; `value` sums all ranks.
`--impl reference` times the fp64 CPU oracle on a bounded sample instead.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import workloads  # noqa: E402

METRIC = "causal GQA prefill TFLOP/s; decode KV-read GB/s (1×GB300, % of roofline)"
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
KERNEL_SOURCES = {
    "prefill_tc": "causal_gqa_attention_02_gb300/csrc/k_prefill_tc.cu",
    "attn_simt": "causal_gqa_attention_02_gb300/csrc/k_simt.cu",
    "decode_split": "causal_gqa_attention_02_gb300/csrc/k_decode.cu",
    "decode_cluster": "causal_gqa_attention_02_gb300/csrc/k_decode_cluster.cu",
}


# ---------------------------------------------------------------------------
# helpers
# ---------------------------------------------------------------------------

def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            return json.load(f), "measured"
    return dict(FALLBACK_PEAKS), "fallback"


def source_sha(kernel):
    """Hash of the kernel's source file and the device headers it includes."""
    h = hashlib.sha256()
    for rel in (KERNEL_SOURCES[kernel], "causal_gqa_attention_02_gb300/csrc/kernels.cuh",
                "causal_gqa_attention_02_gb300/csrc/sm100.cuh"):
        p = os.path.join(ROOT, rel)
        if not os.path.exists(p):
            return None
        h.update(open(p, "rb").read())
    return h.hexdigest()


def traffic_for(workload, kernel, units_scale=1.0):
    """DRAM bytes per launch of `kernel` on `workload` from the committed ncu
    summary, if it was taken on the kernel's current source; else None."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(path):
        return None
    rec = json.load(open(path)).get(workload)
    if not rec or rec.get("kernel") != kernel or rec.get("sha256") != source_sha(kernel):
        return None
    return rec["dram_bytes_per_launch"] * units_scale


class Dist:
    """One process per GPU (RANK / LOCAL_RANK / WORLD_SIZE from the launcher);
    replicas only: the ranks share nothing but a barrier around the timed
    region and the max of their times.  `backend` is nccl on GPUs (gloo lets
    the same logic run on CPU processes)."""

    def __init__(self, backend="nccl"):
        self.world = int(os.environ.get("WORLD_SIZE", "1"))
        self.rank = int(os.environ.get("RANK", "0"))
        self.local = int(os.environ.get("LOCAL_RANK", "0"))
        self.backend = backend
        self.pg = None

    def setup(self, torch):
        if self.backend == "nccl":
            torch.cuda.set_device(self.local)
        if self.world > 1:
            import torch.distributed as dist
            dist.init_process_group(self.backend)
            self.pg = dist

    def barrier(self):
        if self.pg:
            self.pg.barrier()

    def max(self, torch, x):
        if not self.pg:
            return x
        t = torch.tensor([float(x)], device="cuda" if self.backend == "nccl" else "cpu")
        self.pg.all_reduce(t, op=self.pg.ReduceOp.MAX)
        return float(t.item())

    def done(self):
        if self.pg:
            self.pg.destroy_process_group()


class ClockSampler:
    """nvidia-smi samples (SM clock, max clock, throttle reasons) every 100 ms."""

    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")
    REASONS = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")

    def __init__(self, uuid=None):
        self.rows = []
        self.proc = None
        cmd = ["nvidia-smi", "--query-gpu=" + self.FIELDS, "--format=csv,noheader,nounits", "-lms", "100"]
        if uuid:
            cmd += ["-i", uuid]
        try:
            self.proc = subprocess.Popen(cmd, stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except (OSError, ValueError):
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()

    def _read(self):
        for line in self.proc.stdout:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) == 7:
                self.rows.append((time.time(), parts))

    def stop(self):
        if self.proc:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self, t0, t1):
        rows = [r for t, r in self.rows if t0 <= t <= t1]
        note = ("samples during a back-to-back run of the timed step (with its L2 flush) for %.2f s right after "
                "the event-timed region" % (t1 - t0))
        if len(rows) < 3:
            near = sorted(self.rows, key=lambda tr: min(abs(tr[0] - t0), abs(tr[0] - t1)))[:5]
            rows = [r for _, r in near]
            note = "timed region shorter than the sampling period: nearest samples"
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0, "note": "nvidia-smi unavailable"}

        def num(x):
            try:
                return float(x)
            except ValueError:
                return None
        sm = [num(r[0]) for r in rows if num(r[0]) is not None]
        mx = [num(r[1]) for r in rows if num(r[1]) is not None]
        reasons = sorted({name for r in rows for name, val in zip(self.REASONS, r[3:]) if val.strip() == "Active"})
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": reasons, "samples": len(rows), "note": note}


def device_uuid(torch):
    try:
        u = str(torch.cuda.get_device_properties(torch.cuda.current_device()).uuid)
        return u if u.startswith("GPU-") else "GPU-" + u
    except Exception:
        return None


def to_dev(torch, a, dt="bf16"):
    a = np.ascontiguousarray(a)
    if dt == "bf16":
        return torch.from_numpy(a.view(np.int16)).cuda().view(torch.bfloat16)
    return torch.from_numpy(a).cuda()


def pinned(torch, t):
    h = torch.empty(t.shape, dtype=t.dtype, pin_memory=True)
    h.copy_(t)
    return h


def timed_steps(torch, dist, step, K, flush=None):
    """Per-step CUDA events on the current stream; flush (untimed) between."""
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(K)]
    torch.cuda.synchronize()
    dist.barrier()
    t0 = time.time()
    for i in range(K):
        if flush is not None:
            flush.zero_()
        evs[i][0].record()
        step()
        evs[i][1].record()
    torch.cuda.synchronize()
    dist.barrier()
    t1 = time.time()
    ms = [a.elapsed_time(b) for a, b in evs]
    return ms, t0, t1


def sustain(torch, step, flush=None, seconds=0.6):
    """Run the timed step back to back (with its flush) for at least
    `seconds` of wall time, so that the clock sampler sees the GPU under this
    load; returns (t0, t1, steps, median ms per step from events)."""
    torch.cuda.synchronize()
    t0 = time.time()
    evs = []
    while time.time() - t0 < seconds:
        for _ in range(8):
            if flush is not None:
                flush.zero_()
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record()
            step()
            b.record()
            evs.append((a, b))
        evs[-1][1].synchronize()
    torch.cuda.synchronize()
    t1 = time.time()
    return t0, t1, len(evs), statistics.median(a.elapsed_time(b) for a, b in evs)


# ---------------------------------------------------------------------------
# workloads
# ---------------------------------------------------------------------------

def prefill_cpu_baseline(w, budget_s):
    """The fp64 oracle on the host cores, cycling over the workload's
    sequences until about budget_s seconds of CPU work are done."""
    import oracle
    import causal_gqa_attention_02_gb300 as gqa
    nth = oracle.default_threads()
    B, H_q, H_kv, d = w["B"], w["H_q"], w["H_kv"], w["d"]
    done_flops, used, calls = 0, 0.0, 0
    while used < budget_s:
        b = calls % B
        nb = int(w["valid_lengths"][b])
        cm = oracle.CacheModel(workloads.pages_for(nb), 1, workloads.pages_for(nb), H_kv, d, "bf16")
        s = cm.create()
        t0 = time.perf_counter()
        oracle.prefill(cm, [s], w["q"][b:b + 1], w["k"][b:b + 1], w["v"][b:b + 1], [nb], nthreads=nth)
        used += time.perf_counter() - t0
        done_flops += gqa.work.prefill_flops([0], [nb], H_q, d)
        calls += 1
    return {"value": done_flops / used / 1e12, "unit": "TFLOP/s", "cores": nth, "kind": "oracle",
            "sample": "fp64 oracle prefill of the workload's sequences (valid lengths %s, all %d query heads), "
                      "%d sequence calls cycling over them: %.1f GFLOP causal in %.1f s"
                      % (list(map(int, w["valid_lengths"])), H_q, calls, done_flops / 1e9, used)}


def bench_prefill(torch, gqa, dist, args, peaks, peak_src):
    w = workloads.ragged_prefill(workloads.seed_for(2))
    B, n, H_q, H_kv, d = w["B"], w["n"], w["H_q"], w["H_kv"], w["d"]
    nb = [int(x) for x in w["valid_lengths"]]
    flops = gqa.work.prefill_flops([0] * B, nb, H_q, d, args.window)
    pages = sum(workloads.pages_for(x) for x in nb) + 16
    cache = gqa.Cache(H_kv, d, pages, B, workloads.pages_for(n) + 1, dtype="bf16", rope=args.rope,
                      window=args.window, keys_post_position=0 if args.pre_position else 1)
    ids = [cache.seq_create() for _ in range(B)]
    q, k, v = to_dev(torch, w["q"]), to_dev(torch, w["k"]), to_dev(torch, w["v"])
    out = torch.empty_like(q)
    flush = torch.empty(512 << 20, dtype=torch.uint8, device="cuda")

    def step():
        gqa.attn_prefill(cache, ids, q, k, v, nb, out=out)
        for s in ids:
            gqa.kv_truncate(cache, s, 0)

    for _ in range(args.warmup):
        flush.zero_()
        step()
    torch.cuda.synchronize()
    cache.profile_read()
    ms, t0, t1 = timed_steps(torch, dist, step, args.steps, flush)
    region_launches = cache.profile_read()            # launch counts of the timed region
    total_ms = dist.max(torch, sum(ms))
    value = flops * args.steps * dist.world / (total_ms / 1e3) / 1e12
    median_ms = statistics.median(ms)
    # The same step back to back for 0.6 s, for the clock record.
    s0, s1, s_steps, s_med = sustain(torch, step, flush)
    cache.profile_read()
    # Per-kernel durations: a second timed region with each launch bracketed
    # by events on its stream (events between kernels keep them from
    # overlapping, so this region is timed separately from the step).
    cache.profile(True)
    timed_steps(torch, dist, step, args.steps, flush)
    cache.profile(False)
    prof = cache.profile_read()
    kernel = "prefill_tc" if prof["prefill_tc"][0] else "attn_simt"
    launches, kms = prof[kernel]
    avg_ms = kms / max(1, launches)
    achieved = flops / (avg_ms / 1e3) / 1e12
    peak = peaks["bf16_tflops"]
    roofline = {"bound": "tensor", "achieved": round(achieved, 2), "peak": peak, "unit": "TFLOP/s",
                "frac": round(achieved / peak, 4), "traffic": traffic_for("prefill", kernel), "kernel": kernel,
                "kernel_ms": round(avg_ms, 4), "algorithmic_flops_per_launch": flops,
                "peak_source": "%s bf16 dense (burst)" % peak_src}
    gpu_launches = sum(nl for nl, _ in region_launches.values())
    kernels = {name: {"launches": nl, "avg_ms": round(ms / nl, 5)} for name, (nl, ms) in prof.items() if nl}

    # End to end through the public API from pinned host buffers: one
    # attn_prefill_host call per step, which copies each entry's valid rows
    # up, runs it, and copies its valid output rows back, largest entry
    # first, the copies of one entry overlapping the others' attention (only
    # valid rows cross the link).  The step's events are on the compute
    # stream, which the call makes wait for the last copy back.
    qh, kh, vh = pinned(torch, q), pinned(torch, k), pinned(torch, v)
    oh = torch.empty(out.shape, dtype=out.dtype, pin_memory=True)

    def e2e_step():
        gqa.attn_prefill_host(cache, ids, qh, kh, vh, nb, out=oh)
        for s in ids:
            gqa.kv_truncate(cache, s, 0)

    for _ in range(2):
        e2e_step()
    ems, _, _ = timed_steps(torch, dist, e2e_step, args.steps, flush)
    e2e_total = dist.max(torch, sum(ems))
    row_q, row_kv = H_q * d * 2, H_kv * d * 2
    e2e = {"value": round(flops * args.steps * dist.world / (e2e_total / 1e3) / 1e12, 3), "unit": "TFLOP/s",
           "h2d_bytes_per_step": int(sum(nb) * (row_q + 2 * row_kv)), "d2h_bytes_per_step": int(sum(nb) * row_q),
           "ms_per_step": round(e2e_total / args.steps, 4),
           "how": "attn_prefill_host (C ABI, pinned host buffers): valid rows up on the library's upload stream, "
                  "one-entry prefills largest first, valid output rows down on its download stream, overlapping "
                  "the other entries' attention"}
    flags = cache.check()
    cache.close()
    del flush
    cfg = {"workload": "bf16 ragged prefill: B=%d, H_q=%d, H_kv=%d, d_h=%d, padded n=%d, valid_lengths=%s "
                       "(~U{512..2048}, seed %d), right padded, N(0,1); one step = attn_prefill + kv_truncate "
                       "to 0" % (B, H_q, H_kv, d, n, nb, workloads.seed_for(2)),
           "global_batch": B * dist.world, "seq_len": n, "parallelism": "replicas x%d" % dist.world,
           "l2": "flushed (512 MiB write, untimed) before every timed step",
           "causal_gflop_per_step": round(flops / 1e9, 3)}
    if args.rope:
        cfg["position_mechanism"] = ("rotary (base 10000), applied inside the library: keys at write, queries in-kernel"
                                     if not args.pre_position else
                                     "rotary (base 10000), pre-position cache: keys stored as given and rotated when "
                                     "read (CUDA-core kernels), queries in-kernel")
    if args.window:
        cfg["sliding_window"] = "W=%d: position p attends to keys max(0, p-W+1)..p; flops count those pairs" % args.window
    return {"value": value, "ms_per_step": total_ms / args.steps, "ms_per_step_median": round(median_ms, 4),
            "roofline": roofline, "e2e": e2e, "gpu_launches": gpu_launches, "kernels": kernels, "config": cfg,
            "t0": s0, "t1": s1, "sustain": {"steps": s_steps, "ms_per_step_median": round(s_med, 4),
                                            "seconds": round(s1 - s0, 3)},
            "timed_region_s": round(t1 - t0, 4), "device_error_flags": flags, "workload": w}


def bench_decode(torch, gqa, dist, args, peaks, peak_src, want_cpu):
    w = workloads.paged_decode(workloads.seed_for(3))
    B, H_q, H_kv, d = w["B"], w["H_q"], w["H_kv"], w["d"]
    L = [int(x) for x in w["lengths"]]
    W = args.window
    q8 = args.kv == "fp8"                    # quantised cache: 1-byte codes + a 4-byte scale per row
    kv_es, kv_extra = (1, 4) if q8 else (2, 0)
    kv_bytes = gqa.work.decode_kv_bytes(L, H_kv, d, kv_es, W, kv_extra)
    # Under a sliding window the sequences grow by one token a step (a
    # rewind may reach back past the window), so the pool and the tables
    # get room for every step of the run; K/V bytes are counted per step.
    grow = 8 * (args.steps + args.warmup + 4) if W else 0
    spare = B * workloads.pages_for(grow + 16) if W else 0
    cache = gqa.Cache(H_kv, d, w["num_pages"] + spare, B, workloads.pages_for(max(L) + grow) + 1, dtype=args.kv,
                      rope=args.rope, page_order=(list(w["page_order"]) + list(range(w["num_pages"],
                      w["num_pages"] + spare))) if W else w["page_order"], window=W,
                      keys_post_position=0 if args.pre_position else 1)
    ids = [cache.seq_create() for _ in range(B)]
    cache.set_decode_kernel(args.decode_kernel)
    for b in range(B):
        kb = to_dev(torch, w["hist_k"][b][None])
        vb = to_dev(torch, w["hist_v"][b][None])
        gqa.kv_append(cache, [ids[b]], kb, vb)
        del kb, vb
    new_k, new_v, q = to_dev(torch, w["new_k"]), to_dev(torch, w["new_v"]), to_dev(torch, w["q"])
    out = torch.empty_like(q)
    cur = [x - 1 for x in L]             # cached lengths before the next step's append
    moved = [0]                          # algorithmic K/V bytes of the steps run so far

    def advance():
        if W:
            for b in range(B):
                cur[b] += 1
            moved[0] += gqa.work.decode_kv_bytes(cur, H_kv, d, kv_es, W, kv_extra)
        else:
            moved[0] += kv_bytes
            for b in range(B):
                gqa.kv_truncate(cache, ids[b], L[b] - 1)

    def step():
        gqa.attn_decode_append(cache, ids, q, new_k, new_v, out=out)
        advance()

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    cache.profile_read()
    m0 = moved[0]
    ms, t0, t1 = timed_steps(torch, dist, step, args.steps)
    region_bytes = moved[0] - m0
    region_launches = cache.profile_read()
    total_ms = dist.max(torch, sum(ms))
    value = region_bytes * dist.world / (total_ms / 1e3) / 1e9
    cache.profile(True)
    m0 = moved[0]
    timed_steps(torch, dist, step, args.steps)
    kv_bytes = (moved[0] - m0) // args.steps          # per launch (the mean, under a window)
    cache.profile(False)
    prof = cache.profile_read()
    kernel = max(("prefill_tc", "decode_split", "decode_cluster", "attn_simt"), key=lambda x: prof[x][1])
    launches, kms = prof[kernel]
    avg_ms = kms / max(1, launches)
    achieved = kv_bytes / (avg_ms / 1e3) / 1e9
    roofline = {"bound": "hbm", "achieved": round(achieved, 1), "peak": peaks["hbm_gbs"], "unit": "GB/s",
                "frac": round(achieved / peaks["hbm_gbs"], 4), "traffic": traffic_for("decode", kernel),
                "kernel": kernel,
                "kernel_ms": round(avg_ms, 4), "algorithmic_bytes_per_launch": kv_bytes,
                "peak_source": "%s HBM copy bandwidth" % peak_src}

    # The same step back to back for 0.6 s, for the clock record.
    s0, s1, s_steps, s_med = sustain(torch, step)
    cache.profile_read()

    # End to end through the public API: one attn_decode_append_host call
    # per step (pinned host q, k, v up; the step; out back down).
    qh, kh, vh = pinned(torch, q), pinned(torch, new_k), pinned(torch, new_v)
    oh = torch.empty(out.shape, dtype=out.dtype, pin_memory=True)

    def e2e_step():
        gqa.attn_decode_append_host(cache, ids, qh, kh, vh, out=oh)
        advance()

    for _ in range(2):
        e2e_step()
    m0 = moved[0]
    ems, _, _ = timed_steps(torch, dist, e2e_step, args.steps)
    e2e_bytes = moved[0] - m0
    e2e_total = dist.max(torch, sum(ems))
    res = {"metric": "decode KV-read GB/s", "value": round(value, 1), "unit": "GB/s",
           "ms_per_step": round(total_ms / args.steps, 4), "roofline": roofline,
           "e2e": {"value": round(e2e_bytes * dist.world / (e2e_total / 1e3) / 1e9, 1), "unit": "GB/s",
                   "h2d_bytes_per_step": int(q.nbytes + new_k.nbytes + new_v.nbytes),
                   "d2h_bytes_per_step": int(out.nbytes), "ms_per_step": round(e2e_total / args.steps, 4),
                   "how": "attn_decode_append_host (C ABI, pinned host buffers): q, k, v up, the fused step, out "
                          "down, all on the caller's stream"},
           "ms_per_step_median": round(statistics.median(ms), 4),
           "sustain": {"steps": s_steps, "ms_per_step_median": round(s_med, 4), "seconds": round(s1 - s0, 3)},
           "gpu_launches": sum(nl for nl, _ in region_launches.values()),
           "kernels": {name: {"launches": nl, "avg_ms": round(ms / nl, 5)} for name, (nl, ms) in prof.items() if nl},
           "config": {"workload": "bf16 paged decode: B=%d, H_q=%d, H_kv=%d, d_h=%d, cache lengths ~U{1024..8192} "
                                  "(seed %d, sum %d tokens) incl. the appended token, pages placed by a seeded "
                                  "random permutation; one step = attn_decode_append (the token appended and attended in one call) + kv_truncate back"
                                  % (B, H_q, H_kv, d, workloads.seed_for(3), sum(L)),
                      "l2": "not flushed: %.2f GB of K/V per step exceeds the 129 MB L2" % (kv_bytes / 1e9),
                      "kv_bytes_per_step": kv_bytes}}
    if args.rope:
        res["config"]["position_mechanism"] = ("rotary (base 10000): queries rotated in-kernel" if not args.pre_position
                                               else "rotary (base 10000), pre-position cache: keys rotated as the "
                                                    "split-K decode reads them, queries in-kernel")
    if W:
        res["config"]["sliding_window"] = ("W=%d: a decode reads the last min(L, W) tokens; sequences grow by one "
                                           "token a step (no rewind), K/V bytes counted per step" % W)
    if want_cpu:
        import oracle
        nth = oracle.default_threads()
        cm = oracle.CacheModel(sum(workloads.pages_for(x) for x in L[:8]), 8, workloads.pages_for(max(L)) + 1,
                               H_kv, d, args.kv, window=W)
        sm = [cm.create() for _ in range(8)]
        for j in range(8):
            cm.write([sm[j]], [w["hist_k"][j]], [w["hist_v"][j]])
        oracle.append(cm, sm, w["new_k"][:8], w["new_v"][:8])
        dt, reps = 0.0, 0
        while dt < args.cpu_budget:
            t0c = time.perf_counter()
            oracle.decode(cm, sm, w["q"][:8], nthreads=nth)
            dt += time.perf_counter() - t0c
            reps += 1
        by = gqa.work.decode_kv_bytes(L[:8], H_kv, d, kv_es, W, kv_extra) * reps
        res["cpu_baseline"] = {"value": round(by / dt / 1e9, 3), "unit": "GB/s", "cores": nth, "kind": "oracle",
                               "sample": "fp64 oracle decode of sequences 0..7 (%d cached tokens, %.1f MB of "
                                         "bf16 K/V), %d repetitions: %.1f GB in %.1f s"
                                         % (sum(L[:8]), by / reps / 1e6, reps, by / 1e9, dt)}
    if q8:
        res["config"]["kv_cache"] = ("FP8 E4M3 codes + one fp32 scale per (token, head) row, written by the "
                                     "library from the bf16 K/V; bytes counted as read (codes and scales)")
    if not W and not q8:
        res["multi_token"] = bench_multi_token(torch, gqa, dist, args, peaks, peak_src, cache, ids, L, w)
    res["device_error_flags"] = cache.check()
    res["t0"], res["t1"] = s0, s1
    cache.close()
    return res


def bench_multi_token(torch, gqa, dist, args, peaks, peak_src, cache, ids, L, w, T=4):
    """Multi-token decode over the paged-decode cache: T new tokens per
    sequence (a speculative draft block) attend causally to the cached
    L_b - 1 tokens and to each other, through attn_prefill with n = T; one
    step = the chunk + kv_truncate back.  HBM-bound like decode: the work is
    the K/V bytes read, sum_b (L_b - 1 + T) tokens."""
    B, H_q, H_kv, d = w["B"], w["H_q"], w["H_kv"], w["d"]
    ch = workloads.draft_chunk(workloads.seed_for(6), B, T, H_q, H_kv, d)
    q, k, v = to_dev(torch, ch["q"]), to_dev(torch, ch["k"]), to_dev(torch, ch["v"])
    out = torch.empty_like(q)
    counts = [T] * B
    kv_bytes = gqa.work.decode_kv_bytes([x - 1 + T for x in L], H_kv, d, 2)
    flops = gqa.work.prefill_flops([x - 1 for x in L], counts, H_q, d)

    def step():
        gqa.attn_prefill(cache, ids, q, k, v, counts, out=out)
        for b in range(B):
            gqa.kv_truncate(cache, ids[b], L[b] - 1)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    cache.profile_read()
    ms, _, _ = timed_steps(torch, dist, step, args.steps)
    region = cache.profile_read()
    total_ms = dist.max(torch, sum(ms))
    prof = profiled(torch, dist, cache, step, args.steps)
    kernel = "prefill_tc" if prof["prefill_tc"][0] else "attn_simt"
    launches, kms = prof[kernel]
    avg_ms = kms / max(1, launches)
    achieved = kv_bytes / (avg_ms / 1e3) / 1e9
    return {"metric": "multi-token decode KV-read GB/s", "unit": "GB/s",
            "value": round(kv_bytes * args.steps * dist.world / (total_ms / 1e3) / 1e9, 1),
            "ms_per_step": round(total_ms / args.steps, 4),
            "tflops": round(flops * args.steps * dist.world / (total_ms / 1e3) / 1e12, 2),
            "roofline": {"bound": "hbm", "achieved": round(achieved, 1), "peak": peaks["hbm_gbs"], "unit": "GB/s",
                         "frac": round(achieved / peaks["hbm_gbs"], 4), "kernel": kernel,
                         "kernel_ms": round(avg_ms, 4), "algorithmic_bytes_per_launch": kv_bytes,
                         "peak_source": "%s HBM copy bandwidth" % peak_src},
            "gpu_launches": sum(nl for nl, _ in region.values()),
            "kernels": {name: {"launches": nl, "avg_ms": round(x / nl, 5)} for name, (nl, x) in prof.items() if nl},
            "config": {"workload": "bf16 multi-token decode: the paged-decode cache (B=%d, H_q=%d, H_kv=%d, d_h=%d, "
                                   "L_b - 1 cached tokens) plus T=%d new tokens per sequence, N(0,1) (seed %d); "
                                   "one step = attn_prefill(n=T) + kv_truncate back" % (B, H_q, H_kv, d, T,
                                                                                        workloads.seed_for(6)),
                       "kv_bytes_per_step": kv_bytes, "causal_gflop_per_step": round(flops / 1e9, 3)}}


def profiled(torch, dist, cache, step, K, flush=None):
    """Per-kernel (launches, total ms) of K steps, each launch bracketed by
    events on its stream."""
    cache.profile_read()
    cache.profile(True)
    timed_steps(torch, dist, step, K, flush)
    cache.profile(False)
    return cache.profile_read()


def tensor_roofline(flops, prof, peaks):
    kernel = "prefill_tc" if prof["prefill_tc"][0] else "attn_simt"
    nl, kms = prof[kernel]
    avg = kms / max(1, nl)
    achieved = flops / (avg / 1e3) / 1e12
    return {"kernel": kernel, "kernel_ms": round(avg, 4), "achieved_tflops": round(achieved, 1),
            "frac": round(achieved / peaks["bf16_tflops"], 4),
            "roofline": {"bound": "tensor", "achieved": round(achieved, 1), "peak": peaks["bf16_tflops"],
                         "unit": "TFLOP/s", "frac": round(achieved / peaks["bf16_tflops"], 4), "traffic": None,
                         "kernel": kernel, "kernel_ms": round(avg, 4), "algorithmic_flops_per_launch": flops}}


def oracle_group_rate(q_bits, k_bits, v_bits, qpos, g, budget_s, what):
    """The fp64 oracle on the host cores over KV group 0 (its g query heads)
    of the given query rows, repeated until about budget_s seconds; causal
    TFLOP/s counted as for the GPU (4 d_h per visible pair and head)."""
    import oracle
    nth = oracle.default_threads()
    d = q_bits.shape[-1]
    Q = oracle.to_f64(q_bits[:, :g], "bf16")
    K = oracle.to_f64(k_bits[:, :1], "bf16")
    V = oracle.to_f64(v_bits[:, :1], "bf16")
    qpos = np.asarray(qpos)
    flops = 4 * d * g * int(np.sum(qpos + 1))
    used, reps = 0.0, 0
    while used < budget_s:
        t0 = time.perf_counter()
        oracle.attention(Q, K, V, qpos, nthreads=nth)
        used += time.perf_counter() - t0
        reps += 1
    return {"value": round(flops * reps / used / 1e12, 4), "unit": "TFLOP/s", "cores": nth, "kind": "oracle",
            "sample": "%s: KV group 0 (%d query heads), %d query rows at positions %d..%d, %d repetitions: %.2f "
                      "GFLOP causal in %.1f s" % (what, g, len(qpos), qpos.min(), qpos.max(), reps,
                                                 flops * reps / 1e9, used)}


def bench_wide(torch, gqa, dist, args, peaks, want_cpu=False):
    """Wide-GQA long context: B=1, H_q=48, H_kv=8, prefill T=8192, then 256
    steps of attn_decode_append (L = 8193..8448)."""
    w = workloads.wide_gqa(workloads.seed_for(4))
    T, H_q, H_kv, d, steps = w["n"], w["H_q"], w["H_kv"], w["d"], w["steps"]
    per_seq = workloads.pages_for(T + steps) + 1
    c = gqa.Cache(H_kv, d, per_seq + 4, 1, per_seq, dtype="bf16")
    c.set_decode_kernel(args.decode_kernel)
    s = c.seq_create()
    q, k, v = to_dev(torch, w["q"]), to_dev(torch, w["k"]), to_dev(torch, w["v"])
    out = torch.empty_like(q)
    flush = torch.empty(512 << 20, dtype=torch.uint8, device="cuda")
    flops = gqa.work.prefill_flops([0], [T], H_q, d)

    def pre_step():
        gqa.attn_prefill(c, [s], q, k, v, [T], out=out)
        gqa.kv_truncate(c, s, 0)

    for _ in range(args.warmup):
        flush.zero_()
        pre_step()
    ms, _, _ = timed_steps(torch, dist, pre_step, args.steps, flush)
    pre = {"tflops_step": round(flops * args.steps / (sum(ms) / 1e3) / 1e12, 1),
           "ms_per_step": round(sum(ms) / args.steps, 4), "gflop": round(flops / 1e9, 1)}
    pre.update(tensor_roofline(flops, profiled(torch, dist, c, pre_step, args.steps, flush), peaks))
    if want_cpu:
        rows = np.arange(T - 256, T)
        pre["cpu_baseline"] = oracle_group_rate(w["q"][0, rows], w["k"][0], w["v"][0], rows, H_q // H_kv,
                                                min(args.cpu_budget, 4.0), "fp64 oracle, wide-GQA prefill")

    gqa.attn_prefill(c, [s], q, k, v, [T], out=out)
    dq, dk, dv = to_dev(torch, w["dec_q"]), to_dev(torch, w["dec_k"]), to_dev(torch, w["dec_v"])
    dout = torch.empty_like(dq[0])
    kv_bytes = gqa.work.decode_kv_bytes([T + t + 1 for t in range(steps)], H_kv, d, 2)

    def decode_all():
        for t in range(steps):
            gqa.attn_decode_append(c, [s], dq[t], dk[t], dv[t], out=dout)
        gqa.kv_truncate(c, s, T)

    decode_all()
    ms_res, _, _ = timed_steps(torch, dist, decode_all, 3)
    t_res = sum(ms_res) / 3
    # Device time with the host running ahead: a sleep kernel holds the GPU
    # while every step is queued (1.5x the host's queueing time at 2.1 GHz),
    # so no launch waits for the host; per-launch events and the span of the
    # whole queued run are then GPU time.
    torch.cuda.synchronize()
    h0 = time.perf_counter()
    decode_all()
    host_s = time.perf_counter() - h0
    torch.cuda.synchronize()
    c.profile_read()
    c.profile(True)
    qa, qb = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda._sleep(int(host_s * 1.5 * 2.1e9))
    qa.record()
    h0 = time.perf_counter()
    decode_all()
    host_q = time.perf_counter() - h0
    qb.record()
    qb.synchronize()
    c.profile(False)
    prof = c.profile_read()
    q_ms = qa.elapsed_time(qb)
    kname = max(("prefill_tc", "decode_split", "decode_cluster", "attn_simt"), key=lambda x: prof[x][0])
    k_us = prof[kname][1] / max(1, prof[kname][0]) * 1e3
    # The same queued run without per-launch events: the device time of a
    # step as a decode loop sees it (launch gaps included, no event pairs).
    torch.cuda.synchronize()
    na, nb = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda._sleep(int(host_s * 1.5 * 2.1e9))
    na.record()
    decode_all()
    nb.record()
    nb.synchronize()
    n_us = na.elapsed_time(nb) / steps * 1e3
    step_ms = []
    for t in range(steps):                          # L2 flushed before every step
        flush.zero_()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record()
        gqa.attn_decode_append(c, [s], dq[t], dk[t], dv[t], out=dout)
        b.record()
        b.synchronize()
        step_ms.append(a.elapsed_time(b))
    gqa.kv_truncate(c, s, T)
    dec = {"steps": steps, "kv_gb": round(kv_bytes / 1e9, 3),
           "l2_resident": {"us_per_step": round(t_res / steps * 1e3, 2),
                           "gbs": round(kv_bytes / (t_res / 1e3) / 1e9, 1)},
           "kernel": {"name": kname, "us_per_launch_events": round(k_us, 2),
                      "gbs": round(kv_bytes / steps / (k_us / 1e6) / 1e9, 1),
                      "note": "each launch bracketed by the library's profiling events (start event after the "
                              "host-side preparation): launch latency and event overhead included",
                      "append_us_per_launch": round(prof["cache_write"][1] / max(1, prof["cache_write"][0]) * 1e3, 2)},
           "queued": {"us_per_step": round(q_ms / steps * 1e3, 2), "gbs": round(kv_bytes / (q_ms / 1e3) / 1e9, 1),
                      "host_us_per_step": round(host_q / steps * 1e6, 2),
                      "how": "all steps queued behind a sleep kernel; span of the run on the GPU (append + "
                             "decode + profiling events)"},
           "queued_no_events": {"us_per_step": round(n_us, 2), "gbs": round(kv_bytes / steps / (n_us / 1e6) / 1e9, 1),
                                "how": "the queued run again without per-launch events: device time per step "
                                       "(block-table uploads when the sequence takes a new page, launch gaps "
                                       "and the fused append+decode kernel; the descriptors travel in the "
                                       "launch parameters)"},
           "l2_flushed": {"us_per_step": round(sum(step_ms) / steps * 1e3, 2),
                          "gbs": round(kv_bytes / (sum(step_ms) / 1e3) / 1e9, 1),
                          "frac_hbm": round(kv_bytes / (sum(step_ms) / 1e3) / 1e9 / peaks["hbm_gbs"], 4)},
           "roofline": {"bound": "hbm", "achieved": round(kv_bytes / steps / (n_us / 1e6) / 1e9, 1),
                        "peak": peaks["hbm_gbs"], "unit": "GB/s",
                        "frac": round(kv_bytes / steps / (n_us / 1e6) / 1e9 / peaks["hbm_gbs"], 4),
                        "traffic": traffic_for("wide_decode", kname),
                        "kernel": kname, "kernel_ms": round(n_us / 1e3, 5),
                        "algorithmic_bytes_per_launch": kv_bytes // steps,
                        "note": "device time per queued step, one event pair around all steps (no per-launch "
                                "events); the 34 MB of K/V is L2-resident; traffic: one launch with cold caches "
                                "under ncu"},
           "note": "one step = attn_decode_append of one sequence, called from Python: the step times "
                   "include the host side of the call, which is longer than the GPU work; 34 MB of K/V fits "
                   "in L2; queued_no_events = device time per step with the steps queued ahead of the GPU and "
                   "no per-launch events (L2-resident); kernel = each launch bracketed by events; l2_flushed = "
                   "each step after a 512 MiB L2 flush"}
    flags = c.check()
    c.close()
    return {"workload": "bf16 wide GQA: B=1, H_q=48, H_kv=8 (g=6), d_h=128, prefill T=%d, then %d append+decode "
                        "steps (seed %d)" % (T, steps, workloads.seed_for(4)),
            "prefill": pre, "decode": dec, "device_error_flags": flags}


def bench_prefix(torch, gqa, dist, args, peaks, want_cpu=False):
    """Prefix reuse and edit: one 4096-token prefix, 8 forks each prefilling
    512 new tokens over it (P = 4096); fork 0 edited at m = 2000 (truncate +
    re-prefill of the 2608 following tokens)."""
    w = workloads.prefix_edit(workloads.seed_for(5))
    P0, B, n_new, m = w["prefix"], w["B"], w["n_new"], w["m"]
    H_q, H_kv, d = w["H_q"], w["H_kv"], w["d"]
    per_seq = workloads.pages_for(P0 + n_new) + 1
    pages = workloads.pages_for(P0) + B * workloads.pages_for(n_new) + workloads.pages_for(P0 + n_new) + 16
    c = gqa.Cache(H_kv, d, pages, B + 2, per_seq, dtype="bf16")
    root = c.seq_create()
    gqa.attn_prefill(c, [root], to_dev(torch, w["pre_q"]), to_dev(torch, w["pre_k"]), to_dev(torch, w["pre_v"]), [P0])
    forks = [c.seq_fork(root, P0) for _ in range(B)]
    nq, nk, nv = to_dev(torch, w["new_q"]), to_dev(torch, w["new_k"]), to_dev(torch, w["new_v"])
    out = torch.empty_like(nq)
    flush = torch.empty(512 << 20, dtype=torch.uint8, device="cuda")
    flops = gqa.work.prefill_flops([P0] * B, [n_new] * B, H_q, d)

    def inc_step():
        gqa.attn_prefill(c, forks, nq, nk, nv, [n_new] * B, out=out)
        for f in forks:
            gqa.kv_truncate(c, f, P0)

    for _ in range(args.warmup):
        flush.zero_()
        inc_step()
    ms, _, _ = timed_steps(torch, dist, inc_step, args.steps, flush)
    inc = {"tflops_step": round(flops * args.steps / (sum(ms) / 1e3) / 1e12, 1),
           "ms_per_step": round(sum(ms) / args.steps, 4), "gflop": round(flops / 1e9, 1)}
    inc.update(tensor_roofline(flops, profiled(torch, dist, c, inc_step, args.steps, flush), peaks))
    if want_cpu:
        rows = P0 + np.arange(n_new)
        inc["cpu_baseline"] = oracle_group_rate(w["new_q"][0], np.concatenate([w["pre_k"][0], w["new_k"][0]]),
                                                np.concatenate([w["pre_v"][0], w["new_v"][0]]), rows,
                                                H_q // H_kv, min(args.cpu_budget, 3.0),
                                                "fp64 oracle, fork 0's incremental prefill")

    gqa.attn_prefill(c, forks, nq, nk, nv, [n_new] * B, out=out)
    n_re = P0 + n_new - m
    eq, ek, ev = to_dev(torch, w["edit_q"]), to_dev(torch, w["edit_k"]), to_dev(torch, w["edit_v"])
    eout = torch.empty_like(eq)
    eflops = gqa.work.prefill_flops([m], [n_re], H_q, d)

    def edit_step():
        gqa.kv_truncate(c, forks[0], m)
        gqa.attn_prefill(c, [forks[0]], eq, ek, ev, [n_re], out=eout)

    for _ in range(args.warmup):
        flush.zero_()
        edit_step()
    ms, _, _ = timed_steps(torch, dist, edit_step, args.steps, flush)
    ed = {"tflops_step": round(eflops * args.steps / (sum(ms) / 1e3) / 1e12, 1),
          "ms_per_step": round(sum(ms) / args.steps, 4), "gflop": round(eflops / 1e9, 1)}
    ed.update(tensor_roofline(eflops, profiled(torch, dist, c, edit_step, args.steps, flush), peaks))
    flags = c.check()
    c.close()
    return {"workload": "bf16 prefix reuse: a %d-token prefix shared by %d forks, each prefilling %d new tokens "
                        "(P=%d); edit of fork 0 at m=%d: truncate + re-prefill of %d tokens (seed %d)"
                        % (P0, B, n_new, P0, m, n_re, workloads.seed_for(5)),
            "incremental": inc, "edit": ed, "device_error_flags": flags}


# ---------------------------------------------------------------------------
# reference arm: the fp64 oracle on the host cores
# ---------------------------------------------------------------------------

def run_reference(args, dist):
    if dist.rank != 0:
        return 0
    import oracle
    w = workloads.ragged_prefill(workloads.seed_for(2))
    B, n, H_q, H_kv, d = w["B"], w["n"], w["H_q"], w["H_kv"], w["d"]
    g = H_q // H_kv
    nth = oracle.default_threads()

    def work(b):
        nb = int(w["valid_lengths"][b])
        return 4 * d * g * (nb * (nb + 1) // 2)

    def step(i):
        b = i % B
        nb = int(w["valid_lengths"][b])
        cm = oracle.CacheModel(workloads.pages_for(nb), 1, workloads.pages_for(nb), 1, d, "bf16")
        s = cm.create()
        # KV group 0 only: its g query heads and its one KV head.
        oracle.prefill(cm, [s], w["q"][b:b + 1, :, :g], w["k"][b:b + 1, :, :1], w["v"][b:b + 1, :, :1], [nb],
                       nthreads=nth)
        return work(b)

    for i in range(args.warmup):
        step(i)
    flops, t = 0, 0.0
    for i in range(args.steps):
        t0 = time.perf_counter()
        flops += step(i)
        t += time.perf_counter() - t0
    value = flops / t / 1e12
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": t / args.steps * 1e3,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": "bf16 ragged prefill: B=4, H_q=32, H_kv=8, d_h=128, padded n=2048, valid "
                                   "lengths %s (seed %d); each reference step is one sequence's KV group 0 "
                                   "(%d query heads)" % (list(map(int, w["valid_lengths"])),
                                                         workloads.seed_for(2), g)},
            "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": nth, "kind": "oracle",
                             "sample": "per step: fp64 oracle prefill of one sequence (cycling 0..3), KV group 0"},
            "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line))
    return 0


# ---------------------------------------------------------------------------

def main():
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["gqa", "reference"], default="gqa")
    ap.add_argument("--no-decode", action="store_true", help="skip the decode object")
    ap.add_argument("--no-prefill", action="store_true", help="decode only (for profiling runs)")
    ap.add_argument("--no-cpu", action="store_true", help="skip the CPU oracle baseline")
    ap.add_argument("--rope", action="store_true",
                    help="caches with the rotary position mechanism applied by the library")
    ap.add_argument("--pre-position", action="store_true",
                    help="with --rope: caches that store keys before the rotation and rotate them when read")
    ap.add_argument("--decode-kernel", choices=["auto", "tensor_core", "cuda_core", "cluster"], default="auto",
                    help="decode kernel of attn_decode (auto: tensor-core for bf16, d_h = 128)")
    ap.add_argument("--kv", choices=["bf16", "fp8"], default="bf16",
                    help="decode cache type (fp8: FP8 E4M3 codes with per-row scales; decode only)")
    ap.add_argument("--window", type=int, default=0,
                    help="caches with a sliding window of this many tokens (0 = none)")
    ap.add_argument("--no-extra", action="store_true",
                    help="skip the wide-GQA long-context and prefix-reuse/edit workloads")
    ap.add_argument("--cpu-budget", type=float, default=10.0,
                    help="seconds of fp64 oracle work per CPU baseline (rank 0, N=1)")
    args = ap.parse_args()
    args.warmup = max(3, args.warmup)
    if args.pre_position and not args.rope:
        ap.error("--pre-position needs --rope (the cache rotates the keys it stores before the rotation)")
    args.extra = not args.no_extra
    if args.kv == "fp8":
        args.no_prefill = True               # the quantised cache is measured on decode
        args.extra = False
    dist = Dist()
    if args.impl == "reference":
        return run_reference(args, dist)

    import torch
    import causal_gqa_attention_02_gb300 as gqa
    dist.setup(torch)
    peaks, peak_src = load_peaks()
    clocks = ClockSampler(device_uuid(torch)) if dist.rank == 0 else None
    want_cpu = dist.rank == 0 and dist.world == 1 and not args.no_cpu
    wide = prefix = None
    try:
        time.sleep(0.3 if clocks else 0)
        pre = None if args.no_prefill else bench_prefill(torch, gqa, dist, args, peaks, peak_src)
        dec = None if args.no_decode else bench_decode(torch, gqa, dist, args, peaks, peak_src, want_cpu=want_cpu)
        # Every rank runs the replicas (the timed regions have barriers).
        if pre is not None and args.extra:
            wide = bench_wide(torch, gqa, dist, args, peaks, want_cpu)
            prefix = bench_prefix(torch, gqa, dist, args, peaks, want_cpu)
    finally:
        if clocks:
            clocks.stop()
    if dist.rank == 0 and pre is None:
        dec["clocks"] = clocks.summary(dec.pop("t0"), dec.pop("t1"))
        print(json.dumps({"decode": dec}))
    elif dist.rank == 0:
        line = {"metric": METRIC, "value": round(pre["value"], 3), "unit": "TFLOP/s", "n_gpus": dist.world,
                "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(pre["ms_per_step"], 4),
                "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
                "data": "synthetic", "config": pre["config"], "roofline": pre["roofline"], "e2e": pre["e2e"],
                "ms_per_step_median": pre["ms_per_step_median"],
                "gpu_launches": pre["gpu_launches"], "kernels": pre["kernels"],
                "clocks": clocks.summary(pre["t0"], pre["t1"]), "sustain": pre["sustain"],
                "timed_region_s": pre["timed_region_s"],
                "device_error_flags": pre["device_error_flags"]}
        if line["clocks"].get("sm_mhz"):
            # time x clock: the step's cost in clock cycles, comparable across clocks
            line["clocks"]["ms_per_step_x_ghz"] = round(pre["ms_per_step"] * line["clocks"]["sm_mhz"] / 1e3, 5)
        if not args.no_cpu and dist.world == 1:
            line["cpu_baseline"] = prefill_cpu_baseline(pre["workload"], args.cpu_budget)
        if dec is not None:
            dec["clocks"] = clocks.summary(dec.pop("t0"), dec.pop("t1"))
            line["decode"] = dec
        if wide is not None:
            line["wide_gqa"] = wide
            line["prefix_reuse"] = prefix
        print(json.dumps(line))
    dist.done()
    return 0


if __name__ == "__main__":
    sys.exit(main())
