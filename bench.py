#!/usr/bin/env python
"""Benchmark of one tree-verify step on GB300.

A step is one pass of the whole verify path over one batch: draft-KV scatter,
KV index marshaling, tree-mask packing and tree-verify attention (with its
split merge). By default the three marshaling steps run as one launch
(mla_tree_prepare, which packs the mask in its bit form: one bit per (row,
column)) ahead of mla_tree_verify_bits; --marshal separate --mask bytes runs
the four separate calls with the byte mask.

Default workload (--config 5): the ragged mixed batch of 64 requests,
prefixes floor(exp(U(ln 128, ln 131072))), tree sizes U{8..64} (even
requests chains, odd ones random trees), 64 heads, 2^22-slot pool, run as
one captured CUDA graph per step. --config 1..4 select the other four
workloads (the live 9-node shape, 8 requests of 1k-4k keys, 32 requests of
8192 keys, 4 requests of 200000 keys).

Timing: the whole step is captured once as a CUDA graph (what a serving
engine replays; there the verify kernel starts while the marshaling kernel
finishes) and the timed steps replay it between CUDA events on the launching
stream. The same number of steps is then replayed call by call (one graph
per call, events between them) for the per-call times, which give
us_per_call and the roofline of the verify call. L2 is flushed
between steps by writing a 256 MiB buffer (outside the events): the buffer is
written and then read back, so L2 holds only clean lines of it and the timed
reads pay no write-backs. Inputs are resident in HBM when the timed region
starts.

value = KV bytes the steps had to read (every prefix + draft row of every
request once, 1152 B per row) / device time, summed over ranks / max time.
e2e = the same metric through the public API with host buffers: pinned
host -> device copies of the step's inputs, the step's calls, and the device
-> host read of out and lse, all inside the timed region.

The CPU baseline and --impl reference time the fp64 oracle on the host
cores on a bounded sample of the same workload: whole requests (all their
draft rows and heads, at least 256 rows in all) in a seeded random order,
their index marshaling, mask packing and attention; value = the KV bytes of
the requests done / the time taken.
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

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "tree-verify MLA attention µs/call and KV GB/s (% of GB300 HBM roofline)"
FALLBACK_HBM_GBS, FALLBACK_BF16_TFLOPS = 6800.0, 1900.0
FLUSH_BYTES = 256 << 20
# timed steps per workload when --steps is not given: about a second of
# device time in the timed region
DEFAULT_STEPS = {1: 4000, 2: 4000, 3: 200, 4: 500, 5: 60}


def _peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            p = json.load(f)
        return float(p["hbm_gbs"]), float(p["bf16_tflops"]), float(p.get("bf16_tflops_sustained", 0)), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, FALLBACK_BF16_TFLOPS, 1700.0, "fallback"


def alg_cost(w, mask_bits=False, skip_prefix=False):
    """Algorithmic bytes and flops of one verify call: every key row once,
    its index, the mask (a byte, or a bit in whole 32-bit words, per (row,
    key); with the prefix skip only the draft columns' bytes or words), q
    in, out and lse out; flops over visible (row, key) pairs only."""
    H = w.heads
    qo = w.qo_indptr.tolist()
    byts, flops = 0, 0
    for b in range(w.batch):
        n, P = w.tree_sizes[b], w.prefix_lens[b]
        L = P + n
        if skip_prefix:  # draft columns only (the words that hold them)
            mask_bytes = n * 4 * ((L + 31) // 32 - P // 32) if mask_bits else n * n
        else:
            mask_bytes = n * 4 * ((L + 31) // 32) if mask_bits else n * L
        byts += L * 1152 + L * 4 + mask_bytes + n * H * (1152 + 1024 + 4)
        par = w.parents[qo[b]:qo[b + 1]].tolist()
        depth = []
        for i, p in enumerate(par):
            depth.append(1 if p < 0 else depth[p] + 1)
        flops += 2 * 1088 * H * (n * P + sum(depth))
    return byts, flops


class ClockSampler:
    """nvidia-smi clock / throttle sampling while the timed region runs."""

    Q = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        self.index = index
        self.proc = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), "--query-gpu=" + self.Q,
                 "--format=csv,noheader,nounits", "-lms", "50"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"], "samples": 0}
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except Exception:
            self.proc.kill()
            out = ""
        sm, mx, reasons, n = [], [], set(), 0
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in out.strip().splitlines():
            f = [x.strip() for x in line.split(",")]
            if len(f) < 8:
                continue
            try:
                sm.append(float(f[0])); mx.append(float(f[1]))
            except ValueError:
                continue
            n += 1
            for nm, v in zip(names, f[4:8]):
                if v.lower() == "active":
                    reasons.add(nm)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(mx) if mx else None,
                "reasons": sorted(reasons), "samples": n}


def _code_tokens(text):
    """C/CUDA source with its comments removed and every run of white space
    outside string and character literals made one space, so that editing a
    comment or the layout does not change what is hashed."""
    out, i, n = [], 0, len(text)

    def space():
        if out and out[-1] != " ":
            out.append(" ")

    while i < n:
        c = text[i]
        if c in "\"'":
            j = i + 1
            while j < n and text[j] != c:
                j += 2 if text[j] == "\\" else 1
            out.append(text[i:j + 1])
            i = j + 1
        elif text.startswith("//", i):
            j = text.find("\n", i)
            i = n if j < 0 else j
        elif text.startswith("/*", i):
            j = text.find("*/", i + 2)
            i = n if j < 0 else j + 2
            space()
        elif c.isspace():
            space()
            i += 1
        else:
            out.append(c)
            i += 1
    return "".join(out).strip()


def _kernel_source_hash():
    """Hash of the kernel sources the DRAM traffic in profiles/traffic.json
    was measured on (code only: see _code_tokens)."""
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "speculative_decode_mla_tree_gb300", "csrc")
    for name in sorted(os.listdir(csrc)):
        if name.startswith("verify") or name.endswith((".cuh", ".h")):
            with open(os.path.join(csrc, name), encoding="utf-8") as f:
                h.update(_code_tokens(f.read()).encode())
    return h.hexdigest()[:16]


def _traffic(key):
    """DRAM bytes per launch of the verify call on one workload (key
    "verify_c<N>") from the committed ncu summary, if it was taken on the
    current kernel sources; else None."""
    try:
        with open(os.path.join(ROOT, "profiles", "traffic.json")) as f:
            t = json.load(f)
        e = t.get(key)
        if e and e.get("source_hash") == _kernel_source_hash():
            return float(e["dram_bytes_per_launch"])
    except Exception:
        pass
    return None


def max_over_ranks(x, device=None):
    """Largest value of x over all ranks of the default process group (x itself
    when not distributed). The step time of a multi-GPU run is the slowest
    rank's: every rank replays the same workload on its own GPU."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return float(x)
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def whole_job_gbs(world, steps, kv_bytes, total_ms):
    """Aggregate KV GB/s of a weak-scaling run: every rank reads kv_bytes per
    step, the job takes the slowest rank's time."""
    return world * steps * kv_bytes / (total_ms * 1e-3) / 1e9


class OracleSampler:
    """The fp64 oracle on whole requests of one workload, in a seeded random
    order. The pool with the draft rows scattered in is built once, before
    any timing (a copy of the whole pool); each timed request then runs the
    oracle's index marshaling, mask packing and attention of all its rows."""

    def __init__(self, w, seed=0):
        import numpy as np
        import torch

        import oracle

        self.np, self.oracle = np, oracle
        self.w = w
        pool_bits = w.dense_pool().view(torch.int16).numpy().view(np.uint16)
        dkv = w.draft_kv.view(torch.int16).numpy().view(np.uint16)
        self.pool = oracle.draft_kv_scatter(pool_bits, dkv, w.out_cache_loc)
        del pool_bits
        self.q_bits = w.q.view(torch.int16).numpy().view(np.uint16)
        self.qo = w.qo_indptr.numpy()
        self.order = np.random.default_rng(seed).permutation(w.batch)
        self.k = 0

    def request(self):
        """One request's oracle work; returns (KV bytes, rows)."""
        w, o = self.w, self.oracle
        b = int(self.order[self.k % w.batch])
        self.k += 1
        kv_indices, kv_indptr = o.kv_indices_build(w.prefix_indices, w.prefix_indptr,
                                                   w.out_cache_loc, w.qo_indptr)
        mask_indptr, mask = o.tree_mask_pack(w.parents, w.qo_indptr, kv_indptr)
        rows = [(t, h) for t in range(self.qo[b], self.qo[b + 1]) for h in range(w.heads)]
        o.verify_attention(self.q_bits, self.pool, kv_indices, kv_indptr, w.qo_indptr, mask,
                           mask_indptr, w.heads, w.sm_scale, rows=rows)
        return (w.prefix_lens[b] + w.tree_sizes[b]) * 1152, len(rows)

    def run(self, budget_s=None, steps=None, min_rows=256):
        """Requests until budget_s seconds have passed (and at least
        min_rows rows are done), or exactly `steps` requests; returns
        (GB/s, seconds, rows, requests)."""
        done = rows = k = 0
        t0 = time.perf_counter()
        while True:
            b, r = self.request()
            done += b
            rows += r
            k += 1
            el = time.perf_counter() - t0
            if steps is not None:
                if k >= steps:
                    break
            elif el >= budget_s and rows >= min_rows:
                break
        return done / el / 1e9, el, rows, k


def cpu_baseline(w, budget_s):
    """Time the fp64 oracle on this host's cores; returns (GB/s, seconds, sample text)."""
    s = OracleSampler(w)
    gbs, el, rows, k = s.run(budget_s=budget_s)
    sample = ("%d whole requests of the workload (%d rows of (draft node, head)) in a seeded random "
              "order: index marshaling, mask packing and attention per request; the pool with the "
              "draft rows scattered in is built once before timing" % (k, rows))
    return gbs, el, sample, k


def run_reference(args):
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return 0
    cores = len(os.sched_getaffinity(0))
    from speculative_decode_mla_tree_gb300 import workloads as W
    steps = args.steps
    s = OracleSampler(W.config(args.config))
    s.run(steps=args.warmup)
    gbs, el, rows, k = s.run(steps=steps)
    sample = ("%d steps of one whole request each (%d rows of (draft node, head) in all), requests "
              "in a seeded random order after %d warm-up requests" % (k, rows, args.warmup))
    line = {"metric": METRIC, "value": gbs, "unit": "GB/s", "n_gpus": args.gpus, "steps": steps,
            "warmup": args.warmup, "ms_per_step": el / k * 1e3, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "impl": "reference",
            "config": {"workload": W.CONFIG_NAMES[args.config], "sample": "one whole request per step"},
            "cpu_baseline": {"value": gbs, "unit": "GB/s", "cores": cores, "kind": "oracle",
                             "sample": sample},
            "e2e": {"value": gbs, "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)
    return 0


def run_ours(args):
    import torch
    import torch.distributed as dist

    import __graft_entry__
    from speculative_decode_mla_tree_gb300 import abi, workloads as W
    from speculative_decode_mla_tree_gb300.step import VerifyStep

    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        dist.init_process_group("nccl")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if rank == 0:
        __graft_entry__.build()
    if world > 1:
        dist.barrier()
    __graft_entry__.build()

    w = W.config(args.config, args.kv_layout)
    fused = args.marshal == "fused"
    if fused and args.mask != "bits":
        raise SystemExit("--marshal fused packs the mask in its bit form: use --mask bits")
    st = VerifyStep(w, dev, max_splits=args.max_splits, path=args.path, mask_bits=args.mask == "bits",
                    fused=fused, skip_prefix=args.skip_prefix)
    stream = torch.cuda.Stream(dev)
    flush = torch.empty(FLUSH_BYTES // 4, dtype=torch.float32, device=dev)
    flush_sink = torch.empty((), dtype=torch.float32, device=dev)

    def flush_l2(v):
        flush.fill_(v)                                  # evict everything else from L2
        torch.sum(flush, dim=0, out=flush_sink)         # write back the dirty lines, leave clean ones

    with torch.cuda.stream(stream):
        for _ in range(2):
            st.run()
    torch.cuda.synchronize()
    assert int(st.status.item()) == 0, "device status %d" % int(st.status.item())

    if fused:
        names = ["prepare", "verify"]
        calls = [lambda: st.prepare(), lambda: st.verify()]
    else:
        names = ["scatter", "kv_indices", "mask_pack", "verify"]
        calls = [lambda: abi.mla_tree_draft_kv_scatter(st.draft_kv, st.out_cache_loc, st.pool, st.status),
                 lambda: abi.mla_tree_kv_indices_build(st.prefix_indices, st.prefix_indptr,
                                                       st.out_cache_loc, st.qo_indptr, st.kv_indices,
                                                       st.kv_indptr, st.status),
                 lambda: st.pack_mask(),
                 lambda: st.verify()]
    ncalls = len(calls)
    # one graph per call (the per-call breakdown) and one graph of the whole
    # step (what a serving engine replays; consecutive kernels overlap there)
    graphs = []
    for c in calls:
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            c()
        graphs.append(g)
    step_graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(step_graph, stream=stream):
        for c in calls:
            c()
    torch.cuda.synchronize()

    def step_calls(ev):
        ev[0].record(stream)
        for i, g in enumerate(graphs):
            g.replay()
            ev[i + 1].record(stream)

    def step_whole(ev):
        ev[0].record(stream)
        step_graph.replay()
        ev[1].record(stream)

    with torch.cuda.stream(stream):
        for _ in range(args.warmup):
            flush_l2(1.0)
            step_whole([torch.cuda.Event(enable_timing=True) for _ in range(2)])
            flush_l2(1.0)
            step_calls([torch.cuda.Event(enable_timing=True) for _ in range(ncalls + 1)])
    torch.cuda.synchronize()

    vis = os.environ.get("CUDA_VISIBLE_DEVICES", "")
    idx = vis.split(",")[local] if vis and vis.split(",")[local].strip().isdigit() else str(local)
    clocks = ClockSampler(idx)
    whole_ev = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(args.steps)]
    events = [[torch.cuda.Event(enable_timing=True) for _ in range(ncalls + 1)] for _ in range(args.steps)]
    clocks.start()
    time.sleep(0.3)
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    with torch.cuda.stream(stream):
        for k in range(args.steps):   # timed steps: the whole step as one graph
            flush_l2(float(k))
            step_whole(whole_ev[k])
    torch.cuda.synchronize()
    if world > 1:
        dist.barrier()
    with torch.cuda.stream(stream):
        for k in range(args.steps):   # the same steps call by call, for the breakdown
            flush_l2(float(k))
            step_calls(events[k])
    torch.cuda.synchronize()
    clk = clocks.stop()

    step_ms = [e[0].elapsed_time(e[1]) for e in whole_ev]
    call_ms = [[e[i].elapsed_time(e[i + 1]) for e in events] for i in range(ncalls)]
    total_ms = max_over_ranks(sum(step_ms), dev)
    assert int(st.status.item()) == 0

    kv_bytes = w.kv_bytes()
    value = whole_job_gbs(world, args.steps, kv_bytes, total_ms)
    byts, flops = alg_cost(w, args.mask == "bits", args.skip_prefix)
    verify_ms = statistics.mean(call_ms[-1])
    hbm, tf_burst, tf_sus, which = _peaks()
    achieved_gbs = byts / (verify_ms * 1e-3) / 1e9
    achieved_tf = flops / (verify_ms * 1e-3) / 1e12
    t_hbm, t_tc = byts / (hbm * 1e9), flops / (tf_burst * 1e12)
    bound = "hbm" if t_hbm >= t_tc else "tensor"
    launches_verify = abi.mla_tree_verify_launch_count(w.batch, w.total_q, w.heads, st.kv_indices.numel(),
                                                       args.max_splits, args.path)
    launches = args.steps * (ncalls - 1 + launches_verify)

    # end to end through the public API with host buffers
    e2e = None
    if not args.no_e2e:
        # the step's inputs packed in pinned host memory with the device
        # layout: one host-to-device copy in, one device-to-host copy out
        host_in = st.packed_inputs()
        host_out = torch.empty(st.outbuf.numel(), dtype=torch.uint8).pin_memory()
        h2d = host_in.numel()
        d2h = host_out.numel()
        ev = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(args.steps)]
        with torch.cuda.stream(stream):
            for k in range(args.warmup + args.steps):
                flush_l2(float(k))
                e = ev[k - args.warmup] if k >= args.warmup else None
                if e:
                    e[0].record(stream)
                st.inbuf.copy_(host_in, non_blocking=True)
                st.run()
                host_out.copy_(st.outbuf, non_blocking=True)
                if e:
                    e[1].record(stream)
        torch.cuda.synchronize()
        e2e_ms = max_over_ranks(sum(e[0].elapsed_time(e[1]) for e in ev), dev)
        e2e = {"value": whole_job_gbs(world, args.steps, kv_bytes, e2e_ms), "unit": "GB/s",
               "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
               "ms_per_step": e2e_ms / args.steps}

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        gbs, el, sample, k = cpu_baseline(w, args.cpu_seconds)
        cpu = {"value": gbs, "unit": "GB/s", "cores": len(os.sched_getaffinity(0)), "kind": "oracle",
               "sample": sample + " (%.1f s)" % el}

    if rank == 0:
        line = {
            "metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": total_ms / args.steps,
            "us_per_call": verify_ms * 1e3, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
            "config": {"workload": W.CONFIG_NAMES[args.config], "batch": w.batch, "heads": w.heads,
                       "draft_tokens": w.total_q, "kv_rows": kv_bytes // 1152,
                       "path": ["auto", "simt", "tensor-core"][args.path],
                       "max_splits": args.max_splits, "mask": args.mask, "marshal": args.marshal,
                       "skip_prefix": args.skip_prefix,
                       "kv_layout": args.kv_layout,
                       "l2": "flushed between steps: 256 MiB written then read back, outside the events",
                       "timing": "whole step as one CUDA graph (value, ms_per_step); per-call graphs "
                                 "(us_per_call, step_ms); CUDA events on the launching stream"},
            "step_ms": dict([(nm, statistics.mean(c)) for nm, c in zip(names, call_ms)] +
                            [("verify_p10", sorted(call_ms[-1])[len(call_ms[-1]) // 10]),
                             ("verify_p90", sorted(call_ms[-1])[(9 * len(call_ms[-1])) // 10])]),
            "roofline": {"kernel": "mla_tree_verify (all launches of the call)", "bound": bound,
                         "achieved": achieved_gbs if bound == "hbm" else achieved_tf,
                         "peak": hbm if bound == "hbm" else tf_burst,
                         "unit": "GB/s" if bound == "hbm" else "TFLOP/s",
                         "frac": (achieved_gbs / hbm) if bound == "hbm" else (achieved_tf / tf_burst),
                         "traffic": _traffic("verify_c%d" % args.config), "peak_source": which,
                         "alg_bytes_per_launch": byts, "alg_flops_per_launch": flops,
                         "hbm_frac": achieved_gbs / hbm, "tensor_frac": achieved_tf / tf_burst},
            "cpu_baseline": cpu,
            "e2e": e2e,
            "gpu_launches": launches,
            "clocks": clk,
        }
        print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()
    return 0


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=None,
                    help="timed steps (default: about a second of device time for the workload)")
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--config", type=int, default=5, choices=[1, 2, 3, 4, 5])
    ap.add_argument("--path", type=int, default=0, choices=[0, 1, 2])
    ap.add_argument("--max-splits", type=int, default=0)
    ap.add_argument("--kv-layout", default="shuffled", choices=["shuffled", "contiguous", "paged64"],
                    help="how pool slots are handed out: shuffled (the workloads' default), one "
                         "contiguous run, or random 64-slot pages")
    ap.add_argument("--marshal", default="fused", choices=["fused", "separate"],
                    help="scatter, index marshaling and mask packing as one launch or three")
    ap.add_argument("--mask", default="bits", choices=["bytes", "bits"],
                    help="tree-mask form: one byte or one bit per (row, column)")
    ap.add_argument("--skip-prefix", action="store_true",
                    help="verify with the prefix-skip switch (prefix columns of the mask unread)")
    ap.add_argument("--cpu-seconds", type=float, default=10.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    if args.steps is None:
        args.steps = DEFAULT_STEPS[args.config]
    if args.impl == "reference":
        return run_reference(args)
    return run_ours(args)


if __name__ == "__main__":
    sys.exit(main())
