#!/usr/bin/env python
"""Benchmark of the fused CSA indexer (score + top-512) on GB300.

One step = one call of csa_index_score_topk_fused over one decode batch: every
visible record of every query is scored against the FP8 compressed-K cache and
each query keeps its top-512 (scoring kernel + merge kernel). The default
workload is the long ragged decode batch: 64 queries, 65536..131072 compressed
records each (256K-512K tokens at 4:1), shuffled 64-record pages, 5% of records
with 8x scale outliers, seed 0. Its ~830 MB of keys per step are larger than
L2, so no flush is needed between steps.

Prints one JSON line. `--impl reference` times the fp64 CPU oracle instead
(the reference arm). Under torchrun each rank scores its own batch (seed =
rank): weak scaling, no collective on the data path.

`--op write_keys` measures the compressed-K writer instead: one step rewrites
every record of the workload's cache from bf16 key rows resident in HBM.
`--op recall` measures the Level-1 recall: one step scores the workload's
history at `--layers` target layers with 128-head queries and builds the
resident sets and page lists.
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
sys.path.insert(0, ROOT)

METRIC = "CSA indexer keys scored/s and HBM GB/s (fraction of peak), score+top-512"
UNIT = "keys/s"
K_TOP = 512
CSRC = os.path.join(ROOT, "sparse_attention_kv_e4m3_gb300", "csrc")
KERNEL_SOURCES = [os.path.join(CSRC, f)
                  for f in ("csa_index.cu", "csa_score64.cuh", "csa_ptx.cuh", "csa_select.cuh", "csa_internal.h")]
# committed ncu summary per bench leg: (file under profiles/, the sources its kernel is built from)
PROFILES = {
    "index": ("score_kernel_long_ragged_decode.md", KERNEL_SOURCES),
    "fp4": ("score_kernel_long_ragged_decode_mxfp4.md", KERNEL_SOURCES),
    "write_keys": ("write_keys_long_ragged_cache.md", [os.path.join(CSRC, "csa_writer.cu")]),
}


def kernel_source_hash(paths=None) -> str:
    h = hashlib.sha256()
    for p in paths or KERNEL_SOURCES:
        with open(p, "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def measured_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(p) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    except Exception:
        return 6800.0, "fallback"


def profiled_traffic(leg: str = "index"):
    """DRAM bytes per launch of the leg's kernel from its committed ncu summary,
    or None if there is none or the kernel's sources changed since that capture."""
    if leg not in PROFILES:
        return None
    name, sources = PROFILES[leg]
    try:
        text = open(os.path.join(ROOT, "profiles", name)).read()
    except OSError:
        return None
    vals = {}
    for line in text.splitlines():
        line = line.strip().strip("`")
        if ":" in line:
            k, v = line.split(":", 1)
            vals[k.strip()] = v.strip()
    if vals.get("kernel_source_sha256_16") != kernel_source_hash(sources):
        return None
    try:
        return float(vals["dram_bytes_per_launch"])
    except (KeyError, ValueError):
        return None


def algorithmic_bytes(w) -> int:
    """Bytes the step must move at minimum: 132 per visible record, 4 per
    page-table (and resident-list) entry, 16 KiB of q, 256 B of head weights and
    4 B of length per query, and the k x (4 + 4) output per query."""
    vis = w.visible_counts()
    pages = (vis + 63) // 64
    per_entry = 8 if w.resident is not None else 4
    rec = 68 if getattr(w, "record_format", "e4m3") == "mxfp4" else 132
    return int((vis * rec).sum() + (pages * per_entry).sum()
               + w.num_q * (64 * 128 * 2 + 64 * 4 + 4 + K_TOP * 8))


HEADS, HEAD_DIM = 64, 128
NOMINAL_HBM_GBS = 7900.0  # GB300's nominal HBM3e bandwidth, reported beside the measured copy peak
PER_CONFIG = ("tiny_decode", "decode_batch", "resident_1m", "prefill_chunk")


def algorithmic_flops(w) -> int:
    """The contraction's FLOPs: 2 * H * D per (query, visible record), the cost
    model the pages' per-token FLOP figures follow (FlashMemory-DeepSeek-V4,
    "Per-decode-token FLOPs (whole model)"); the relu, head weights and
    sigmoid (about 3H operations per pair) are not counted."""
    return int(2 * HEADS * HEAD_DIM * int(w.visible_counts().sum()))


def indexer_gflop(layers: int, records_per_query: int, heads: int = HEADS, dim: int = HEAD_DIM) -> float:
    """GFLOP of scoring one decode token's query against `records_per_query`
    records in each of `layers` indexer layers, at 2 * heads * dim per pair."""
    return layers * records_per_query * 2.0 * heads * dim / 1e9


def measured_peak_tflops():
    """(dense bf16 TFLOP/s sustained, its source), from MEASURED_PEAKS.json."""
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(p) as f:
            d = json.load(f)
        return float(d["bf16_tflops_sustained"]), "measured bf16_tflops_sustained"
    except Exception:
        return 1700.0, "fallback bf16 sustained"


def measure_configs(names, dev, steps: int = 20):
    """The other configs of the indexer, one fused score + top-512 call each:
    the median of `steps` event-timed calls, with L2 flushed (a 256 MB write,
    outside the timed region) before every call, since most of these inputs fit
    in the 129 MB L2. Reports us per call, keys/s, GB/s of algorithmic bytes and
    its fraction of the measured copy bandwidth, TFLOP/s of the contraction, and
    for chunked prefill (the contraction-dense config) the fraction of the dense
    e4m3 tensor peak, taken as twice the measured sustained bf16 figure (the
    nominal e4m3 : bf16 ratio, 4.5 : 2.25 PFLOP/s)."""
    import torch
    from sparse_attention_kv_e4m3_gb300 import native, synth

    hbm, hbm_src = measured_peaks()
    bf16, bf16_src = measured_peak_tflops()
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream(dev)
    out = {}
    for name in names:
        w = synth.config(name)
        prob = native.Problem.from_workload(w, device=dev)
        ws = native.alloc_workspace(prob, K_TOP, dev)
        idx = torch.empty((w.num_q, K_TOP), dtype=torch.int32, device=dev)
        vals = torch.empty((w.num_q, K_TOP), dtype=torch.float32, device=dev)
        call = native.PreparedFused(prob, K_TOP, ws, idx, vals, stream=stream)
        for _ in range(3):
            call()
        torch.cuda.synchronize(dev)
        if int(prob.dev_status.item()) != 0:
            raise RuntimeError(f"{name}: device status {int(prob.dev_status.item())}")
        ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(steps)]
        for a, b in ev:
            flush.zero_()
            a.record(stream)
            call()
            b.record(stream)
        torch.cuda.synchronize(dev)
        ms = statistics.median(a.elapsed_time(b) for a, b in ev)
        keys, nbytes, flops = int(w.visible_counts().sum()), algorithmic_bytes(w), algorithmic_flops(w)
        rec = {"us": ms * 1e3, "queries": w.num_q, "records": keys, "keys_per_s": keys / (ms / 1e3),
               "gbs": nbytes / (ms / 1e3) / 1e9, "frac_hbm": nbytes / (ms / 1e3) / 1e9 / hbm,
               "frac_of_nominal": nbytes / (ms / 1e3) / 1e9 / NOMINAL_HBM_GBS,
               "algorithmic_bytes": nbytes, "flops": flops, "tflops": flops / (ms / 1e3) / 1e12}
        if name.startswith("prefill"):
            rec["tensor_frac"] = rec["tflops"] / (2.0 * bf16)
            rec["tensor_peak"] = f"2 x {bf16} TFLOP/s ({bf16_src}, e4m3 at the nominal 2:1 ratio)"
        out[name] = rec
        del call, prob, ws, idx, vals
        torch.cuda.empty_cache()
    out["timing"] = (f"median of {steps} calls, L2 flushed before each; peaks: {hbm} GB/s ({hbm_src})")
    return out


# ---------------------------------------------------------------------- clocks

class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, bus_id=None):
        cmd = ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits", "-lms", "200"]
        if bus_id:
            cmd += ["-i", bus_id]
        self.t0 = time.time()
        try:
            self.p = subprocess.Popen(cmd, stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.p = None

    def stop(self):
        if self.p is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.p.terminate()
        try:
            out, _ = self.p.communicate(timeout=5)
        except subprocess.TimeoutExpired:
            self.p.kill()
            out, _ = self.p.communicate()
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in out.splitlines():
            parts = [x.strip() for x in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                smax.append(float(parts[2]))
            except ValueError:
                continue
            for n, v in zip(names, parts[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(smax) if smax else None,
                "reasons": sorted(reasons), "samples": len(sm)}


# ---------------------------------------------------------------------- ranks

def reduce_over_ranks(keys: float, ms_step: float, dist=None, device=None):
    """Whole-job throughput inputs: keys summed over ranks, step time maxed over
    ranks (every rank scores its own independent batch)."""
    if dist is None:
        return float(keys), float(ms_step)
    import torch

    k = torch.tensor([float(keys)], dtype=torch.float64, device=device)
    m = torch.tensor([float(ms_step)], dtype=torch.float64, device=device)
    dist.all_reduce(k, op=dist.ReduceOp.SUM)
    dist.all_reduce(m, op=dist.ReduceOp.MAX)
    return float(k.item()), float(m.item())


def merge_shard_topk(shards, k: int):
    """Exact top-k of one row from per-shard top-k lists [(positions, logits), ...]
    (context-parallel scoring: each shard holds some of the row's pages). The global
    top-k is contained in the union of the local ones; ties rank lower positions first."""
    pos = np.concatenate([np.asarray(p, dtype=np.int64) for p, _ in shards])
    lg = np.concatenate([np.asarray(v, dtype=np.float64) for _, v in shards])
    keep = pos >= 0
    pos, lg = pos[keep], lg[keep]
    order = np.lexsort((pos, -lg))[:k]
    out_p = np.full(k, -1, dtype=np.int64)
    out_l = np.full(k, -np.inf)
    out_p[: len(order)] = pos[order]
    out_l[: len(order)] = lg[order]
    return out_p, out_l


# ---------------------------------------------------------------------- oracle (reference arm / CPU baseline)

def oracle_rate(w, budget_s: float, min_records: int = 4096):
    """Times the oracle's top-512 on a bounded prefix sample of every row;
    returns (keys/s, records scored, seconds, threads, sample text)."""
    import oracle

    oracle.build()
    P = oracle.Problem(w)
    t = time.perf_counter()
    _, _, n0 = oracle.topk_sample(P, 0, min(4, w.num_q), min_records, K_TOP)
    dt0 = max(time.perf_counter() - t, 1e-6)
    rate0 = n0 / dt0
    per_row = int(max(min_records, min(int(w.visible_counts().max()), rate0 * budget_s / w.num_q)))
    t = time.perf_counter()
    _, _, n = oracle.topk_sample(P, 0, w.num_q, per_row, K_TOP)
    dt = time.perf_counter() - t
    sample = f"the first {per_row} visible records of each of the {w.num_q} rows ({n} records), top-{K_TOP}"
    return n / dt, n, dt, oracle.threads(), sample


def run_reference(args):
    if int(os.environ.get("RANK", "0")) != 0:
        return 0
    from sparse_attention_kv_e4m3_gb300 import synth
    import oracle

    oracle.build()
    w = synth.config(args.workload, seed=0)
    P = oracle.Problem(w)
    # size each step so that warmup + steps fit in about two minutes
    t = time.perf_counter()
    _, _, n0 = oracle.topk_sample(P, 0, 1, 8192, K_TOP)
    rate = n0 / max(time.perf_counter() - t, 1e-6)
    per_step = max(4096, int(rate * 120.0 / max(args.steps + args.warmup, 1)))
    per_row = max(64, min(int(w.visible_counts().max()), per_step // w.num_q))
    for _ in range(args.warmup):
        oracle.topk_sample(P, 0, w.num_q, per_row, K_TOP)
    times, total = [], 0
    for _ in range(args.steps):
        t = time.perf_counter()
        _, _, n = oracle.topk_sample(P, 0, w.num_q, per_row, K_TOP)
        times.append(time.perf_counter() - t)
        total += n
    value = total / sum(times)
    sample = f"each step: the first {per_row} visible records of each of the {w.num_q} rows, top-{K_TOP}"
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * sum(times) / len(times),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": args.workload, "k": K_TOP, "sample": sample},
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": oracle.threads(), "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line))
    return 0


# ---------------------------------------------------------------------- native arm

def run_native(args):
    import torch

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    dist = None
    if world > 1:
        import torch.distributed as dist

        dist.init_process_group("nccl")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)

    from sparse_attention_kv_e4m3_gb300 import build, native, synth

    build.build()
    native.load()
    w = synth.config(args.workload, seed=rank)
    if args.op == "fp4":  # the same rows and pages over an MXFP4 cache (68-byte records)
        w = synth.mxfp4_cache(w, seed=rank)
    prob = native.Problem.from_workload(w, device=dev)
    k = K_TOP
    ws = native.alloc_workspace(prob, k, dev)
    idx = torch.empty((w.num_q, k), dtype=torch.int32, device=dev)
    vals = torch.empty((w.num_q, k), dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream(dev)
    keys = int(w.visible_counts().sum())
    alg_bytes = algorithmic_bytes(w)

    # the C entry point with its arguments marshalled once (native.PreparedFused): a
    # serving loop's host cost per call, not the plain binding's struct building
    step = native.PreparedFused(prob, k, ws, idx, vals, stream=stream)

    step()  # first call: library set-up outside the warm-up
    torch.cuda.synchronize(dev)
    # The clock sampler starts before the warm-up steps, so that the GPU is not left
    # idle between the warm-up and the timed steps (an idle GPU lowers its clocks,
    # and the first timed steps would pay for raising them again).
    bus = None
    try:
        props = torch.cuda.get_device_properties(dev)
        bus = "%08X:%02X:%02X.0" % (props.pci_domain_id, props.pci_bus_id, props.pci_device_id)
    except Exception:
        pass
    sampler = ClockSampler(bus)
    time.sleep(0.3)

    for _ in range(max(args.warmup, 3)):
        step()
    torch.cuda.synchronize(dev)
    if int(prob.dev_status.item()) != 0:
        raise RuntimeError(f"device status {int(prob.dev_status.item())} after warm-up")

    E = lambda: torch.cuda.Event(enable_timing=True)  # noqa: E731
    e0, e1 = E(), E()
    if dist:
        dist.barrier()
    torch.cuda.synchronize(dev)
    t_wall = time.perf_counter()
    e0.record(stream)
    for _ in range(args.steps):  # the timed steps: plain calls, nothing recorded in between
        step()
    e1.record(stream)
    torch.cuda.synchronize(dev)
    wall = time.perf_counter() - t_wall
    if dist:
        dist.barrier()
    # keep the same load running until the clock sampler has seen at least ~1 s of it
    extra = 0
    while time.perf_counter() - t_wall < 1.2:
        step()
        extra += 1
        if extra % 50 == 0:
            torch.cuda.synchronize(dev)
    torch.cuda.synchronize(dev)
    clocks = sampler.stop()
    if extra:
        clocks["window"] = f"timed region ({wall:.3f} s) plus {extra} identical untimed steps"

    ms_total = e0.elapsed_time(e1)
    ms_step = ms_total / args.steps
    # the scoring kernel's own duration (roofline), from a separate loop of the same
    # steps with an event before each call and one between its two kernels; the
    # median, because the first step of the loop also holds the host's launch of
    # that call (the GPU is idle after the synchronize until the call is enqueued)
    n_mark = max(min(args.steps, 200), 5)
    starts, mids = [E() for _ in range(n_mark)], [E() for _ in range(n_mark)]
    for i in range(n_mark):
        starts[i].record(stream)
        step(mark=mids[i])
    torch.cuda.synchronize(dev)
    phase1_ms = statistics.median(starts[i].elapsed_time(mids[i]) for i in range(n_mark))
    status = int(prob.dev_status.item())

    keys_all, ms_max = reduce_over_ranks(keys, ms_step, dist, dev)
    value = keys_all / (ms_max / 1e3)

    # ---- end to end through the public API: per-step inputs from pinned host memory
    host = {n: torch.from_numpy(a).pin_memory() for n, a in
            (("q", w.q.view("int16")), ("fused_w", w.fused_w), ("q_len", w.q_len), ("page_table", w.page_table))}
    h_idx = torch.empty((w.num_q, k), dtype=torch.int32).pin_memory()
    h_vals = torch.empty((w.num_q, k), dtype=torch.float32).pin_memory()
    h2d = sum(t.numel() * t.element_size() for t in host.values())
    d2h = h_idx.numel() * 4 + h_vals.numel() * 4
    ref_idx = idx.cpu()
    # Pipelined like a serving loop: step i + 1's inputs are copied in, and step i's
    # results read back, on a copy stream while the compute stream runs step i (or
    # i + 1); inputs and outputs are double-buffered on the device.
    import dataclasses

    probs = [prob, dataclasses.replace(prob, q=torch.empty_like(prob.q), fused_w=torch.empty_like(prob.fused_w),
                                       q_len=torch.empty_like(prob.q_len),
                                       page_table=torch.empty_like(prob.page_table))]
    outs = [(idx, vals), (torch.empty_like(idx), torch.empty_like(vals))]
    h_outs = [(h_idx, h_vals), (torch.empty_like(h_idx).pin_memory(), torch.empty_like(h_vals).pin_memory())]
    cstream = torch.cuda.Stream(dev)
    ev_in, ev_done, ev_out = ([torch.cuda.Event(), torch.cuda.Event()] for _ in range(3))

    def h2d_into(b):
        p = probs[b]
        with torch.cuda.stream(cstream):
            p.q.view(torch.int16).copy_(host["q"], non_blocking=True)
            p.fused_w.copy_(host["fused_w"], non_blocking=True)
            p.q_len.copy_(host["q_len"], non_blocking=True)
            p.page_table.copy_(host["page_table"], non_blocking=True)
        ev_in[b].record(cstream)

    def e2e_run(n, start_event=None):
        if start_event is not None:
            cstream.wait_event(start_event)
        h2d_into(0)
        for i in range(n):
            b = i % 2
            stream.wait_event(ev_in[b])
            if i >= 2:
                stream.wait_event(ev_out[b])  # step i - 2's results (same buffers) have been read back
            native.csa_index_score_topk_fused(probs[b], k, ws, outs[b][0], outs[b][1], stream=stream)
            ev_done[b].record(stream)
            if i + 1 < n:
                if i >= 1:
                    cstream.wait_event(ev_done[1 - b])  # step i - 1 is done with the other input buffers
                h2d_into(1 - b)
            cstream.wait_event(ev_done[b])
            with torch.cuda.stream(cstream):
                h_outs[b][0].copy_(outs[b][0], non_blocking=True)
                h_outs[b][1].copy_(outs[b][1], non_blocking=True)
            ev_out[b].record(cstream)
        stream.wait_event(ev_out[(n - 1) % 2])

    e2e_run(3)
    torch.cuda.synchronize(dev)
    if dist:
        dist.barrier()
    a0, a1 = E(), E()
    a0.record(stream)
    e2e_run(args.steps, start_event=a0)
    a1.record(stream)
    torch.cuda.synchronize(dev)
    for hb in h_outs[: min(args.steps, 2)]:  # every step has the same inputs: the same top-k
        if not torch.equal(hb[0], ref_idx):
            raise RuntimeError("end-to-end results differ from the device-resident run")
    e2e_ms = a0.elapsed_time(a1) / args.steps
    _, e2e_ms = reduce_over_ranks(0.0, e2e_ms, dist, dev)
    e2e_value = keys_all / (e2e_ms / 1e3)

    peak, peak_src = measured_peaks()
    achieved = alg_bytes / (phase1_ms / 1e3) / 1e9
    traffic = profiled_traffic(args.op)
    line = {
        "metric": METRIC if args.op == "index" else METRIC + ", MXFP4 records", "value": value, "unit": UNIT,
        "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms_max, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "e4m3" if args.op == "index" else "e2m1 (MXFP4) -> e4m3", "data": "synthetic",
        "config": {"workload": args.workload, "record_format": getattr(w, "record_format", "e4m3"),
                   "queries": w.num_q, "k": k, "records_per_step": keys,
                   "records_per_query": "65536..131072" if args.workload == "long_ragged_decode" else None,
                   "key_bytes_per_step": w.k_bytes(), "algorithmic_bytes_per_step": alg_bytes,
                   "l2": "inputs larger than L2 (no flush)", "parallelism": f"replicas x{world}",
                   "seed": rank},
        "queries_per_s": w.num_q * world / (ms_max / 1e3),
        "gbs": alg_bytes * world / (ms_max / 1e3) / 1e9,
        "roofline": {"kernel": ("w64::score_kernel_w64<topk, e4m3> (scoring phase)" if args.op == "index" else
                                "w64::score_kernel_w64<topk, mxfp4> (scoring phase)"), "bound": "hbm", "achieved": achieved,
                     "peak": peak, "peak_source": f"{peak_src} hbm_gbs", "unit": "GB/s",
                     "frac": achieved / peak, "traffic": traffic, "phase1_ms": phase1_ms,
                     "algorithmic_bytes_per_launch": alg_bytes,
                     "frac_of_nominal": achieved / NOMINAL_HBM_GBS,
                     "step_frac": alg_bytes / (ms_max / 1e3) / 1e9 / peak,
                     "step_note": "step_frac: the whole step (scoring kernel and merge kernel) against the same peak"},
        "clocks": clocks,
        "e2e": {"value": e2e_value, "unit": UNIT, "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                "inputs": "q, fused_w, q_len, page_table copied from pinned host memory every step; "
                          "the compressed-K cache stays resident in HBM",
                "pipelining": "a copy stream brings step i+1's inputs in and reads step i's idx/vals back "
                              "while the compute stream runs; device inputs and outputs double-buffered",
                "ms_per_step": e2e_ms},
        "gpu_launches": 2 * args.steps,
        "device_status": status,
        "wall_s": wall,
        "flops_per_step": algorithmic_flops(w),
        "tflops": algorithmic_flops(w) * world / (ms_max / 1e3) / 1e12,
        # the same 2*H*D-per-pair model applied to the pages' 1M-context decode
        # token (21 indexer layers; full history vs KMAX=384 resident pages plus
        # the Level-1 retriever's 3 layers at H=128 every 64 tokens)
        "cost_model_gflop_per_token_1m": {
            "full_history_scoring": indexer_gflop(21, 262144),
            "resident_scoring_and_level1": indexer_gflop(21, 384 * 64) + indexer_gflop(3, 262144, heads=128) / 64},
    }
    if rank == 0 and world == 1 and not args.no_per_config and args.op == "index":
        line["per_config"] = measure_configs(PER_CONFIG, dev)
        # the next-row kernels on the same workload's geometry (their own lines:
        # bench.py --op write_keys / --op recall)
        extra_args = argparse.Namespace(**{**vars(args), "steps": min(args.steps, 200)})
        for op, fn in (("write_keys", run_write_keys), ("recall", run_recall)):
            r = fn(extra_args, emit=False)
            line[op] = {"metric": r["metric"], "value": r["value"], "unit": r["unit"], "ms_per_step": r["ms_per_step"],
                        "gbs": r["roofline"]["achieved"], "frac": r["roofline"]["frac"],
                        "device_status": r["device_status"]}
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        rate, n, dt, threads, sample = oracle_rate(w, budget_s=10.0)
        line["cpu_baseline"] = {"value": rate, "unit": UNIT, "cores": threads, "kind": "oracle",
                                "sample": sample, "seconds": dt,
                                "affinity_cores": len(os.sched_getaffinity(0))}
    if rank == 0:
        print(json.dumps(line))
    if dist:
        dist.destroy_process_group()
    return 0


def run_write_keys(args, emit: bool = True):
    """The compressed-K writer on the workload's cache geometry: every visible
    record of every request rewritten from bf16 rows (one row per record)."""
    import torch
    from sparse_attention_kv_e4m3_gb300 import build, native, synth

    build.build()
    native.load()
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    w = synth.config(args.workload)
    lens = [int(x) for x in w.q_len]
    req = np.concatenate([np.full(L, r, np.int32) for r, L in enumerate(lens)])
    pos = np.concatenate([np.arange(L, dtype=np.int32) for L in lens])
    n = int(req.size)
    g = torch.Generator(device=dev)
    g.manual_seed(0)
    keys = torch.randn((n, 128), generator=g, device=dev, dtype=torch.float32).to(torch.bfloat16)
    req_d, pos_d = torch.from_numpy(req).to(dev), torch.from_numpy(pos).to(dev)
    pt_d = torch.from_numpy(np.ascontiguousarray(w.page_table, dtype=np.int32)).to(dev)
    kv = torch.zeros(w.kv.shape, dtype=torch.uint8, device=dev)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    del w
    stream = torch.cuda.current_stream(dev)

    def step():
        native.csa_index_write_keys(keys, pos_d, kv, pt_d, row_req=req_d, dev_status=status, stream=stream)

    for _ in range(max(args.warmup, 3)):
        step()
    torch.cuda.synchronize(dev)
    bus = None
    try:
        props = torch.cuda.get_device_properties(dev)
        bus = "%08X:%02X:%02X.0" % (props.pci_domain_id, props.pci_bus_id, props.pci_device_id)
    except Exception:
        pass
    sampler = ClockSampler(bus)
    time.sleep(0.3)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    steps = min(args.steps, 200)
    torch.cuda.synchronize(dev)
    t_wall = time.perf_counter()
    e0.record(stream)
    for _ in range(steps):
        step()
    e1.record(stream)
    torch.cuda.synchronize(dev)
    wall = time.perf_counter() - t_wall
    extra = 0
    while time.perf_counter() - t_wall < 1.2:
        step()
        extra += 1
    torch.cuda.synchronize(dev)
    clocks = sampler.stop()
    if extra:
        clocks["window"] = f"timed region ({wall:.3f} s) plus {extra} identical untimed steps"
    ms = e0.elapsed_time(e1) / steps
    # algorithmic bytes per row: the bf16 row, its request and position, one
    # page-table entry, and the 132-byte record written
    alg = n * (256 + 4 + 4 + 4 + 132)
    peak, src = measured_peaks()
    gbs = alg / (ms * 1e-3) / 1e9
    line = {
        "metric": "compressed-K writer rows/s and HBM GB/s (fraction of peak)",
        "value": n / (ms * 1e-3),
        "unit": "rows/s",
        "n_gpus": 1,
        "steps": steps,
        "warmup": max(args.warmup, 3),
        "ms_per_step": ms,
        "higher_is_better": True,
        "dtype": "bf16->e4m3",
        "data": "synthetic",
        "config": {"workload": f"{args.workload} cache rewritten", "rows": n,
                   "l2": "inputs and cache larger than L2; no flush"},
        "roofline": {"kernel": "write_keys_kernel", "bound": "hbm", "achieved": gbs, "peak": peak,
                     "peak_source": f"{src} hbm_gbs", "unit": "GB/s", "frac": gbs / peak,
                     "traffic": profiled_traffic("write_keys"),
                     "algorithmic_bytes_per_launch": alg},
        "clocks": clocks,
        "gpu_launches": steps,
        "device_status": int(status.item()),
    }
    if emit:
        print(json.dumps(line))
    return line


def run_recall(args, emit: bool = True):
    """Level-1 recall over `--layers` target layers of the workload's history
    (each layer its own device copy of the cache and its own 128-head query):
    every visible record scored per layer, combined by max, thresholded, with the
    recency tail and sink, and the resident page list per row."""
    import ctypes
    import dataclasses

    import torch
    from sparse_attention_kv_e4m3_gb300 import build, native, synth

    build.build()
    native.load()
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    w = synth.config(args.workload)
    lw = synth.level1_layers(w, args.layers, seed=1)
    p0 = native.Problem.from_workload(lw[0], device=dev)
    P = [p0]
    for x in lw[1:]:
        q = torch.from_numpy(x.q.view("int16")).to(dev).view(torch.bfloat16)
        P.append(dataclasses.replace(p0, q=q, fused_w=torch.from_numpy(x.fused_w).to(dev), kv=p0.kv.clone(),
                                     dev_status=None))
    records = int(sum(min(int(L), 64 * w.page_table.shape[1]) for L in w.q_len))
    del w, lw
    num_q, pts = p0.num_q, int(p0.page_table.shape[1])
    stride = 64 * pts
    keep = torch.zeros((num_q, stride), dtype=torch.uint8, device=dev)
    sc = torch.zeros((num_q, stride), dtype=torch.float32, device=dev)
    pages = torch.zeros((num_q, pts), dtype=torch.int32, device=dev)
    npg = torch.zeros(num_q, dtype=torch.int32, device=dev)
    out = (keep, pages, npg, sc)
    arr = (native.Args * len(P))(*[p.args() for p in P])
    ra = native.RecallArgs(ctypes.addressof(arr), len(P), native.ENSEMBLE_MAX, args.threshold, args.sink, args.recent,
                           pts, keep.data_ptr(), stride, pages.data_ptr(), npg.data_ptr(), sc.data_ptr())
    lib = native.load()
    ws = torch.empty(lib.csa_recall_workspace_bytes(ctypes.byref(ra)), dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream(dev)

    def step():
        st = lib.csa_recall_level1(ctypes.byref(ra), ws.data_ptr(), ws.numel(), stream.cuda_stream)
        if st:
            raise RuntimeError(native.status_str(st))

    for _ in range(max(args.warmup, 3)):
        step()
    torch.cuda.synchronize(dev)
    bus = None
    try:
        props = torch.cuda.get_device_properties(dev)
        bus = "%08X:%02X:%02X.0" % (props.pci_domain_id, props.pci_bus_id, props.pci_device_id)
    except Exception:
        pass
    sampler = ClockSampler(bus)
    time.sleep(0.3)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    steps = min(args.steps, 100)
    torch.cuda.synchronize(dev)
    t_wall = time.perf_counter()
    e0.record(stream)
    for _ in range(steps):
        step()
    e1.record(stream)
    torch.cuda.synchronize(dev)
    wall = time.perf_counter() - t_wall
    extra = 0
    while time.perf_counter() - t_wall < 1.2:
        step()
        extra += 1
    torch.cuda.synchronize(dev)
    clocks = sampler.stop()
    if extra:
        clocks["window"] = f"timed region ({wall:.3f} s) plus {extra} identical untimed steps"
    ms = e0.elapsed_time(e1) / steps
    # algorithmic bytes: each layer's visible records read once (132 B), and per
    # position the keep byte and the fp32 combined score written
    alg = args.layers * records * 132 + records * 5
    peak, src = measured_peaks()
    gbs = alg / (ms * 1e-3) / 1e9
    # kernels per step: one scorer launch per layer, then the keep and list kernels
    # (the zeroing of the combined-score plane is a memset)
    launches = steps * (args.layers + 2)
    line = {
        "metric": "Level-1 recall chunks/s and HBM GB/s (fraction of peak)",
        "value": records / (ms * 1e-3),
        "unit": "chunks/s",
        "n_gpus": 1,
        "steps": steps,
        "warmup": max(args.warmup, 3),
        "ms_per_step": ms,
        "higher_is_better": True,
        "dtype": "e4m3 x bf16 -> f32",
        "data": "synthetic",
        "config": {"workload": f"{args.workload} history, Level-1 recall", "layers": args.layers,
                   "heads": 128, "ensemble": "max", "threshold": args.threshold, "sink": args.sink,
                   "recent": args.recent, "chunks": records,
                   "l2": "each layer's cache larger than L2; no flush"},
        "roofline": {"kernel": "whole step", "bound": "hbm", "achieved": gbs, "peak": peak,
                     "peak_source": f"{src} hbm_gbs", "unit": "GB/s", "frac": gbs / peak, "traffic": None,
                     "algorithmic_bytes_per_launch": alg},
        "clocks": clocks,
        "gpu_launches": launches,
        "device_status": int(p0.dev_status.item()),
        "resident_pages_mean": float(npg.float().mean().item()),
    }
    if emit:
        print(json.dumps(line))
    return line


def main():
    ap = argparse.ArgumentParser(description=__doc__.splitlines()[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", default="native", choices=["native", "reference"])
    ap.add_argument("--workload", default="long_ragged_decode")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-per-config", action="store_true", help="skip the other configs' measurements")
    ap.add_argument("--op", default="index", choices=["index", "fp4", "write_keys", "recall"],
                    help="index: the indexer on e4m3 records (headline); fp4: the same on MXFP4 records")
    ap.add_argument("--layers", type=int, default=3, help="recall: target layers")
    ap.add_argument("--threshold", type=float, default=0.5, help="recall: keep threshold")
    ap.add_argument("--sink", type=int, default=4, help="recall: attention-sink chunks")
    ap.add_argument("--recent", type=int, default=512, help="recall: recency-tail chunks")
    args = ap.parse_args()
    if args.op == "write_keys":
        run_write_keys(args)
        return 0
    if args.op == "recall":
        run_recall(args)
        return 0
    if args.impl == "reference":
        return run_reference(args)
    return run_native(args)


if __name__ == "__main__":
    sys.exit(main())
